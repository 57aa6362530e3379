"""Schedule parity: the device reverse index is bit-exact against the oracle.

"Sparse Attention" (dinara-dl), Chapter 5 "Reverse index"; "Kernel optimization for
MiniMax M3", load-balancing and no-D2H sections.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.util import BF16_MAX_ABS, BF16_REL_L2, LSE_MAX_ABS, TILE, WINDOW, check_worklist, compare_outputs

pytestmark = pytest.mark.gpu


def _msa():
    import block_sparse_gqa_gb300 as msa
    return msa


def gpu_schedule(idx_np, nblocks, schedule=None):
    msa = _msa()
    idx = torch.from_numpy(np.ascontiguousarray(idx_np, np.int32)).cuda()
    s = msa.build_schedule(idx, nblocks, schedule=schedule)
    return s, s.export()


def assert_same(exp, ref, N, Lkv):
    for k in ("counts", "offsets", "qlist", "slot", "cmap"):
        np.testing.assert_array_equal(exp[k], ref[k], err_msg=k)
    assert exp["E"] == ref["E"] and exp["nsb"] == ref["nsb"]
    assert exp["path"] == oracle.dispatch(ref["E"], ref["nsb"])
    check_worklist(exp, ref, N)
    tiles, wt = oracle.worklist(ref["offsets"], ref["qlist"], N, window=WINDOW, tile_rows=TILE)
    np.testing.assert_array_equal(np.asarray(exp["window_tiles"]), wt, err_msg="window_tiles")
    np.testing.assert_array_equal(np.asarray(exp["tiles"]).reshape(-1, 4), tiles, err_msg="tiles")


@pytest.mark.parametrize("name", ["tiny", "m3", "long", "lowreuse", "fp8"])
def test_schedule_matches_oracle(name):
    cfg = workloads.CONFIGS[name]
    idx = workloads.make_indices(cfg)
    ref = oracle.schedule(idx, Lkv=cfg.Lkv)
    s, exp = gpu_schedule(idx, cfg.nblocks)
    assert exp["status"] == 0
    assert_same(exp, ref, cfg.N, cfg.Lkv)
    s.close()


def test_schedule_edge_cases():
    rng = np.random.default_rng(0)
    cases = []
    # pads, duplicates, future blocks; N not a multiple of 32 or 256; queries at the tail
    N, Lkv, Hkv, topK = 300, 1024, 2, 6
    nb = Lkv // 128
    idx = rng.integers(-1, nb, size=(N, Hkv, topK)).astype(np.int32)
    idx[:, :, -1] = idx[:, :, 0]
    cases.append((idx, Lkv))
    cases.append((np.array([[[0]]], np.int32), 128))                       # one query, topK 1
    cases.append((np.full((64, 1, 4), -1, np.int32), 512))                 # no entries at all
    full = np.tile(np.arange(8, dtype=np.int32)[::-1], (1024, 3, 1))       # every block, most in the future
    cases.append((full, 1024))
    for idx, Lkv in cases:
        ref = oracle.schedule(idx, Lkv=Lkv)
        s, exp = gpu_schedule(idx, Lkv // 128)
        assert_same(exp, ref, idx.shape[0], Lkv)
        s.close()


def test_schedule_bad_index_flagged_and_ignored():
    msa = _msa()
    idx = np.array([[[0, 5, -3, 0]], [[1, 0, -1, 99]]], np.int32)  # nblocks = 2, N = 2 at the tail of 256
    ref = oracle.schedule(idx, Lkv=256)
    s, exp = gpu_schedule(idx, 2)
    assert exp["status"] & 1 and ref["status"] == 1
    for k in ("counts", "offsets", "qlist", "slot", "cmap"):
        np.testing.assert_array_equal(exp[k], ref[k])
    assert s.query()["status_code"] == 5  # MSA_ERR_BAD_INDEX
    assert msa.lib().msa_schedule_status(s.handle) == 5  # the same sticky bit through msa_schedule_status
    s.close()
    clean, _ = gpu_schedule(np.array([[[0, -1]], [[1, 0]]], np.int32), 2)
    assert msa.lib().msa_schedule_status(clean.handle) == 0
    clean.close()
    with pytest.raises(msa.MsaError):
        msa.build_schedule(torch.zeros((4, 1, 2), dtype=torch.int32, device="cuda"), 0)


def test_schedule_deterministic_and_reusable():
    cfg = workloads.CONFIGS["m3"]
    idx = workloads.make_indices(cfg)
    s, a = gpu_schedule(idx, cfg.nblocks)
    _, b = gpu_schedule(idx, cfg.nblocks, schedule=s)
    for k in ("counts", "offsets", "qlist", "slot", "cmap", "tiles", "window_tiles"):
        np.testing.assert_array_equal(a[k], b[k])
    idx2 = workloads.make_indices(cfg, seed=77)
    _, c = gpu_schedule(idx2, cfg.nblocks, schedule=s)
    assert_same(c, oracle.schedule(idx2, Lkv=cfg.Lkv), cfg.N, cfg.Lkv)
    s.close()


@pytest.mark.parametrize("name", ["m3", "lowreuse"])
def test_schedule_rebuilds_start_clean(name):
    """A rebuild of the same schedule starts from the bitmask and status the previous
    build's row scan cleared (no memset after the first build): other lists, a bad id
    (flagged), then clean lists again (the flag is gone).  m3 takes the CTA-per-row scan,
    lowreuse (8 bitmask words per row) the warp-per-row one."""
    msa = _msa()
    cfg = workloads.CONFIGS[name]
    idx = workloads.make_indices(cfg)
    s, _ = gpu_schedule(idx, cfg.nblocks)
    bad = workloads.make_indices(cfg, seed=5)
    bad[3, 1, 2] = cfg.nblocks + 7  # invalid: ignored and flagged
    _, b = gpu_schedule(bad, cfg.nblocks, schedule=s)
    ref_b = oracle.schedule(bad, Lkv=cfg.Lkv)
    assert b["status"] & 1 and ref_b["status"] == 1
    assert_same(b, ref_b, cfg.N, cfg.Lkv)
    assert msa.lib().msa_schedule_status(s.handle) == 5
    for seed in (6, None):
        idx2 = workloads.make_indices(cfg, seed=seed)
        _, c = gpu_schedule(idx2, cfg.nblocks, schedule=s)
        assert c["status"] == 0 and msa.lib().msa_schedule_status(s.handle) == 0
        assert_same(c, oracle.schedule(idx2, Lkv=cfg.Lkv), cfg.N, cfg.Lkv)
    s.close()


@pytest.mark.parametrize("N,Lkv,Hkv,topK", [(1, 131072, 4, 16), (5, 2048, 1, 3), (31, 65536, 4, 8), (33, 8192, 2, 15),
                                            (64, 4096, 1, 16), (64, 4096, 4, 4), (65, 4096, 4, 4), (16, 65536, 4, 17),
                                            (300, 2048, 1, 3), (1024, 1024, 1, 1)])
def test_schedule_small_inputs_match_oracle(N, Lkv, Hkv, topK):
    """Tiny inputs (at most 1024 list slots and 8192 bitmask words) are scheduled by one
    CTA; the shapes here sit on both sides of that limit, with pads, duplicates, future
    blocks and one invalid id.  (Several query windows are exercised by the workloads of
    test_schedule_matches_oracle: 4 at M3, 16 on the long workload, 32 at fp8.)"""
    rng = np.random.default_rng(N * 100 + topK)
    nb = Lkv // 128
    idx = rng.integers(-1, nb, size=(N, Hkv, topK)).astype(np.int32)
    idx[:, :, 0] = ((Lkv - N + np.arange(N)) // 128)[:, None]
    if topK > 2:
        idx[::2, :, 2] = idx[::2, :, 1]
    idx[0, 0, -1] = nb + 3  # invalid: ignored and flagged
    ref = oracle.schedule(idx, Lkv=Lkv)
    s, exp = gpu_schedule(idx, nb)
    assert exp["status"] & 1 and ref["status"] == 1
    assert_same(exp, ref, N, Lkv)
    s.close()


@pytest.mark.parametrize("N,expected", [(3536, 2), (3537, 1)])
def test_dispatch_at_the_boundary(N, expected):
    """Own-block lists at the tail of 3584 tokens (28 blocks, one KV head): E = N and
    nsb = 28, so 10 E - 13 nsb is 34996 (Q-outer) or 35006 (KV-outer).  The device's AUTO
    choice equals the oracle's on both sides, and the forward it runs matches the oracle."""
    Lkv, nb = 3584, 28
    idx = ((Lkv - N + np.arange(N)) // 128).astype(np.int32).reshape(N, 1, 1)
    ref = oracle.schedule(idx, Lkv=Lkv)
    assert (ref["E"], ref["nsb"]) == (N, nb)
    s, exp = gpu_schedule(idx, nb)
    assert exp["path"] == oracle.dispatch(ref["E"], ref["nsb"]) == expected
    gen = torch.Generator().manual_seed(N)
    Q = torch.randn((N, 16, 128), generator=gen).to(torch.bfloat16)
    K = torch.randn((Lkv, 1, 128), generator=gen).to(torch.bfloat16)
    V = torch.randn((Lkv, 1, 128), generator=gen).to(torch.bfloat16)
    msa = _msa()
    O, LSE = msa.sparse_attn_fwd(Q.cuda(), K.cuda(), V.cuda(), s, scale=0.09)
    torch.cuda.synchronize()
    s.close()
    qids = np.array([0, 1, 127, 128, N // 2, N - 2, N - 1], np.int32)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    Or, Lr, _ = oracle.attn_fwd(bits(Q), bits(K), bits(V), idx, Lkv=Lkv, scale=0.09, qids=qids)
    rel, mabs, lerr = compare_outputs(O.float().cpu().numpy()[qids], LSE.cpu().numpy()[qids], Or, Lr)
    assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS, (rel, mabs, lerr)


def test_schedule_one_pass_scan_ragged():
    """Rows and segments that the chunked scan would take in more than two passes go through
    the one-pass scan (values held in registers, 512 per warp): 3 heads x 3000 blocks =
    9000 rows and 9000 segments, the last warp's share partly filled."""
    rng = np.random.default_rng(11)
    N, Hkv, topK, nb = 300, 3, 5, 3000
    Lkv = nb * 128
    idx = rng.integers(-1, nb, size=(N, Hkv, topK)).astype(np.int32)
    idx[:, :, 0] = ((Lkv - N + np.arange(N)) // 128)[:, None]
    idx[::3, :, 3] = idx[::3, :, 1]
    ref = oracle.schedule(idx, Lkv=Lkv)
    s, exp = gpu_schedule(idx, nb)
    assert exp["status"] == 0
    assert_same(exp, ref, N, Lkv)
    s.close()


@pytest.mark.parametrize("N,expected", [(55, 2), (56, 1)])
def test_host_decided_auto_at_its_bound(N, expected):
    """Where N * Hkv * topK * (10 N - 13) <= 35000 N the sizes alone fix AUTO's choice and the
    forward launches the Q-outer kernel only; at Hkv 4, topK 16 that holds up to N = 55.
    Lists in which every query picks the same 16 blocks make 10 E - 13 nsb as large as it
    can be: 34368 at N = 55 (Q-outer, decided on the host) and 35008 at N = 56 (KV-outer,
    decided on the device).  The device's choice equals the oracle's on both sides, and the
    AUTO forward matches the oracle."""
    Lkv, Hkv, topK = 16384, 4, 16
    idx = np.ascontiguousarray(np.broadcast_to(np.arange(topK, dtype=np.int32), (N, Hkv, topK)))
    ref = oracle.schedule(idx, Lkv=Lkv)
    assert 10 * ref["E"] - 13 * ref["nsb"] == (34368 if N == 55 else 35008)
    s, exp = gpu_schedule(idx, Lkv // 128)
    assert exp["path"] == oracle.dispatch(ref["E"], ref["nsb"]) == expected
    gen = torch.Generator().manual_seed(N)
    Q = torch.randn((N, 16 * Hkv, 128), generator=gen).to(torch.bfloat16)
    K = torch.randn((Lkv, Hkv, 128), generator=gen).to(torch.bfloat16)
    V = torch.randn((Lkv, Hkv, 128), generator=gen).to(torch.bfloat16)
    msa = _msa()
    O, LSE = msa.sparse_attn_fwd(Q.cuda(), K.cuda(), V.cuda(), s, scale=0.09)
    torch.cuda.synchronize()
    assert s.query()["status"] == 0
    s.close()
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    Or, Lr, _ = oracle.attn_fwd(bits(Q), bits(K), bits(V), idx, Lkv=Lkv, scale=0.09)
    rel, mabs, lerr = compare_outputs(O.float().cpu().numpy(), LSE.cpu().numpy(), Or, Lr)
    assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS, (rel, mabs, lerr)
