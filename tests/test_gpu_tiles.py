"""Shared-list forward (msa_sparse_attn_fwd_tiles) against the fp64 oracle.

"Sparse Attention" (dinara-dl), Chapters 3-4: lists chosen per tile of consecutive
queries and GQA group; per query the result is the plain definition on the expanded
per-query lists (the oracle evaluates exactly those).  Tolerances as for bf16
elsewhere: relative L2 over O <= 1e-2, max |dO| <= 2e-2, max |dLSE| <= 1e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.util import BF16_MAX_ABS, BF16_REL_L2, LSE_MAX_ABS, compare_outputs

pytestmark = pytest.mark.gpu


def _msa():
    import block_sparse_gqa_gb300 as msa
    return msa


def bf16(rng, shape):
    return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def tile_case(seed, N, Lkv, Hkv, topK, tile, extras=True):
    rng = np.random.default_rng(seed)
    nb = Lkv // 128
    Q, K, V = bf16(rng, (N, 16 * Hkv, 128)), bf16(rng, (Lkv, Hkv, 128)), bf16(rng, (Lkv, Hkv, 128))
    nt = -(-N // tile)
    lists = rng.integers(0, nb, size=(nt, Hkv, topK)).astype(np.int32)
    for t in range(nt):  # the own block of the tile's last query first
        last = min(tile * t + tile - 1, N - 1)
        lists[t, :, 0] = (Lkv - N + last) // 128
    if extras:
        lists[:, :, -1] = -1
        lists[::2, :, 1] = lists[::2, :, 0]  # duplicate
    return Q, K, V, lists


def run(Q, K, V, lists, tile, scale, status=None):
    dev = torch.device("cuda")
    O, L = _msa().sparse_attn_fwd_tiles(Q.to(dev), K.to(dev), V.to(dev), torch.from_numpy(lists).to(dev), tile,
                                        scale=scale, status=status)
    torch.cuda.synchronize()
    return O.float().cpu().numpy(), L.cpu().numpy()


def expand(lists, N, tile):
    return np.ascontiguousarray(np.repeat(lists, tile, axis=0)[:N])


@pytest.mark.parametrize("N,Lkv,Hkv,topK,tile", [(1024, 1024, 1, 4, 128), (333, 2048, 2, 8, 16), (2048, 4096, 2, 16, 64),
                                                 (17, 1024, 1, 3, 16), (1, 512, 1, 2, 16)])
def test_tiles_match_oracle(N, Lkv, Hkv, topK, tile):
    Q, K, V, lists = tile_case(N + Lkv + tile, N, Lkv, Hkv, topK, tile)
    Og, Lg = run(Q, K, V, lists, tile, 1 / np.sqrt(128))
    Or, Lr, _ = oracle.attn_fwd(bits(Q), bits(K), bits(V), expand(lists, N, tile), Lkv=Lkv, scale=1 / np.sqrt(128))
    rel, mabs, lerr = compare_outputs(Og, Lg, Or, Lr)
    assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS, (rel, mabs, lerr)


def test_tiles_sharp_scores_and_negative_scale():
    """Large score range (rescale path) and a negative scale (row minimum)."""
    Q, K, V, lists = tile_case(7, 512, 2048, 1, 8, 32, extras=False)
    for scale in (0.9, -0.3):
        Og, Lg = run(Q, K, V, lists, 32, scale)
        Or, Lr, _ = oracle.attn_fwd(bits(Q), bits(K), bits(V), expand(lists, 512, 32), Lkv=2048, scale=scale)
        rel, mabs, lerr = compare_outputs(Og, Lg, Or, Lr)
        assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS, (scale, rel, mabs, lerr)


def test_tiles_empty_lists_and_bad_ids():
    Q, K, V, lists = tile_case(9, 256, 1024, 1, 4, 16, extras=False)
    lists[1] = -1                # queries 16..31: no blocks at all
    lists[2, 0, 1] = 99          # invalid id: ignored, flagged
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    Og, Lg = run(Q, K, V, lists, 16, 0.1, status=status)
    assert np.all(Og[16:32] == 0) and np.all(np.isneginf(Lg[16:32]))
    assert int(status.item()) & 1 == 1
    ref = lists.copy()
    ref[2, 0, 1] = -1
    Or, Lr, _ = oracle.attn_fwd(bits(Q), bits(K), bits(V), expand(ref, 256, 16), Lkv=1024, scale=0.1)
    rel, mabs, lerr = compare_outputs(Og, Lg, Or, Lr)
    assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS


def test_tiles_equal_kv_outer_on_shared_lists():
    """M3 shape with R1 selector lists (shared per 128-query tile): the shared-list forward
    and the general path agree, and sampled queries match the oracle."""
    msa = _msa()
    cfg = workloads.CONFIGS["m3"]
    wl = workloads.make_workload(cfg)
    dev = torch.device("cuda")
    Q, K, V = (t.to(dev) for t in (wl.Q, wl.K, wl.V))
    idx = msa.select_blocks_r1(Q, K, cfg.topK)
    lists = idx[::128].contiguous()
    Ot, Lt = msa.sparse_attn_fwd_tiles(Q, K, V, lists, 128, scale=cfg.scale)
    s = msa.build_schedule(idx, cfg.nblocks)
    Ok, Lk = msa.sparse_attn_fwd(Q, K, V, s, scale=cfg.scale)
    torch.cuda.synchronize()
    s.close()
    a, b = Ot.float(), Ok.float()
    assert (torch.linalg.norm(a - b) / torch.linalg.norm(b)).item() <= BF16_REL_L2
    assert (Lt - Lk).abs().max().item() <= LSE_MAX_ABS
    qids = workloads.sample_queries(cfg, 48)
    Or, Lr, _ = oracle.attn_fwd(bits(wl.Q), bits(wl.K), bits(wl.V), idx.cpu().numpy(), Lkv=cfg.Lkv, scale=cfg.scale,
                                qids=qids)
    rel, mabs, lerr = compare_outputs(Ot.float().cpu().numpy()[qids], Lt.cpu().numpy()[qids], Or, Lr)
    assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS


def test_tiles_rejects_bad_arguments():
    msa = _msa()
    dev = torch.device("cuda")
    Q = torch.zeros((64, 16, 128), dtype=torch.bfloat16, device=dev)
    K = torch.zeros((256, 1, 128), dtype=torch.bfloat16, device=dev)
    lists = torch.zeros((4, 1, 2), dtype=torch.int32, device=dev)
    with pytest.raises(msa.MsaError) as e:
        msa.sparse_attn_fwd_tiles(Q, K, K, lists, 24)  # tile not a multiple of 16
    assert e.value.status == 1
    with pytest.raises(msa.MsaError) as e:
        msa.sparse_attn_fwd_tiles(Q, K, K, torch.zeros((4, 1, 65), dtype=torch.int32, device=dev), 16)
    assert e.value.status == 2
