"""Block selectors R1 and R4: the GPU lists against the fp64 oracle.

"Sparse Attention" (dinara-dl), Chapter 4, "R1: One Representative" and "R4: Four
Representatives".  Floating point
decides which blocks are chosen and the GPU scores in fp32 while the oracle scores in
fp64, so lists are compared where the choice is unique and checked for validity where
near-ties make several lists correct: the own blocks come first, every entry is a
candidate, no entry repeats, padding only after the candidates run out, and the chosen
set is a top-K set of the oracle's scores within a tolerance derived from fp32
rounding of the means and dot products.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads

pytestmark = pytest.mark.gpu


def _msa():
    import block_sparse_gqa_gb300 as msa
    return msa


def bf16(rng, shape, scale=1.0):
    return torch.from_numpy((scale * rng.standard_normal(shape)).astype(np.float32)).to(torch.bfloat16)


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def check_lists(got, want, scores, N, Lkv, topK):
    """got/want [N, Hkv, topK]; scores [ntiles, Hkv, nblocks] from the oracle."""
    ntiles, Hkv, nblocks = scores.shape
    exact = 0
    for t in range(ntiles):
        i0, i1 = 128 * t, min(128 * t + 128, N)
        assert np.all(got[i0:i1] == got[i0]), "every query of a tile shares its list"
        for g in range(Hkv):
            sc = scores[t, g]
            lg, lw = got[i0, g], want[i0, g]
            finite = sc[np.isfinite(sc)]
            tol = 1e-4 * max(1.0, float(np.abs(finite).max()) if finite.size else 1.0)
            cand = np.flatnonzero(~np.isneginf(sc))
            n = min(topK, cand.size)
            assert np.all(lg[n:] == -1) and np.all(lg[:n] >= 0)
            sel = lg[:n]
            assert len(set(sel.tolist())) == n and np.all(~np.isneginf(sc[sel]))
            forced = np.flatnonzero(np.isposinf(sc))
            assert list(sel[:len(forced)]) == sorted(forced.tolist())
            rest = np.setdiff1d(cand, sel)
            if rest.size and n:
                assert sc[sel].min() >= sc[rest].max() - tol
            assert np.all(np.diff(np.where(np.isposinf(sc[sel]), 1e300, sc[sel])) <= tol)
            # unique where the k-th and (k+1)-th oracle scores are further apart than tol
            order = sorted(cand.tolist(), key=lambda b: (-sc[b], b))
            vals = [sc[b] for b in order] + [-np.inf]
            if all(np.isposinf(vals[k]) or vals[k] - vals[k + 1] > tol for k in range(n)):
                assert np.array_equal(lg, lw)
                exact += 1
    return exact


SELECTORS = {"r1": ("select_blocks_r1", oracle.select_r1), "r4": ("select_blocks_r4", oracle.select_r4)}


@pytest.mark.parametrize("sel", ["r1", "r4"])
@pytest.mark.parametrize("N,Lkv,Hkv,topK", [(1024, 1024, 1, 4), (300, 2048, 2, 8), (2048, 8192, 4, 16), (5, 4096, 1, 64),
                                            (170, 1024, 1, 6)])
def test_select_matches_oracle(sel, N, Lkv, Hkv, topK):
    """Ragged last tiles (N = 300: 44 queries, N = 170: 42, N = 5) leave R4 quarters empty."""
    rng = np.random.default_rng(N + Lkv + topK)
    Q, K = bf16(rng, (N, 16 * Hkv, 128)), bf16(rng, (Lkv, Hkv, 128))
    dev = torch.device("cuda")
    entry, ref = SELECTORS[sel]
    got = getattr(_msa(), entry)(Q.to(dev), K.to(dev), topK).cpu().numpy()
    want, scores = ref(bits(Q), bits(K), Lkv=Lkv, topK=topK)
    exact = check_lists(got, want, scores, N, Lkv, topK)
    assert exact >= 1


def test_select_r4_finds_quarter_on_gpu():
    """A block whose mean key is zero but whose first quarter points along the queries:
    R4 (GPU) ranks it first after the own block, R1 (GPU) does not choose it."""
    rng = np.random.default_rng(23)
    N, Lkv = 128, 1024
    Q = np.zeros((N, 16, 128), np.float32); Q[:, :, 0] = 1.0
    K = (0.01 * rng.standard_normal((Lkv, 1, 128))).astype(np.float32)
    K[:, :, 0] = 0.1 * np.abs(rng.standard_normal((Lkv, 1)))
    K[256:288, :, 0] = 6.0
    K[288:384, :, 0] = -2.0
    K[256:384, :, 1:] = 0.0
    dev = torch.device("cuda")
    Qt, Kt = (torch.from_numpy(x).to(torch.bfloat16).to(dev) for x in (Q, K))
    l4 = _msa().select_blocks_r4(Qt, Kt, 3).cpu().numpy()
    l1 = _msa().select_blocks_r1(Qt, Kt, 3).cpu().numpy()
    assert l4[0, 0, 0] == 7 and l4[0, 0, 1] == 2 and 2 not in l1[0, 0].tolist()


@pytest.mark.parametrize("sel", ["r1", "r4"])
def test_select_m3_shape_and_pipeline(sel):
    """M3 shape: the lists feed the schedule and the attention, whose output matches
    the oracle on the same lists (sampled queries)."""
    msa = _msa()
    cfg = workloads.CONFIGS["m3"]
    wl = workloads.make_workload(cfg)
    dev = torch.device("cuda")
    Q, K, V = (t.to(dev) for t in (wl.Q, wl.K, wl.V))
    entry, ref = SELECTORS[sel]
    idx = getattr(msa, entry)(Q, K, cfg.topK)
    got = idx.cpu().numpy()
    want, scores = ref(bits(wl.Q), bits(wl.K), Lkv=cfg.Lkv, topK=cfg.topK)
    check_lists(got, want, scores, cfg.N, cfg.Lkv, cfg.topK)
    s = msa.build_schedule(idx, cfg.nblocks)
    O, L = msa.sparse_attn_fwd(Q, K, V, s, scale=cfg.scale)
    torch.cuda.synchronize()
    assert s.query()["status"] == 0
    s.close()
    qids = workloads.sample_queries(cfg, 64)
    Or, Lr, _ = oracle.attn_fwd(bits(wl.Q), bits(wl.K), bits(wl.V), got, Lkv=cfg.Lkv, scale=cfg.scale, qids=qids)
    Og = O.float().cpu().numpy()[qids]
    rel = np.linalg.norm(Og - Or) / np.linalg.norm(Or)
    assert rel <= 1e-2 and np.abs(L.cpu().numpy()[qids] - Lr).max() <= 1e-3


def test_select_rejects_bad_arguments():
    msa = _msa()
    dev = torch.device("cuda")
    Q = torch.zeros((128, 16, 128), dtype=torch.bfloat16, device=dev)
    K = torch.zeros((256, 1, 128), dtype=torch.bfloat16, device=dev)
    with pytest.raises(msa.MsaError) as e:
        msa.select_blocks_r1(Q, K, 65)
    assert e.value.status == 2
    with pytest.raises(msa.MsaError) as e:
        msa.select_blocks_r1(Q, K[:200], 4)  # Lkv not a multiple of 128
    assert e.value.status == 1
    with pytest.raises(msa.MsaError) as e:
        msa.select_blocks_r1(Q, K, 4, workspace=torch.empty(16, dtype=torch.uint8, device=dev))
    assert e.value.status == 1
    with pytest.raises(msa.MsaError) as e:
        msa.select_blocks_r4(Q, K, 65)
    assert e.value.status == 2
