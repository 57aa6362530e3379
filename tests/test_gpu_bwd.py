"""Backward parity: dQ, dK, dV from libmsa against the fp64 oracle.

"Flash-MSA: accelerating million-token training with sparse attention", order of
operations: the forward's block indices and log-sum-exp are kept for the backward,
which takes the main-attention gradients over the same blocks.  The library runs its
own forward first (O, LSE) and feeds them to the backward, so the comparison covers
the whole training-step path; the oracle takes the exact gradients of the forward's
definition.  Tolerance: relative L2 <= 2e-2 per gradient tensor; exact zeros where no
query sees a key (dK, dV) and for queries without entries (dQ).
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.util import BWD_REL_L2, rel_l2

pytestmark = pytest.mark.gpu


def _msa():
    import block_sparse_gqa_gb300 as msa
    return msa


def bf16(rng, shape, sigma=1.0):
    return torch.from_numpy((sigma * rng.standard_normal(shape)).astype(np.float32)).to(torch.bfloat16)


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def run_gpu(Q, K, V, dO, idx, nblocks, scale):
    msa = _msa()
    dev = torch.device("cuda")
    s = msa.build_schedule(torch.from_numpy(np.ascontiguousarray(idx, np.int32)).to(dev), nblocks)
    Qd, Kd, Vd, dOd = (t.to(dev) for t in (Q, K, V, dO))
    O, LSE = msa.sparse_attn_fwd(Qd, Kd, Vd, s, scale=scale)
    dQ, dK, dV = msa.sparse_attn_bwd(Qd, Kd, Vd, O, dOd, LSE, s, scale=scale)
    torch.cuda.synchronize()
    st = s.query()
    s.close()
    assert st["status"] & 2 == 0, "device wait timed out"
    return tuple(t.float().cpu().numpy() for t in (dQ, dK, dV))


def lists(rng, N, Lkv, Hkv, topK, extras=True):
    nb = Lkv // 128
    idx = rng.integers(0, nb, size=(N, Hkv, topK)).astype(np.int32)  # future blocks included
    idx[:, :, 0] = ((Lkv - N + np.arange(N)) // 128)[:, None]
    if extras:
        idx[::3, :, -1] = -1
        idx[1::4, :, 1 % topK] = idx[1::4, :, 0]
    return idx


def check(got, ref, tol=BWD_REL_L2):
    errs = [rel_l2(g, r) for g, r in zip(got, ref)]
    assert max(errs) <= tol, errs
    return errs


@pytest.mark.parametrize("N,Lkv,Hkv,topK", [(1024, 1024, 1, 4), (333, 2048, 2, 5), (2048, 2048, 2, 8)])
def test_bwd_random_lists(N, Lkv, Hkv, topK):
    """Pads, duplicates, future blocks, ragged N and tiles; rows long enough for several
    units (at most 256 entries each)."""
    rng = np.random.default_rng(N + Lkv + topK)
    Q, K, V, dO = bf16(rng, (N, 16 * Hkv, 128)), bf16(rng, (Lkv, Hkv, 128)), bf16(rng, (Lkv, Hkv, 128)), \
        bf16(rng, (N, 16 * Hkv, 128))
    idx = lists(rng, N, Lkv, Hkv, topK)
    scale = 128 ** -0.5
    got = run_gpu(Q, K, V, dO, idx, Lkv // 128, scale)
    ref = oracle.attn_bwd(bits(Q), bits(K), bits(V), bits(dO), idx, Lkv=Lkv, scale=scale)[:3]
    print("rel-L2 dQ dK dV", check(got, ref))


def test_bwd_sharp_scores():
    """Large score range (sharp softmax) and a scale far from 1/sqrt(D)."""
    rng = np.random.default_rng(11)
    N, Lkv, Hkv, topK = 512, 1024, 1, 6
    Q, K, V, dO = bf16(rng, (N, 16, 128), 2.0), bf16(rng, (Lkv, 1, 128), 2.0), bf16(rng, (Lkv, 1, 128)), \
        bf16(rng, (N, 16, 128), 0.1)
    idx = lists(rng, N, Lkv, Hkv, topK)
    got = run_gpu(Q, K, V, dO, idx, Lkv // 128, 0.3)
    ref = oracle.attn_bwd(bits(Q), bits(K), bits(V), bits(dO), idx, Lkv=Lkv, scale=0.3)[:3]
    print("rel-L2 dQ dK dV", check(got, ref))


def test_bwd_empty_queries_and_blocks():
    """Queries whose lists are all padding get dQ = 0; keys no query sees get dK = dV = 0."""
    rng = np.random.default_rng(5)
    N, Lkv, Hkv, topK = 640, 1024, 2, 3
    Q, K, V, dO = bf16(rng, (N, 32, 128)), bf16(rng, (Lkv, 2, 128)), bf16(rng, (Lkv, 2, 128)), bf16(rng, (N, 32, 128))
    idx = lists(rng, N, Lkv, Hkv, topK, extras=False)
    idx[idx == 2] = 3          # block 2 is never selected ...
    idx[::5] = -1              # ... and every fifth query selects nothing
    scale = 128 ** -0.5
    dQ, dK, dV = run_gpu(Q, K, V, dO, idx, Lkv // 128, scale)
    assert np.all(dQ[::5] == 0)
    assert np.all(dK[256:384] == 0) and np.all(dV[256:384] == 0)
    ref = oracle.attn_bwd(bits(Q), bits(K), bits(V), bits(dO), idx, Lkv=Lkv, scale=scale)[:3]
    check((dQ, dK, dV), ref)


def test_bwd_deterministic():
    rng = np.random.default_rng(9)
    N, Lkv, Hkv, topK = 1024, 2048, 2, 8
    Q, K, V, dO = bf16(rng, (N, 32, 128)), bf16(rng, (Lkv, 2, 128)), bf16(rng, (Lkv, 2, 128)), bf16(rng, (N, 32, 128))
    idx = lists(rng, N, Lkv, Hkv, topK)
    a = run_gpu(Q, K, V, dO, idx, Lkv // 128, 0.09)
    b = run_gpu(Q, K, V, dO, idx, Lkv // 128, 0.09)
    for x, y in zip(a, b):
        assert np.array_equal(x, y)


def test_bwd_m3_sampled():
    """The M3 shape (N = Lkv = 8192, Hq 64, Hkv 4, topK 16, uniform picks) at full size:
    dQ of sampled queries, dK and dV of sampled (group, block) rows, including the last
    block (masked) and an early, heavily selected block."""
    wl = workloads.make_workload("m3")
    cfg = wl.cfg
    rng = np.random.default_rng(42)
    dO = bf16(rng, (cfg.N, cfg.Hq, cfg.D))
    dQ, dK, dV = run_gpu(wl.Q, wl.K, wl.V, dO, wl.indices.numpy(), cfg.nblocks, cfg.scale)
    qids = workloads.sample_queries(cfg, 48)
    rows = np.array([0 * cfg.nblocks + 63, 1 * cfg.nblocks + 30, 3 * cfg.nblocks + 5], np.int32)
    Qb, Kb, Vb = wl.np_inputs()
    rQ, rK, rV, _ = oracle.attn_bwd(Qb, Kb, Vb, bits(dO), wl.indices.numpy(), Lkv=cfg.Lkv, scale=cfg.scale,
                                    qids=qids, rows=rows)
    gK = np.stack([dK[(r % cfg.nblocks) * 128:(r % cfg.nblocks + 1) * 128, r // cfg.nblocks] for r in rows])
    gV = np.stack([dV[(r % cfg.nblocks) * 128:(r % cfg.nblocks + 1) * 128, r // cfg.nblocks] for r in rows])
    print("rel-L2 dQ dK dV", check((dQ[qids], gK, gV), (rQ, rK, rV)))


def test_bwd_rejects_unsupported():
    msa = _msa()
    dev = torch.device("cuda")
    rng = np.random.default_rng(1)
    N, Lkv = 256, 512
    idx = torch.from_numpy(lists(rng, N, Lkv, 1, 2)).to(dev)
    s = msa.build_schedule(idx, Lkv // 128)
    Q, K, V, dO = (bf16(rng, sh).to(dev) for sh in [(N, 16, 128), (Lkv, 1, 128), (Lkv, 1, 128), (N, 16, 128)])
    O, LSE = msa.sparse_attn_fwd(Q, K, V, s)
    with pytest.raises(msa.MsaError) as e:  # E4M3 inputs
        msa.sparse_attn_bwd(Q.view(torch.uint8)[:, :, :128].contiguous(), K, V, O, dO, LSE, s)
    assert e.value.status in (1, 2)
    with pytest.raises(msa.MsaError) as e:  # K does not match the schedule
        msa.sparse_attn_bwd(Q, K[:384].contiguous(), V[:384].contiguous(), O, dO, LSE, s)
    assert e.value.status == 1
    s.close()


def test_bwd_long_sampled():
    """The long workload (N = 32768 at the tail of Lkv = 131072, lists shared by runs of 64
    queries, Zipf-weighted picks) at full size: dQ of sampled queries, dK and dV of the two
    last blocks of groups 0 and 3 (the own blocks of the last queries, masked)."""
    wl = workloads.make_workload("long")
    cfg = wl.cfg
    rng = np.random.default_rng(43)
    dO = bf16(rng, (cfg.N, cfg.Hq, cfg.D))
    dQ, dK, dV = run_gpu(wl.Q, wl.K, wl.V, dO, wl.indices.numpy(), cfg.nblocks, cfg.scale)
    qids = workloads.sample_queries(cfg, 32)
    nb = cfg.nblocks
    rows = np.array([0 * nb + nb - 1, 0 * nb + nb - 2, 3 * nb + nb - 1], np.int32)
    Qb, Kb, Vb = wl.np_inputs()
    rQ, rK, rV, _ = oracle.attn_bwd(Qb, Kb, Vb, bits(dO), wl.indices.numpy(), Lkv=cfg.Lkv, scale=cfg.scale,
                                    qids=qids, rows=rows)
    gK = np.stack([dK[(r % nb) * 128:(r % nb + 1) * 128, r // nb] for r in rows])
    gV = np.stack([dV[(r % nb) * 128:(r % nb + 1) * 128, r // nb] for r in rows])
    print("rel-L2 dQ dK dV", check((dQ[qids], gK, gV), (rQ, rK, rV)))
