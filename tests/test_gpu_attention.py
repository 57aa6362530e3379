"""Attention parity: O and LSE from libmsa against the fp64 oracle.

Tolerances for bf16 inputs: relative L2 over O <= 1e-2, max |dO| <= 2e-2,
max |dLSE| <= 1e-3 (natural log).  Softmax over the union of selected blocks
("Sparse Attention", Ch. 1); local block causally masked ("Flash-MSA");
KV-outer partials + LSE combine and the Q-outer alternative ("Kernel optimization
for MiniMax M3"; "Sparse Attention", Ch. 5: both organisations compute the same
attention).
"""
import math

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


def run_gpu(Q, K, V, idx, nblocks, scale, path="auto"):
    msa = _msa()
    dev = torch.device("cuda")
    s = msa.build_schedule(torch.from_numpy(np.ascontiguousarray(idx, np.int32)).to(dev), nblocks)
    O, LSE = msa.sparse_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), s, scale=scale, path=path)
    torch.cuda.synchronize()
    st = s.query()
    s.close()
    assert st["status"] & 2 == 0, "device wait timed out"
    return O.float().cpu().numpy(), LSE.cpu().numpy(), st


def run_oracle(Q, K, V, idx, Lkv, scale, qids=None):
    bits = [t.view(torch.int16).numpy().view(np.uint16) for t in (Q, K, V)]
    O, L, _ = oracle.attn_fwd(*bits, idx, Lkv=Lkv, scale=scale, qids=qids)
    return O, L


def assert_parity(Og, Lg, Or, Lr, rel_tol=BF16_REL_L2):
    rel, mabs, lerr = compare_outputs(Og, Lg, Or, Lr)
    assert rel <= rel_tol and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS, (rel, mabs, lerr)
    return rel, mabs, lerr


def test_tiny_all_queries():
    wl = workloads.make_workload("tiny")
    cfg = wl.cfg
    Or, Lr = run_oracle(wl.Q, wl.K, wl.V, wl.indices.numpy(), cfg.Lkv, cfg.scale)
    ref = oracle.schedule(wl.indices.numpy(), Lkv=cfg.Lkv)
    for path in ("auto", "kv_outer", "q_outer"):
        Og, Lg, st = run_gpu(wl.Q, wl.K, wl.V, wl.indices.numpy(), cfg.nblocks, cfg.scale, path=path)
        assert st["path"] == oracle.dispatch(ref["E"], ref["nsb"])  # the device's AUTO choice
        assert_parity(Og, Lg, Or, Lr)


def random_case(seed, N, Lkv, Hkv, topK, pad_dup=True):
    rng = np.random.default_rng(seed)
    nb = Lkv // 128
    Hq = 16 * Hkv
    Q, K, V = bf16(rng, (N, Hq, 128)), bf16(rng, (Lkv, Hkv, 128)), bf16(rng, (Lkv, Hkv, 128))
    idx = rng.integers(0, nb, size=(N, Hkv, topK)).astype(np.int32)
    lb = (Lkv - N + np.arange(N)) // 128
    idx[:, :, 0] = lb[:, None]
    if pad_dup:
        idx[:, :, -1] = -1
        idx[::3, :, 1] = idx[::3, :, 0]  # duplicate of the local block
    return Q, K, V, idx


@pytest.mark.parametrize("N,Lkv,Hkv,topK", [(2048, 2048, 2, 8), (333, 2048, 1, 5), (1, 1024, 2, 4)])
def test_random_lists_both_paths(N, Lkv, Hkv, topK):
    """Pads, duplicates, future blocks, ragged N; KV-outer and Q-outer forced in turn."""
    Q, K, V, idx = random_case(N + Lkv, N, Lkv, Hkv, topK)
    scale = 1 / math.sqrt(128)
    Or, Lr = run_oracle(Q, K, V, idx, Lkv, scale)
    for path in ("kv_outer", "q_outer"):
        Og, Lg, _ = run_gpu(Q, K, V, idx, Lkv // 128, scale, path=path)
        assert_parity(Og, Lg, Or, Lr)


def test_empty_lists_give_zero_and_neg_inf():
    rng = np.random.default_rng(5)
    N = Lkv = 512
    Q, K, V = bf16(rng, (N, 16, 128)), bf16(rng, (Lkv, 1, 128)), bf16(rng, (Lkv, 1, 128))
    idx = np.full((N, 1, 3), -1, np.int32)
    idx[::2, 0, 0] = (np.arange(0, N, 2)) // 128  # only even queries have a block
    for path in ("kv_outer", "q_outer"):
        Og, Lg, _ = run_gpu(Q, K, V, idx, Lkv // 128, 0.1, path=path)
        assert np.all(Og[1::2] == 0) and np.all(np.isneginf(Lg[1::2]))
        Or, Lr = run_oracle(Q, K, V, idx, Lkv, 0.1)
        assert_parity(Og, Lg, Or, Lr)


def test_paths_agree_and_deterministic():
    Q, K, V, idx = random_case(11, 1024, 4096, 2, 16, pad_dup=False)
    a = run_gpu(Q, K, V, idx, 32, 0.09, path="kv_outer")
    b = run_gpu(Q, K, V, idx, 32, 0.09, path="kv_outer")
    c = run_gpu(Q, K, V, idx, 32, 0.09, path="q_outer")
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    rel = np.linalg.norm(a[0] - c[0]) / np.linalg.norm(c[0])
    assert rel <= BF16_REL_L2 and np.abs(a[1] - c[1]).max() <= LSE_MAX_ABS


@pytest.mark.parametrize("name,nq", [("m3", 192), ("lowreuse", 64), ("long", 96)])
def test_full_size_sampled(name, nq):
    """Full-size workloads in the benchmark's launch configuration, sampled queries."""
    wl = workloads.make_workload(name)
    cfg = wl.cfg
    Og, Lg, st = run_gpu(wl.Q, wl.K, wl.V, wl.indices.numpy(), cfg.nblocks, cfg.scale)
    assert st["path"] == (2 if name == "lowreuse" else 1)
    qids = workloads.sample_queries(cfg, nq)
    Or, Lr = run_oracle(wl.Q, wl.K, wl.V, wl.indices.numpy(), cfg.Lkv, cfg.scale, qids=qids)
    assert_parity(Og[qids], Lg[qids], Or, Lr)
