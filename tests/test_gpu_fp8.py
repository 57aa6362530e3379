"""E4M3 attention parity: O and LSE from libmsa against the fp64 oracle on the same
E4M3 inputs (decoded exactly, descales applied).

The KV-outer kernel reads fp8 data and writes bf16 partial outputs ("Kernel
optimization for MiniMax M3", introduction and bandwidth roofline); per-tensor
descales give the real values.  Tolerances:
relative L2 over O <= 5e-2, max |dLSE| <= 1e-3 (natural log).  Empty lists give
O = 0 and LSE = -inf exactly.
"""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.util import FP8_REL_L2, LSE_MAX_ABS, compare_outputs

pytestmark = pytest.mark.gpu


def _msa():
    import block_sparse_gqa_gb300 as msa
    return msa


def fp8_case(seed, N, Lkv, Hkv, topK, pad_dup=True, sigma=(1.0, 1.0, 1.0)):
    rng = np.random.default_rng(seed)
    nb = Lkv // 128
    Hq = 16 * Hkv
    shapes = [(N, Hq, 128), (Lkv, Hkv, 128), (Lkv, Hkv, 128)]
    xs = [torch.from_numpy((s * rng.standard_normal(sh)).astype(np.float32)) for s, sh in zip(sigma, shapes)]
    (Q, dq), (K, dk), (V, dv) = (workloads.quantize_e4m3(x) for x in xs)
    idx = rng.integers(0, nb, size=(N, Hkv, topK)).astype(np.int32)
    idx[:, :, 0] = ((Lkv - N + np.arange(N)) // 128)[:, None]
    if pad_dup:
        idx[:, :, -1] = -1
        idx[::3, :, 1] = idx[::3, :, 0]
    return Q, K, V, (dq, dk, dv), idx


def run_gpu(Q, K, V, descales, idx, nblocks, scale, path="auto"):
    msa = _msa()
    dev = torch.device("cuda")
    s = msa.build_schedule(torch.from_numpy(np.ascontiguousarray(idx, np.int32)).to(dev), nblocks)
    O, LSE = msa.sparse_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), s, scale=scale, path=path, descales=descales)
    torch.cuda.synchronize()
    st = s.query()
    s.close()
    assert st["status"] & 2 == 0, "device wait timed out"
    return O.float().cpu().numpy(), LSE.cpu().numpy()


def run_oracle(Q, K, V, descales, idx, Lkv, scale, qids=None):
    dq, dk, dv = descales
    O, L, _ = oracle.attn_fwd(Q.numpy(), K.numpy(), V.numpy(), idx, Lkv=Lkv, scale=scale, q_descale=dq,
                              k_descale=dk, v_descale=dv, qids=qids)
    return O, L


def assert_parity(Og, Lg, Or, Lr):
    rel, mabs, lerr = compare_outputs(Og, Lg, Or, Lr)
    assert rel <= FP8_REL_L2 and lerr <= LSE_MAX_ABS, (rel, mabs, lerr)
    return rel, mabs, lerr


@pytest.mark.parametrize("N,Lkv,Hkv,topK", [(2048, 2048, 2, 8), (333, 2048, 1, 5), (1, 1024, 2, 4)])
def test_fp8_random_lists(N, Lkv, Hkv, topK):
    """Pads, duplicates, future blocks, ragged N (high reuse: the KV-outer kernel)."""
    Q, K, V, ds, idx = fp8_case(7 * N + Lkv, N, Lkv, Hkv, topK)
    scale = 1 / math.sqrt(128)
    Og, Lg = run_gpu(Q, K, V, ds, idx, Lkv // 128, scale)
    Or, Lr = run_oracle(Q, K, V, ds, idx, Lkv, scale)
    assert_parity(Og, Lg, Or, Lr)


@pytest.mark.parametrize("N,Lkv,Hkv,topK,sigma,scale", [(2048, 2048, 2, 8, (1.0, 1.0, 1.0), 1 / math.sqrt(128)),
                                                        (333, 2048, 1, 5, (1.0, 1.0, 1.0), 1 / math.sqrt(128)),
                                                        (1024, 4096, 2, 12, (4.0, 3.0, 0.01), 0.5)])
def test_fp8_e4m3_pv_option(N, Lkv, Hkv, topK, sigma, scale):
    """The optional E4M3 P V of the KV-outer kernel (debug_flags bit 1: P rounded to E4M3 in
    shared memory, V transposed per block): within the E4M3 tolerance, with pads,
    duplicates, masked tiles and a sharp softmax."""
    msa = _msa()
    Q, K, V, ds, idx = fp8_case(7 * N + Lkv, N, Lkv, Hkv, topK, sigma=sigma)
    dev = torch.device("cuda")
    s = msa.build_schedule(torch.from_numpy(np.ascontiguousarray(idx, np.int32)).to(dev), Lkv // 128)
    O, LSE = msa.sparse_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), s, scale=scale, path="kv_outer", descales=ds,
                                 debug_flags=2)
    torch.cuda.synchronize()
    assert s.status() == 0
    s.close()
    Or, Lr = run_oracle(Q, K, V, ds, idx, Lkv, scale)
    assert_parity(O.float().cpu().numpy(), LSE.cpu().numpy(), Or, Lr)


def test_fp8_peaked_scores_and_descales():
    """Large score range (sharp softmax) and descales far from 1."""
    Q, K, V, ds, idx = fp8_case(3, 1024, 4096, 2, 12, sigma=(4.0, 3.0, 0.01))
    scale = 0.5
    Og, Lg = run_gpu(Q, K, V, ds, idx, 32, scale)
    Or, Lr = run_oracle(Q, K, V, ds, idx, 4096, scale)
    assert_parity(Og, Lg, Or, Lr)


def test_fp8_empty_lists():
    Q, K, V, ds, idx = fp8_case(5, 512, 512, 1, 3, pad_dup=False)
    idx[:] = -1
    idx[::2, 0, 0] = np.arange(0, 512, 2) // 128
    Og, Lg = run_gpu(Q, K, V, ds, idx, 4, 0.1)
    assert np.all(Og[1::2] == 0) and np.all(np.isneginf(Lg[1::2]))
    Or, Lr = run_oracle(Q, K, V, ds, idx, 512, 0.1)
    assert_parity(Og, Lg, Or, Lr)


def test_fp8_deterministic():
    Q, K, V, ds, idx = fp8_case(11, 1024, 4096, 2, 16, pad_dup=False)
    a = run_gpu(Q, K, V, ds, idx, 32, 0.09)
    b = run_gpu(Q, K, V, ds, idx, 32, 0.09)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


@pytest.mark.parametrize("N,Lkv,Hkv,topK", [(64, 65536, 4, 16), (37, 131072, 2, 9), (1, 16384, 4, 16)])
def test_fp8_low_reuse_q_outer(N, Lkv, Hkv, topK):
    """E4M3 at low reuse (nsb / N far above the crossover): AUTO takes the Q-outer kernel's
    E4M3 instance; forced Q-outer and forced KV-outer give the same answer within the
    E4M3 tolerance, with pads and duplicates in the lists."""
    msa = _msa()
    Q, K, V, ds, idx = fp8_case(13 * N + Lkv, N, Lkv, Hkv, topK)
    scale = 1 / math.sqrt(128)
    dev = torch.device("cuda")
    s = msa.build_schedule(torch.from_numpy(np.ascontiguousarray(idx, np.int32)).to(dev), Lkv // 128)
    assert s.query()["path"] == 2  # the device chose Q-outer
    s.close()
    Or, Lr = run_oracle(Q, K, V, ds, idx, Lkv, scale)
    for path in ("auto", "q_outer", "kv_outer"):
        Og, Lg = run_gpu(Q, K, V, ds, idx, Lkv // 128, scale, path=path)
        assert_parity(Og, Lg, Or, Lr)


def test_fp8_q_outer_sharp_and_empty():
    """Forced Q-outer on E4M3: a sharp softmax with descales far from 1, and empty lists
    (O = 0, LSE = -inf)."""
    Q, K, V, ds, idx = fp8_case(17, 512, 4096, 2, 12, sigma=(4.0, 3.0, 0.01))
    idx[5::7] = -1
    Og, Lg = run_gpu(Q, K, V, ds, idx, 32, 0.5, path="q_outer")
    assert np.all(Og[5::7] == 0) and np.all(np.isneginf(Lg[5::7]))
    Or, Lr = run_oracle(Q, K, V, ds, idx, 4096, 0.5)
    assert_parity(Og, Lg, Or, Lr)


def test_fp8_rejects_bad_descales():
    msa = _msa()
    Q, K, V, ds, idx = fp8_case(1, 256, 1024, 1, 4)
    dev = torch.device("cuda")
    s = msa.build_schedule(torch.from_numpy(idx).to(dev), 8)
    Qd, Kd, Vd = Q.to(dev), K.to(dev), V.to(dev)
    for bad in ((0.0, 1.0, 1.0), (1.0, -1.0, 1.0), (1.0, 1.0, float("nan"))):
        with pytest.raises(msa.MsaError) as e:
            msa.sparse_attn_fwd(Qd, Kd, Vd, s, descales=bad)
        assert e.value.status == 1  # MSA_ERR_INVALID_ARG
    with pytest.raises(msa.MsaError) as e:  # mixed dtypes
        msa.sparse_attn_fwd(Qd, Kd.view(torch.uint8).to(torch.bfloat16), Vd, s, descales=ds)
    assert e.value.status == 2
    s.close()


def test_fp8_full_size_sampled():
    """The E4M3 workload (N = Lkv = 65536, Gaussian-local picks) at full size, sampled queries."""
    wl = workloads.make_workload("fp8")
    cfg = wl.cfg
    ds = (wl.q_descale, wl.k_descale, wl.v_descale)
    Og, Lg = run_gpu(wl.Q, wl.K, wl.V, ds, wl.indices.numpy(), cfg.nblocks, cfg.scale)
    qids = workloads.sample_queries(cfg, 96)
    Or, Lr = run_oracle(wl.Q, wl.K, wl.V, ds, wl.indices.numpy(), cfg.Lkv, cfg.scale, qids=qids)
    assert_parity(Og[qids], Lg[qids], Or, Lr)
