"""fp32 partial outputs ("Sparse Attention", Chapter 5, "Partial outputs and Combine": the
partials' format is the main data-movement cost of the KV-outer path; the chapter times
the same kernel with fp32 and with bf16 partials).

The library's opt-in fp32 partials keep each block's P V sum unrounded until the combine;
the output is bf16 either way.  Parity against the fp64 oracle with the bf16 tolerances;
at the M3 shape the fp32 format must be at least as accurate as bf16 partials; a
schedule whose workspace was sized for fp32 serves bf16 forwards and the backward.
"""
import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.util import BF16_MAX_ABS, BF16_REL_L2, BWD_REL_L2, LSE_MAX_ABS, compare_outputs, rel_l2

pytestmark = pytest.mark.gpu


def _msa():
    import block_sparse_gqa_gb300 as msa
    return msa


def bf16(rng, shape):
    return torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def lists(rng, N, Lkv, Hkv, topK):
    idx = rng.integers(0, Lkv // 128, size=(N, Hkv, topK)).astype(np.int32)
    idx[:, :, 0] = ((Lkv - N + np.arange(N)) // 128)[:, None]
    idx[::3, :, -1] = -1
    idx[1::4, :, 1] = idx[1::4, :, 0]
    return idx


@pytest.mark.parametrize("N,Lkv,Hkv,topK", [(2048, 2048, 2, 8), (333, 2048, 1, 5)])
def test_fp32_partials_random_lists(N, Lkv, Hkv, topK):
    msa = _msa()
    dev = torch.device("cuda")
    rng = np.random.default_rng(N + topK)
    Q, K, V = bf16(rng, (N, 16 * Hkv, 128)), bf16(rng, (Lkv, Hkv, 128)), bf16(rng, (Lkv, Hkv, 128))
    idx = lists(rng, N, Lkv, Hkv, topK)
    s = msa.build_schedule(torch.from_numpy(idx).to(dev), Lkv // 128)
    O, LSE = msa.sparse_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), s, path="kv_outer", partials_fp32=True)
    torch.cuda.synchronize()
    assert s.query()["status"] == 0
    s.close()
    Or, Lr, _ = oracle.attn_fwd(bits(Q), bits(K), bits(V), idx, Lkv=Lkv, scale=128 ** -0.5)
    rel, mabs, lerr = compare_outputs(O.float().cpu().numpy(), LSE.cpu().numpy(), Or, Lr)
    assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS, (rel, mabs, lerr)


def test_fp32_partials_m3_more_accurate_and_workspace_reuse():
    """M3 at full size: fp32 partials are at least as accurate as bf16 partials on sampled
    queries; the fp32-sized workspace then serves a bf16 forward (bit-identical to a fresh
    schedule's) and the backward."""
    msa = _msa()
    dev = torch.device("cuda")
    wl = workloads.make_workload("m3")
    cfg = wl.cfg
    idx = wl.indices.to(dev)
    Q, K, V = (t.to(dev) for t in (wl.Q, wl.K, wl.V))
    s = msa.build_schedule(idx, cfg.nblocks)
    O32, L32 = msa.sparse_attn_fwd(Q, K, V, s, scale=cfg.scale, partials_fp32=True)
    O16, L16 = msa.sparse_attn_fwd(Q, K, V, s, scale=cfg.scale)
    s2 = msa.build_schedule(idx, cfg.nblocks)
    Of, Lf = msa.sparse_attn_fwd(Q, K, V, s2, scale=cfg.scale)
    torch.cuda.synchronize()
    assert torch.equal(O16, Of) and torch.equal(L16, Lf)
    s2.close()
    qids = workloads.sample_queries(cfg, 96)
    Qb, Kb, Vb = wl.np_inputs()
    Or, Lr, _ = oracle.attn_fwd(Qb, Kb, Vb, wl.indices.numpy(), Lkv=cfg.Lkv, scale=cfg.scale, qids=qids)
    e32 = compare_outputs(O32.float().cpu().numpy()[qids], L32.cpu().numpy()[qids], Or, Lr)
    e16 = compare_outputs(O16.float().cpu().numpy()[qids], L16.cpu().numpy()[qids], Or, Lr)
    print("rel-L2 / max-abs / LSE: fp32 partials", e32, "bf16 partials", e16)
    assert e32[0] <= BF16_REL_L2 and e32[1] <= BF16_MAX_ABS and e32[2] <= LSE_MAX_ABS
    assert e32[0] <= e16[0]
    # the backward on the fp32-sized workspace
    rng = np.random.default_rng(2)
    dO = bf16(rng, (cfg.N, cfg.Hq, cfg.D))
    dQ, dK, dV = msa.sparse_attn_bwd(Q, K, V, O16, dO.to(dev), L16, s, scale=cfg.scale)
    torch.cuda.synchronize()
    assert s.query()["status"] == 0
    s.close()
    q8 = qids[:24]
    rQ, _, _, _ = oracle.attn_bwd(Qb, Kb, Vb, bits(dO), wl.indices.numpy(), Lkv=cfg.Lkv, scale=cfg.scale, qids=q8,
                                  rows=())
    assert rel_l2(dQ.float().cpu().numpy()[q8], rQ) <= BWD_REL_L2


def test_fp32_partials_e4m3():
    msa = _msa()
    dev = torch.device("cuda")
    rng = np.random.default_rng(4)
    N, Lkv, Hkv, topK = 1024, 2048, 2, 6
    xs = [torch.from_numpy(rng.standard_normal(sh).astype(np.float32))
          for sh in [(N, 16 * Hkv, 128), (Lkv, Hkv, 128), (Lkv, Hkv, 128)]]
    (Q, dq), (K, dk), (V, dv) = (workloads.quantize_e4m3(x) for x in xs)
    idx = lists(rng, N, Lkv, Hkv, topK)
    s = msa.build_schedule(torch.from_numpy(idx).to(dev), Lkv // 128)
    O, LSE = msa.sparse_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), s, scale=0.1, descales=(dq, dk, dv),
                                 partials_fp32=True)
    torch.cuda.synchronize()
    s.close()
    Or, Lr, _ = oracle.attn_fwd(Q.numpy(), K.numpy(), V.numpy(), idx, Lkv=Lkv, scale=0.1, q_descale=dq,
                                k_descale=dk, v_descale=dv)
    rel, mabs, lerr = compare_outputs(O.float().cpu().numpy(), LSE.cpu().numpy(), Or, Lr)
    assert rel <= 5e-2 and lerr <= LSE_MAX_ABS, (rel, mabs, lerr)
