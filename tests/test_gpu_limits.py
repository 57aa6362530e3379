"""Long lists: the largest list length the library takes (topK = 64, which fills both
32-slot words of a Q-outer unit's list) and 33 (one id in the second word), through AUTO,
both forced paths, the split Q-outer units of a single query, and (one case) the
backward, against the fp64 oracle; with bf16 and with E4M3 inputs.

Lists hold up to topK distinct visible blocks in random order, so most queries attend
many blocks; some lists also carry a duplicate, a future block or pads.  Tolerances as in
the other parity tests: relative L2 <= 1e-2 over O, |dO| <= 2e-2 element-wise, |dLSE| <= 1e-3,
relative L2 <= 2e-2 per gradient.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.util import BF16_MAX_ABS, BF16_REL_L2, BWD_REL_L2, LSE_MAX_ABS, compare_outputs, rel_l2

pytestmark = pytest.mark.gpu


def lists(rng, N, Lkv, Hkv, topK):
    nb = Lkv // 128
    lb = (Lkv - N + np.arange(N)) // 128
    idx = np.full((N, Hkv, topK), -1, np.int32)
    for i in range(N):
        for g in range(Hkv):
            picks = rng.permutation(int(lb[i]) + 1)[:topK]
            idx[i, g, :len(picks)] = picks
    # a duplicate, a future block and a pad in some lists
    some = rng.random((N, Hkv)) < 0.2
    idx[:, :, topK - 1] = np.where(some, idx[:, :, 0], idx[:, :, topK - 1])
    fut = rng.random((N, Hkv)) < 0.1
    idx[:, :, topK - 2] = np.where(fut, np.minimum(lb[:, None] + 1, nb - 1), idx[:, :, topK - 2])
    pad = rng.random((N, Hkv)) < 0.1
    idx[:, :, 1] = np.where(pad, -1, idx[:, :, 1])
    return idx


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("N,Lkv,Hkv,topK,bwd", [(96, 16384, 2, 64, True), (96, 16384, 2, 33, False),
                                                (1, 16384, 4, 64, False), (300, 8960, 1, 64, False)])
def test_long_lists_match_oracle(N, Lkv, Hkv, topK, bwd):
    import block_sparse_gqa_gb300 as msa
    rng = np.random.default_rng(N * 1000 + topK)
    mk = lambda shape: torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
    Q, K, V, dO = mk((N, 16 * Hkv, 128)), mk((Lkv, Hkv, 128)), mk((Lkv, Hkv, 128)), mk((N, 16 * Hkv, 128))
    idx = lists(rng, N, Lkv, Hkv, topK)
    scale = 0.088
    dev = torch.device("cuda")
    Qd, Kd, Vd, dOd = (t.to(dev) for t in (Q, K, V, dO))
    s = msa.build_schedule(torch.from_numpy(idx).to(dev), Lkv // 128)
    Or, Lr, _ = oracle.attn_fwd(bits(Q), bits(K), bits(V), idx, Lkv=Lkv, scale=scale)
    outs = {}
    for path in ("auto", "kv_outer", "q_outer"):
        O, LSE = msa.sparse_attn_fwd(Qd, Kd, Vd, s, scale=scale, path=path)
        torch.cuda.synchronize()
        outs[path] = (O, LSE)
        rel, mabs, lerr = compare_outputs(O.float().cpu().numpy(), LSE.cpu().numpy(), Or, Lr)
        assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS, (path, rel, mabs, lerr)
    assert s.query()["status"] == 0
    if not bwd:  # (the oracle's backward takes 10-20 s per case: one case carries it)
        s.close()
        return
    O, LSE = outs["kv_outer"]
    dQ, dK, dV = msa.sparse_attn_bwd(Qd, Kd, Vd, O, dOd, LSE, s, scale=scale)
    torch.cuda.synchronize()
    assert s.query()["status"] == 0
    s.close()
    rQ, rK, rV, _ = oracle.attn_bwd(bits(Q), bits(K), bits(V), bits(dO), idx, Lkv=Lkv, scale=scale)
    for got, ref in ((dQ, rQ), (dK, rK), (dV, rV)):
        assert rel_l2(got.float().cpu().numpy(), ref) <= BWD_REL_L2


@pytest.mark.parametrize("N,Lkv,Hkv,topK", [(96, 16384, 2, 64), (1, 16384, 4, 64)])
def test_long_lists_e4m3_match_oracle(N, Lkv, Hkv, topK):
    """The same long lists with E4M3 inputs (per-tensor descales): the KV-outer path (V
    widened to f16 once per call) and the Q-outer path (V widened per block in shared
    memory), against the oracle on the decoded E4M3 values; relative L2 over O <= 5e-2,
    |dLSE| <= 1e-3."""
    import block_sparse_gqa_gb300 as msa
    import workloads
    from tests.util import FP8_REL_L2
    rng = np.random.default_rng(N * 1000 + topK + 7)
    shapes = [(N, 16 * Hkv, 128), (Lkv, Hkv, 128), (Lkv, Hkv, 128)]
    (Q, dq), (K, dk), (V, dv) = (workloads.quantize_e4m3(torch.from_numpy(rng.standard_normal(sh).astype(np.float32)))
                                 for sh in shapes)
    idx = lists(rng, N, Lkv, Hkv, topK)
    scale = 0.088
    dev = torch.device("cuda")
    s = msa.build_schedule(torch.from_numpy(idx).to(dev), Lkv // 128)
    Or, Lr, _ = oracle.attn_fwd(Q.numpy(), K.numpy(), V.numpy(), idx, Lkv=Lkv, scale=scale, q_descale=dq,
                                k_descale=dk, v_descale=dv)
    for path in ("auto", "kv_outer", "q_outer"):
        O, LSE = msa.sparse_attn_fwd(Q.to(dev), K.to(dev), V.to(dev), s, scale=scale, path=path, descales=(dq, dk, dv))
        torch.cuda.synchronize()
        rel, mabs, lerr = compare_outputs(O.float().cpu().numpy(), LSE.cpu().numpy(), Or, Lr)
        assert rel <= FP8_REL_L2 and lerr <= LSE_MAX_ABS, (path, rel, mabs, lerr)
    assert s.query()["status"] == 0
    s.close()
