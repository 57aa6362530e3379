"""The allocation-free forward against the allocating one, and against the oracle.

msa_sparse_attn_fwd_noalloc serves callers that cannot call cudaMalloc (a device-
memory budget fixed at start-up, a runtime that owns all device memory, or a loop
that cannot absorb an allocation's device-wide synchronisation).  It runs the same
kernels as msa_build_schedule + msa_sparse_attn_fwd with its scratch in a fixed
device array inside libmsa, so its outputs must be bit-identical to that pair's.  Two
calls in a row share that array, so the second call (with fewer entries than the
first) also shows that nothing from the first leaks into its result.

This file is collected last on purpose (pytest orders files by name).
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads
from tests.util import BF16_MAX_ABS, BF16_REL_L2, LSE_MAX_ABS, compare_outputs

pytestmark = pytest.mark.gpu
MSA_ERR_UNSUPPORTED = 2
MSA_ERR_CAPACITY = 7


def noalloc_fwd(msa, idx, nblocks, Q, K, V, scale, status=None, **opt_fields):
    L = msa.lib()
    fn = L.msa_sparse_attn_fwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, msa.Tensor, msa.Tensor,
                   msa.Tensor, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.c_void_p,
                   ctypes.POINTER(msa.FwdOpts)]
    N, Hkv, topK = idx.shape
    O = torch.empty((N, Q.shape[1], Q.shape[2]), dtype=torch.bfloat16, device=Q.device)
    LSE = torch.empty((N, Q.shape[1]), dtype=torch.float32, device=Q.device)
    opts = msa.FwdOpts()
    L.msa_fwd_opts_init(ctypes.byref(opts))
    opts.stream = torch.cuda.current_stream().cuda_stream
    for k, v in opt_fields.items():
        setattr(opts, k, v)
    st = fn(idx.data_ptr(), N, Hkv, topK, nblocks, msa._tensor(Q), msa._tensor(K), msa._tensor(V), O.data_ptr(),
            LSE.data_ptr(), float(scale), None if status is None else status.data_ptr(), ctypes.byref(opts))
    return st, O, LSE


def inputs(seed, sparser):
    wl = workloads.make_workload("tiny", seed=seed)
    idx = wl.indices.clone()
    if sparser:  # fewer entries than the previous call, so stale scratch would show
        idx[::2, :, 2:] = -1
    return wl.cfg, idx, wl.Q, wl.K, wl.V


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


def test_noalloc_matches_allocating_path_on_two_calls_in_a_row():
    import block_sparse_gqa_gb300 as msa
    dev = torch.device("cuda")
    # the KV-outer path keeps its partial outputs in the shared array; the tiny workload's
    # own choice (AUTO) is the Q-outer kernel, which needs no partials
    for (seed, sparser), path in (((1000, False), "kv_outer"), ((4242, True), "kv_outer"), ((1000, False), "auto")):
        cfg, idx_h, Qh, Kh, Vh = inputs(seed, sparser)
        idx, Q, K, V = idx_h.to(dev), Qh.to(dev), Kh.to(dev), Vh.to(dev)
        sched = msa.build_schedule(idx, cfg.nblocks)
        O_ref, L_ref = msa.sparse_attn_fwd(Q, K, V, sched, scale=cfg.scale, path=path)
        status = torch.full((1,), -1, dtype=torch.int32, device=dev)
        st, O, LSE = noalloc_fwd(msa, idx, cfg.nblocks, Q, K, V, cfg.scale, status=status, path=msa.PATHS[path])
        torch.cuda.synchronize()
        sched.close()
        assert st == 0, msa.lib().msa_status_string(st)
        assert int(status.item()) == 0
        # the same kernels on the same inputs: bit-identical outputs
        assert torch.equal(O.view(torch.int16), O_ref.view(torch.int16)), seed
        assert torch.equal(LSE.view(torch.int32), L_ref.view(torch.int32)), seed
        # and a sample of queries against the oracle
        qids = np.unique(np.concatenate([[0, cfg.N - 1], np.random.default_rng(seed).integers(0, cfg.N, 62)]))
        Or, Lr, _ = oracle.attn_fwd(bits(Qh), bits(Kh), bits(Vh), idx_h.numpy(), Lkv=cfg.Lkv, scale=cfg.scale,
                                    qids=qids.astype(np.int32))
        rel, mabs, lerr = compare_outputs(O.float().cpu().numpy()[qids], LSE.cpu().numpy()[qids], Or, Lr)
        assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS, (seed, rel, mabs, lerr)


def test_noalloc_decode_step_matches_allocating_path():
    """A decode-size call (one query at the tail of a 128K-token context): AUTO is decided by
    the sizes alone, so both entry points launch only the Q-outer kernel, with the query's
    list split over several CTAs whose workspace the scratch array holds.  Bit-identical to
    the allocating pair, and equal to the oracle."""
    import block_sparse_gqa_gb300 as msa
    dev = torch.device("cuda")
    wl = workloads.make_workload("decode")
    cfg = wl.cfg
    idx, Q, K, V = wl.indices.to(dev), wl.Q.to(dev), wl.K.to(dev), wl.V.to(dev)
    sched = msa.build_schedule(idx, cfg.nblocks)
    O_ref, L_ref = msa.sparse_attn_fwd(Q, K, V, sched, scale=cfg.scale)
    status = torch.full((1,), -1, dtype=torch.int32, device=dev)
    st, O, LSE = noalloc_fwd(msa, idx, cfg.nblocks, Q, K, V, cfg.scale, status=status)
    torch.cuda.synchronize()
    assert sched.query()["path"] == 2  # the device's own choice agrees: Q-outer
    sched.close()
    assert st == 0, msa.lib().msa_status_string(st)
    assert int(status.item()) == 0
    assert torch.equal(O.view(torch.int16), O_ref.view(torch.int16))
    assert torch.equal(LSE.view(torch.int32), L_ref.view(torch.int32))
    Or, Lr, _ = oracle.attn_fwd(bits(wl.Q), bits(wl.K), bits(wl.V), wl.indices.numpy(), Lkv=cfg.Lkv, scale=cfg.scale)
    rel, mabs, lerr = compare_outputs(O.float().cpu().numpy(), LSE.cpu().numpy(), Or, Lr)
    assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS, (rel, mabs, lerr)


def test_noalloc_reports_bad_block_ids_through_status():
    import block_sparse_gqa_gb300 as msa
    dev = torch.device("cuda")
    cfg, idx_h, Qh, Kh, Vh = inputs(1000, False)
    idx_h = idx_h.clone()
    idx_h[5, 0, 1] = cfg.nblocks + 7  # out of range: ignored like a pad, and reported
    idx, Q, K, V = idx_h.to(dev), Qh.to(dev), Kh.to(dev), Vh.to(dev)
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    st, O, LSE = noalloc_fwd(msa, idx, cfg.nblocks, Q, K, V, cfg.scale, status=status, path=1)
    torch.cuda.synchronize()
    assert st == 0 and int(status.item()) & 1
    sched = msa.build_schedule(idx, cfg.nblocks)
    O_ref, _ = msa.sparse_attn_fwd(Q, K, V, sched, scale=cfg.scale, path="kv_outer")
    torch.cuda.synchronize()
    assert sched.status() == 5  # MSA_ERR_BAD_INDEX on the allocating pair too
    sched.close()
    assert torch.equal(O.view(torch.int16), O_ref.view(torch.int16))
    # a clean call right after clears the bit (the shared array keeps no stale status)
    cfg, idx_h, Qh, Kh, Vh = inputs(1000, False)
    st, _, _ = noalloc_fwd(msa, idx_h.to(dev), cfg.nblocks, Qh.to(dev), Kh.to(dev), Vh.to(dev), cfg.scale,
                           status=status)
    torch.cuda.synchronize()
    assert st == 0 and int(status.item()) == 0


def test_noalloc_rejects_problems_beyond_its_scratch_and_unsupported_options():
    import block_sparse_gqa_gb300 as msa
    cfg = workloads.CONFIGS["m3"]
    dev = torch.device("cuda")
    idx = torch.zeros((cfg.N, cfg.Hkv, cfg.topK), dtype=torch.int32, device=dev)
    Q = torch.empty((cfg.N, cfg.Hq, cfg.D), dtype=torch.bfloat16, device=dev)
    K = torch.empty((cfg.Lkv, cfg.Hkv, cfg.D), dtype=torch.bfloat16, device=dev)
    st, _, _ = noalloc_fwd(msa, idx, cfg.nblocks, Q, K, K, cfg.scale)
    assert st == MSA_ERR_CAPACITY
    cfg, idx_h, Qh, Kh, Vh = inputs(1000, False)
    args = (idx_h.to(dev), cfg.nblocks, Qh.to(dev), Kh.to(dev), Vh.to(dev), cfg.scale)
    assert noalloc_fwd(msa, *args, partials_fp32=1)[0] == MSA_ERR_UNSUPPORTED
    assert noalloc_fwd(msa, *args, debug_flags=1)[0] == MSA_ERR_UNSUPPORTED
