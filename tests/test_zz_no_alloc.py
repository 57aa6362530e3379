"""The allocation-free forward against the allocating one.

msa_sparse_attn_fwd_noalloc serves callers that cannot call cudaMalloc (a device-
memory budget fixed at start-up, a runtime that owns all device memory, or a loop
that cannot absorb an allocation's device-wide synchronisation).  It runs the same
kernels as msa_build_schedule + msa_sparse_attn_fwd with its scratch in a fixed
device array inside libmsa.  Two calls in a row share that array, so the second
call also shows that nothing from the first leaks into its result.

This file is collected last on purpose (pytest orders files by name).
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads
from tests.util import BF16_MAX_ABS, BF16_REL_L2, LSE_MAX_ABS, compare_outputs

pytestmark = pytest.mark.gpu
MSA_ERR_CAPACITY = 7


def noalloc_fwd(msa, idx, nblocks, Q, K, V, scale):
    L = msa.lib()
    fn = L.msa_sparse_attn_fwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, msa.Tensor, msa.Tensor,
                   msa.Tensor, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_float, ctypes.POINTER(msa.FwdOpts)]
    N, Hkv, topK = idx.shape
    O = torch.empty((N, Q.shape[1], Q.shape[2]), dtype=torch.bfloat16, device=Q.device)
    LSE = torch.empty((N, Q.shape[1]), dtype=torch.float32, device=Q.device)
    opts = msa.FwdOpts()
    L.msa_fwd_opts_init(ctypes.byref(opts))
    opts.stream = torch.cuda.current_stream().cuda_stream
    st = fn(idx.data_ptr(), N, Hkv, topK, nblocks, msa._tensor(Q), msa._tensor(K), msa._tensor(V), O.data_ptr(),
            LSE.data_ptr(), float(scale), ctypes.byref(opts))
    return st, O, LSE


def inputs(seed, sparser):
    wl = workloads.make_workload("tiny", seed=seed)
    idx = wl.indices.clone()
    if sparser:  # fewer entries than the previous call, so stale scratch would show
        idx[::2, :, 2:] = -1
    dev = torch.device("cuda")
    return wl.cfg, idx.to(dev), wl.Q.to(dev), wl.K.to(dev), wl.V.to(dev)


def test_noalloc_matches_allocating_path_on_two_calls_in_a_row():
    import block_sparse_gqa_gb300 as msa
    for seed, sparser in ((1000, False), (4242, True)):
        cfg, idx, Q, K, V = inputs(seed, sparser)
        sched = msa.build_schedule(idx, cfg.nblocks)
        O_ref, L_ref = msa.sparse_attn_fwd(Q, K, V, sched, scale=cfg.scale)
        st, O, LSE = noalloc_fwd(msa, idx, cfg.nblocks, Q, K, V, cfg.scale)
        torch.cuda.synchronize()
        sched.close()
        assert st == 0, msa.lib().msa_status_string(st)
        rel, mabs, lerr = compare_outputs(O.float().cpu().numpy(), LSE.cpu().numpy(),
                                          O_ref.float().cpu().numpy().astype(np.float64),
                                          L_ref.cpu().numpy().astype(np.float64))
        assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS, (seed, rel, mabs, lerr)


def test_noalloc_rejects_problems_beyond_its_scratch():
    import block_sparse_gqa_gb300 as msa
    cfg = workloads.CONFIGS["m3"]
    dev = torch.device("cuda")
    idx = torch.zeros((cfg.N, cfg.Hkv, cfg.topK), dtype=torch.int32, device=dev)
    Q = torch.empty((cfg.N, cfg.Hq, cfg.D), dtype=torch.bfloat16, device=dev)
    K = torch.empty((cfg.Lkv, cfg.Hkv, cfg.D), dtype=torch.bfloat16, device=dev)
    st, _, _ = noalloc_fwd(msa, idx, cfg.nblocks, Q, K, K, cfg.scale)
    assert st == MSA_ERR_CAPACITY
