"""Bounded device waits: a wait that runs out reports a status and leaves the device usable.

Every mbarrier wait in the kernels gives up after 2 s of %globaltimer, sets the
schedule's timeout bit and lets the role leave its loop (warps that decide together do
so through one reduction barrier), and the CTA frees its tensor memory and exits.  The
test withholds the signal those waits expect (debug flag: the KV-outer scheduler warp
publishes no work; nothing faults, traps or hangs), reads MSA_ERR_TIMEOUT back, then
rebuilds the schedule and checks that a normal forward on the same device is correct.
"""
import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def test_kv_outer_wait_expires_and_device_recovers():
    import block_sparse_gqa_gb300 as msa
    dev = torch.device("cuda")
    rng = np.random.default_rng(3)
    N, Lkv, Hkv, topK = 512, 1024, 1, 4
    Q, K, V = (torch.from_numpy(rng.standard_normal(sh).astype(np.float32)).to(torch.bfloat16)
               for sh in [(N, 16, 128), (Lkv, 1, 128), (Lkv, 1, 128)])
    idx = rng.integers(0, Lkv // 128, size=(N, Hkv, topK)).astype(np.int32)
    idx[:, :, 0] = ((Lkv - N + np.arange(N)) // 128)[:, None]
    idx_d = torch.from_numpy(idx).to(dev)
    Qd, Kd, Vd = Q.to(dev), K.to(dev), V.to(dev)
    s = msa.build_schedule(idx_d, Lkv // 128)
    msa.sparse_attn_fwd(Qd, Kd, Vd, s, path="kv_outer", num_ctas=4, debug_flags=1)
    torch.cuda.synchronize()
    info = s.query()
    assert info["status"] & 2 and info["status_code"] == 6  # MSA_ERR_TIMEOUT
    assert s.status() == 6  # msa_schedule_status reports the same sticky bit
    # the same schedule rebuilt (clears the sticky bits), a normal forward, parity
    msa.build_schedule(idx_d, Lkv // 128, schedule=s)
    O, LSE = msa.sparse_attn_fwd(Qd, Kd, Vd, s, path="kv_outer")
    torch.cuda.synchronize()
    assert s.query()["status"] == 0 and s.status() == 0
    s.close()
    bits = [t.view(torch.int16).numpy().view(np.uint16) for t in (Q, K, V)]
    Or, Lr, _ = oracle.attn_fwd(*bits, idx, Lkv=Lkv, scale=128 ** -0.5)
    rel = np.linalg.norm(O.float().cpu().numpy() - Or) / np.linalg.norm(Or)
    assert rel <= 1e-2 and np.abs(LSE.cpu().numpy() - Lr).max() <= 1e-3
