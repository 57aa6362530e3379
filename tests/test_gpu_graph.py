"""CUDA-graph capture of the whole step.

"Kernel optimization for MiniMax M3", integration notes: the operator is exported ahead
of time and driven from a C++ op with all tensor shapes fixed per request and no
device-to-host synchronisation.  After a first (allocating) call, the schedule build,
the forward and the backward only enqueue memsets and kernels on the caller's stream,
so a serving loop can capture them once and replay the graph for every new batch of the
same shape.  Replays on new inputs written in place must give exactly what eager calls
give (every kernel is deterministic).
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu


def _msa():
    import block_sparse_gqa_gb300 as msa
    return msa


def make(rng, N, Lkv, Hkv, topK):
    Q = torch.from_numpy(rng.standard_normal((N, 16 * Hkv, 128)).astype(np.float32)).to(torch.bfloat16)
    K = torch.from_numpy(rng.standard_normal((Lkv, Hkv, 128)).astype(np.float32)).to(torch.bfloat16)
    V = torch.from_numpy(rng.standard_normal((Lkv, Hkv, 128)).astype(np.float32)).to(torch.bfloat16)
    idx = rng.integers(0, Lkv // 128, size=(N, Hkv, topK)).astype(np.int32)
    idx[:, :, 0] = ((Lkv - N + np.arange(N)) // 128)[:, None]
    return Q, K, V, torch.from_numpy(idx)


@pytest.mark.parametrize("N,Lkv,Hkv,topK,path", [(1024, 2048, 2, 8, "auto"), (16, 65536, 4, 16, "auto"),
                                                 (1024, 2048, 2, 8, "kv_outer")])
def test_forward_and_backward_graph_replay(N, Lkv, Hkv, topK, path):
    msa = _msa()
    dev = torch.device("cuda")
    rng = np.random.default_rng(N + Lkv)
    Q, K, V, idx = (t.to(dev) for t in make(rng, N, Lkv, Hkv, topK))
    dO = torch.randn_like(Q)
    O, LSE = torch.empty_like(Q), torch.empty((N, 16 * Hkv), dtype=torch.float32, device=dev)
    dQ, dK, dV = torch.empty_like(Q), torch.empty_like(K), torch.empty_like(V)
    s = msa.build_schedule(idx, Lkv // 128)

    def step():
        msa.build_schedule(idx, Lkv // 128, schedule=s)
        msa.sparse_attn_fwd(Q, K, V, s, O=O, LSE=LSE, path=path)
        msa.sparse_attn_bwd(Q, K, V, O, dO, LSE, s, dQ=dQ, dK=dK, dV=dV)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # first calls allocate the workspaces; nothing is allocated afterwards
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for seed in (1, 2):
        # new inputs of the same shape, written in place
        Qn, Kn, Vn, idxn = make(np.random.default_rng(seed), N, Lkv, Hkv, topK)
        Q.copy_(Qn); K.copy_(Kn); V.copy_(Vn); idx.copy_(idxn)
        dO.copy_(torch.randn_like(dO))
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (O, LSE, dQ, dK, dV)]
        step()
        torch.cuda.synchronize()
        for a, b in zip(got, (O, LSE, dQ, dK, dV)):
            assert torch.equal(a, b)
        assert s.query()["status"] == 0
    s.close()
