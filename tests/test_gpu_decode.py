"""Decode-size N on the Q-outer path with split units.

"Kernel optimization for MiniMax M3", Q-outer vs KV-outer section: with few queries
each query walks its own selected blocks.  At decode sizes the (query, group) units are
fewer than the SMs, so the Q-outer kernel splits every unit's deduplicated block list
into chunks handled by different CTAs and merges the chunks' partial outputs by their
softmax statistics, in chunk order (with 4 to 8 chunks per unit, when the units fill at
most a quarter of the SMs).  Parity against the fp64 oracle over small N, KV head
counts and list lengths: fewer valid blocks than chunks, a unit whose list is all
padding, duplicates and future blocks, and shapes just past the split limit.
Repeated calls are bit-identical.
"""
import numpy as np
import pytest
import torch

import oracle
from tests.util import BF16_MAX_ABS, BF16_REL_L2, LSE_MAX_ABS, compare_outputs

pytestmark = pytest.mark.gpu


def _msa():
    import block_sparse_gqa_gb300 as msa
    return msa


def bits(t):
    return t.view(torch.int16).numpy().view(np.uint16)


@pytest.mark.parametrize("N,Lkv,Hkv,topK", [(1, 65536, 4, 16), (1, 8192, 1, 6), (2, 16384, 2, 33),
                                            (5, 32768, 4, 16), (16, 65536, 4, 16), (40, 4096, 1, 8)])
def test_decode_split_parity(N, Lkv, Hkv, topK):
    msa = _msa()
    dev = torch.device("cuda")
    rng = np.random.default_rng(N * 31 + topK)
    mk = lambda shape: torch.from_numpy(rng.standard_normal(shape).astype(np.float32)).to(torch.bfloat16)
    Q, K, V = mk((N, 16 * Hkv, 128)), mk((Lkv, Hkv, 128)), mk((Lkv, Hkv, 128))
    nb = Lkv // 128
    idx = rng.integers(-1, nb, size=(N, Hkv, topK)).astype(np.int32)  # pads and (for N > 1) future blocks
    idx[:, :, 0] = ((Lkv - N + np.arange(N)) // 128)[:, None]
    if topK > 2:
        idx[:, :, 2] = idx[:, :, 1]  # duplicates
    if N > 1:
        idx[1, 0, :] = -1  # a unit without blocks: O = 0, LSE = -inf
    s = msa.build_schedule(torch.from_numpy(idx).to(dev), nb)
    Qd, Kd, Vd = Q.to(dev), K.to(dev), V.to(dev)
    O, LSE = msa.sparse_attn_fwd(Qd, Kd, Vd, s, path="q_outer")
    O2, LSE2 = msa.sparse_attn_fwd(Qd, Kd, Vd, s, path="q_outer")
    torch.cuda.synchronize()
    assert torch.equal(O, O2) and torch.equal(LSE, LSE2)
    assert s.query()["status"] == 0
    s.close()
    Or, Lr, _ = oracle.attn_fwd(bits(Q), bits(K), bits(V), idx, Lkv=Lkv, scale=128 ** -0.5)
    rel, mabs, lerr = compare_outputs(O.float().cpu().numpy(), LSE.cpu().numpy(), Or, Lr)
    assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS, (rel, mabs, lerr)
    if N > 1:
        assert torch.all(O[1, :16] == 0) and torch.all(torch.isinf(LSE[1, :16]))
