"""Pins for the oracle's backward: each checks it against something other than itself.

"Flash-MSA: accelerating million-token training with sparse attention", order of
operations: the block indices and the log-sum-exp of the forward are kept for the
backward, which takes the main-attention gradients over the same blocks.  The pins
fix those gradients by (1) central finite differences of the oracle's own forward (a
different computation: no gradient formula is involved), (2) torch autograd of dense
causal attention when every list holds every visible block, (3) closed forms for
constant V and uniform weights, (4) invariance to list order, duplicates and pads,
and (5) the sampled outputs agree with the full ones.
"""
import numpy as np
import pytest
import torch

import oracle


def lists(rng, N, Lkv, Hkv, topK, block, extras=True):
    nb = Lkv // block
    idx = rng.integers(0, nb, size=(N, Hkv, topK)).astype(np.int32)  # includes future blocks
    idx[:, :, 0] = ((Lkv - N + np.arange(N)) // block)[:, None]
    if extras:
        idx[::3, :, -1] = -1
        idx[1::4, :, 1 % topK] = idx[1::4, :, 0]
    return idx


def objective(Q, K, V, dO, idx, Lkv, block, scale):
    O, _, _ = oracle.attn_fwd(Q, K, V, idx, Lkv=Lkv, block=block, scale=scale, nthreads=1)
    return float((O * dO).sum())


def test_finite_differences_every_element():
    """Every element of dQ, dK and dV against a central difference of sum(dO * O)."""
    rng = np.random.default_rng(1)
    N, Lkv, Hq, Hkv, D, block, topK, scale = 12, 16, 4, 2, 6, 4, 3, 0.4
    Q, K, V, dO = (rng.standard_normal(s) for s in [(N, Hq, D), (Lkv, Hkv, D), (Lkv, Hkv, D), (N, Hq, D)])
    idx = lists(rng, N, Lkv, Hkv, topK, block)
    dQ, dK, dV, st = oracle.attn_bwd(Q, K, V, dO, idx, Lkv=Lkv, block=block, scale=scale, nthreads=3)
    assert st == 0
    eps = 1e-5
    for arr, grad in ((Q, dQ), (K, dK), (V, dV)):
        num = np.zeros_like(arr)
        for ix in np.ndindex(arr.shape):
            old = arr[ix]
            arr[ix] = old + eps
            fp = objective(Q, K, V, dO, idx, Lkv, block, scale)
            arr[ix] = old - eps
            fm = objective(Q, K, V, dO, idx, Lkv, block, scale)
            arr[ix] = old
            num[ix] = (fp - fm) / (2 * eps)
        assert np.max(np.abs(num - grad)) < 1e-7 * max(1.0, np.max(np.abs(grad))), np.max(np.abs(num - grad))
    # keys no query sees (blocks never selected) get exactly zero
    seen = np.zeros((Lkv, Hkv), bool)
    for i in range(N):
        pos = Lkv - N + i
        for g in range(Hkv):
            for b in set(idx[i, g].tolist()):
                if 0 <= b <= pos // block:
                    seen[b * block:min(b * block + block, pos + 1), g] = True
    assert np.all(dK[~seen] == 0) and np.all(dV[~seen] == 0)


@pytest.mark.parametrize("N,Lkv", [(64, 64), (40, 96)])
def test_dense_equivalence_torch_autograd(N, Lkv):
    """Lists holding every block up to the query's own: the gradients of textbook causal
    attention (bottom-right aligned), taken by torch autograd in float64."""
    rng = np.random.default_rng(N + Lkv)
    Hq, Hkv, D, block, scale = 4, 2, 16, 16, 0.25
    nb = Lkv // block
    Q, K, V, dO = (rng.standard_normal(s) for s in [(N, Hq, D), (Lkv, Hkv, D), (Lkv, Hkv, D), (N, Hq, D)])
    idx = np.full((N, Hkv, nb), -1, np.int32)
    for i in range(N):
        lb = (Lkv - N + i) // block
        idx[i, :, : lb + 1] = rng.permutation(lb + 1)
    dQ, dK, dV, _ = oracle.attn_bwd(Q, K, V, dO, idx, Lkv=Lkv, block=block, scale=scale)

    tQ, tK, tV = (torch.tensor(a, requires_grad=True) for a in (Q, K, V))
    G = Hq // Hkv
    S = torch.einsum("nhd,jhd->hnj", tQ, tK.repeat_interleave(G, 1)) * scale
    pos = Lkv - N + torch.arange(N)
    mask = torch.arange(Lkv)[None, :] <= pos[:, None]
    S = S.masked_fill(~mask[None], float("-inf"))
    O = torch.einsum("hnj,jhd->nhd", torch.softmax(S, -1), tV.repeat_interleave(G, 1))
    O.backward(torch.tensor(dO))
    for mine, ref in ((dQ, tQ.grad), (dK, tK.grad), (dV, tV.grad)):
        np.testing.assert_allclose(mine, ref.numpy(), rtol=0, atol=1e-11)


def test_closed_forms():
    rng = np.random.default_rng(7)
    N, Lkv, Hq, Hkv, D, block, topK, scale = 20, 24, 4, 2, 8, 4, 3, 0.3
    Q, K, dO = (rng.standard_normal(s) for s in [(N, Hq, D), (Lkv, Hkv, D), (N, Hq, D)])
    idx = lists(rng, N, Lkv, Hkv, topK, block)
    # V constant: O does not depend on Q or K, so dQ = dK = 0
    V = np.full((Lkv, Hkv, D), 0.75)
    dQ, dK, dV, _ = oracle.attn_bwd(Q, K, V, dO, idx, Lkv=Lkv, block=block, scale=scale)
    assert np.max(np.abs(dQ)) < 1e-13 and np.max(np.abs(dK)) < 1e-13
    # Q = 0: uniform weights 1/|J| over the visible keys, so dV_j sums dO / |J|
    V = rng.standard_normal((Lkv, Hkv, D))
    _, _, dV, _ = oracle.attn_bwd(np.zeros_like(Q), K, V, dO, idx, Lkv=Lkv, block=block, scale=scale)
    ref = np.zeros_like(dV)
    G = Hq // Hkv
    for i in range(N):
        pos = Lkv - N + i
        for g in range(Hkv):
            blocks = {b for b in idx[i, g].tolist() if 0 <= b <= pos // block}
            keys = [j for b in blocks for j in range(b * block, b * block + block) if j <= pos]
            for j in keys:
                ref[j, g] += dO[i, g * G:(g + 1) * G].sum(0) / len(keys)
    np.testing.assert_allclose(dV, ref, rtol=0, atol=1e-12)


def test_order_duplicate_pad_invariance():
    rng = np.random.default_rng(3)
    N, Lkv, Hq, Hkv, D, block, topK, scale = 24, 32, 4, 2, 8, 8, 3, 0.35
    Q, K, V, dO = (rng.standard_normal(s) for s in [(N, Hq, D), (Lkv, Hkv, D), (Lkv, Hkv, D), (N, Hq, D)])
    idx = lists(rng, N, Lkv, Hkv, topK, block, extras=False)
    a = oracle.attn_bwd(Q, K, V, dO, idx, Lkv=Lkv, block=block, scale=scale)
    shuffled = np.ascontiguousarray(rng.permuted(idx, axis=2))
    padded = np.concatenate([shuffled, shuffled[:, :, :1], np.full((N, Hkv, 2), -1, np.int32)], axis=2)
    b = oracle.attn_bwd(Q, K, V, dO, padded, Lkv=Lkv, block=block, scale=scale)
    for x, y in zip(a[:3], b[:3]):
        np.testing.assert_allclose(x, y, rtol=0, atol=1e-12)


def test_sampled_outputs_match_full():
    rng = np.random.default_rng(5)
    N, Lkv, Hq, Hkv, D, block, topK, scale = 30, 32, 4, 2, 8, 8, 3, 0.2
    Q, K, V, dO = (rng.standard_normal(s) for s in [(N, Hq, D), (Lkv, Hkv, D), (Lkv, Hkv, D), (N, Hq, D)])
    idx = lists(rng, N, Lkv, Hkv, topK, block)
    dQ, dK, dV, _ = oracle.attn_bwd(Q, K, V, dO, idx, Lkv=Lkv, block=block, scale=scale)
    qids = np.array([29, 0, 17], np.int32)
    rows = np.array([5, 0, 3], np.int32)  # row r = g * nblocks + b
    sQ, sK, sV, _ = oracle.attn_bwd(Q, K, V, dO, idx, Lkv=Lkv, block=block, scale=scale, qids=qids, rows=rows,
                                    nthreads=2)
    np.testing.assert_allclose(sQ, dQ[qids], rtol=0, atol=1e-13)
    nb = Lkv // block
    for k, r in enumerate(rows):
        g, b = divmod(int(r), nb)
        np.testing.assert_allclose(sK[k], dK[b * block:(b + 1) * block, g], rtol=0, atol=1e-13)
        np.testing.assert_allclose(sV[k], dV[b * block:(b + 1) * block, g], rtol=0, atol=1e-13)


def test_bf16_bits_equal_decoded_f64():
    rng = np.random.default_rng(9)
    N, Lkv, Hq, Hkv, D, block, topK = 8, 16, 2, 1, 8, 8, 2
    xs = [torch.from_numpy(rng.standard_normal(s)).to(torch.bfloat16)
          for s in [(N, Hq, D), (Lkv, Hkv, D), (Lkv, Hkv, D), (N, Hq, D)]]
    bits = [x.view(torch.int16).numpy().view(np.uint16) for x in xs]
    dec = [x.double().numpy() for x in xs]
    idx = lists(rng, N, Lkv, Hkv, topK, block)
    a = oracle.attn_bwd(*bits, idx, Lkv=Lkv, block=block, scale=0.3)
    b = oracle.attn_bwd(*dec, idx, Lkv=Lkv, block=block, scale=0.3)
    for x, y in zip(a[:3], b[:3]):
        assert np.array_equal(x, y)
