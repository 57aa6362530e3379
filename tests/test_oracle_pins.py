"""Pins for the oracle: each checks it against something other than itself.

Sources: "Sparse Attention" (dinara-dl) Ch. 1 (softmax over the union of selected
blocks), Ch. 2 (worked example [2, 5, 8]), Ch. 5 (reverse index; LSE-weighted
combine); "Flash-MSA" (local block always attended, causally); "Kernel optimization
for MiniMax M3" (block 128, GQA groups, crossover nsb/N < 2.85).
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rnd(rng, *shape):
    return rng.standard_normal(shape)


def dense_causal(Q, K, V, Lkv, scale):
    """Textbook causal GQA attention as full matrices (bottom-right aligned)."""
    N, Hq, D = Q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    Kx = np.repeat(K, G, axis=1)
    Vx = np.repeat(V, G, axis=1)
    S = np.einsum("nhd,jhd->hnj", Q, Kx) * scale
    pos = Lkv - N + np.arange(N)
    mask = np.arange(Lkv)[None, :] <= pos[:, None]
    S = np.where(mask[None], S, -np.inf)
    m = S.max(-1, keepdims=True)
    P = np.exp(S - m)
    l = P.sum(-1, keepdims=True)
    O = np.einsum("hnj,jhd->nhd", P / l, Vx)
    return O, (m + np.log(l))[..., 0].T


def masked_bruteforce(Q, K, V, indices, Lkv, block, scale):
    """Dense 0/1 mask built from the lists with Python sets, then a masked softmax."""
    N, Hq, D = Q.shape
    Hkv = K.shape[1]
    G = Hq // Hkv
    nb = Lkv // block
    O = np.zeros((N, Hq, D))
    LSE = np.full((N, Hq), -np.inf)
    for i in range(N):
        pos = Lkv - N + i
        for h in range(Hq):
            g = h // G
            chosen = {int(b) for b in indices[i, g] if 0 <= b < nb}
            keys = [j for j in range(Lkv) if (j // block) in chosen and j <= pos]
            if not keys:
                continue
            s = np.array([scale * float(Q[i, h] @ K[j, g]) for j in keys])
            w = np.exp(s - s.max())
            O[i, h] = (w / w.sum()) @ V[keys, g]
            LSE[i, h] = s.max() + math.log(w.sum())
    return O, LSE


def full_lists(N, Lkv, Hkv, block, topK=None):
    """Lists lb(i), lb(i)-1, ..., 0 (local block first), cut to topK and -1 padded."""
    nb = Lkv // block
    topK = topK or nb
    idx = np.full((N, Hkv, topK), -1, np.int32)
    for i in range(N):
        lb = (Lkv - N + i) // block
        n = min(lb + 1, topK)
        for g in range(Hkv):
            idx[i, g, :n] = np.arange(lb + 1)[::-1][:n]
    return idx


@pytest.mark.parametrize("N,Lkv", [(256, 256), (96, 256)])
def test_dense_equivalence(N, Lkv):
    """Lists holding every block 0..lb(i) reduce to dense causal GQA attention."""
    rng = np.random.default_rng(1)
    Hq, Hkv, D, block = 4, 2, 16, 32
    Q, K, V = rnd(rng, N, Hq, D), rnd(rng, Lkv, Hkv, D), rnd(rng, Lkv, Hkv, D)
    scale = 1 / math.sqrt(D)
    idx = full_lists(N, Lkv, Hkv, block)
    O, LSE, st = oracle.attn_fwd(Q, K, V, idx, Lkv=Lkv, block=block, scale=scale)
    Od, LSEd = dense_causal(Q, K, V, Lkv, scale)
    assert st == 0
    np.testing.assert_allclose(O, Od, rtol=0, atol=1e-12)
    np.testing.assert_allclose(LSE, LSEd, rtol=0, atol=1e-12)


def test_topk1_local_block_only():
    """topK = 1: an explicit causal softmax over keys 128*lb(i) .. pos(i)."""
    rng = np.random.default_rng(2)
    N = Lkv = 256
    Hq, Hkv, D, block = 2, 1, 8, 128
    Q, K, V = rnd(rng, N, Hq, D), rnd(rng, Lkv, Hkv, D), rnd(rng, Lkv, Hkv, D)
    scale = 0.37
    idx = np.array([[[i // block]] for i in range(N)], np.int32)
    O, LSE, _ = oracle.attn_fwd(Q, K, V, idx, Lkv=Lkv, block=block, scale=scale)
    for i in [0, 1, 77, 127, 128, 129, 200, 255]:
        for h in range(Hq):
            lo = 128 * (i // 128)
            s = np.array([scale * np.dot(Q[i, h], K[j, 0]) for j in range(lo, i + 1)])
            e = np.exp(s - s.max())
            ref = sum(e[t] * V[lo + t, 0] for t in range(len(e))) / e.sum()
            assert np.max(np.abs(O[i, h] - ref)) < 1e-12
            assert abs(LSE[i, h] - (s.max() + math.log(e.sum()))) < 1e-12


def test_bruteforce_random_lists():
    """Random lists with pads, duplicates and future blocks vs a set-built dense mask."""
    rng = np.random.default_rng(3)
    N, Lkv, Hq, Hkv, D, block, topK = 40, 64, 6, 3, 8, 8, 5
    nb = Lkv // block
    Q, K, V = rnd(rng, N, Hq, D), rnd(rng, Lkv, Hkv, D), rnd(rng, Lkv, Hkv, D)
    idx = rng.integers(-1, nb, size=(N, Hkv, topK)).astype(np.int32)
    scale = 0.25
    O, LSE, st = oracle.attn_fwd(Q, K, V, idx, Lkv=Lkv, block=block, scale=scale)
    Ob, LSEb = masked_bruteforce(Q, K, V, idx, Lkv, block, scale)
    assert st == 0
    np.testing.assert_allclose(O, Ob, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(LSE), np.isinf(LSEb))
    fin = np.isfinite(LSEb)
    np.testing.assert_allclose(LSE[fin], LSEb[fin], atol=1e-12)
    assert np.all(O[~fin] == 0.0)


def test_order_duplicate_pad_invariance():
    """Shuffling lists, appending duplicates and -1 pads changes neither O/LSE nor the CSR."""
    rng = np.random.default_rng(4)
    N = Lkv = 512
    Hq, Hkv, D, block, topK = 4, 2, 16, 64, 4
    Q, K, V = rnd(rng, N, Hq, D), rnd(rng, Lkv, Hkv, D), rnd(rng, Lkv, Hkv, D)
    idx = np.full((N, Hkv, topK), -1, np.int32)
    for i in range(N):
        lb = i // block
        for g in range(Hkv):
            picks = rng.permutation(lb)[: topK - 1] if lb else []
            idx[i, g, 0] = lb
            idx[i, g, 1 : 1 + len(picks)] = picks
    shuf = idx.copy()
    for i in range(N):
        for g in range(Hkv):
            rng.shuffle(shuf[i, g])
    extra = np.concatenate([shuf, shuf[:, :, :2], np.full((N, Hkv, 3), -1, np.int32)], axis=2)
    O1, L1, _ = oracle.attn_fwd(Q, K, V, idx, Lkv=Lkv, block=block, scale=0.3)
    O2, L2, _ = oracle.attn_fwd(Q, K, V, extra, Lkv=Lkv, block=block, scale=0.3)
    np.testing.assert_allclose(O1, O2, atol=1e-13)
    np.testing.assert_allclose(L1, L2, atol=1e-13)
    s1 = oracle.schedule(idx, Lkv=Lkv, block=block)
    s2 = oracle.schedule(extra, Lkv=Lkv, block=block)
    for k in ("counts", "offsets", "qlist"):
        np.testing.assert_array_equal(s1[k], s2[k])
    assert s1["nsb"] == s2["nsb"] and s1["E"] == s2["E"]


def test_closed_forms():
    rng = np.random.default_rng(5)
    N = Lkv = 384
    Hq, Hkv, D, block = 4, 2, 8, 128
    idx = full_lists(N, Lkv, Hkv, block, topK=3)
    K = rnd(rng, Lkv, Hkv, D)
    # V constant -> O equals the constant
    c = 1.75
    Q = rnd(rng, N, Hq, D)
    O, _, _ = oracle.attn_fwd(Q, K, np.full((Lkv, Hkv, D), c), idx, Lkv=Lkv, block=block, scale=0.5)
    assert np.max(np.abs(O - c)) < 1e-14
    # Q zero -> O is the mean of the visible V rows, LSE = log |J| = log(pos + 1)
    V = rnd(rng, Lkv, Hkv, D)
    O, LSE, _ = oracle.attn_fwd(np.zeros((N, Hq, D)), K, V, idx, Lkv=Lkv, block=block, scale=0.5)
    G = Hq // Hkv
    for i in [0, 5, 130, 383]:
        for h in range(Hq):
            ref = V[: i + 1, h // G].mean(axis=0)
            assert np.max(np.abs(O[i, h] - ref)) < 1e-13
            assert abs(LSE[i, h] - math.log(i + 1)) < 1e-13
    # query at pos = 128 b with only its local block: O = V[pos], LSE = scale * q.k[pos]
    only_local = np.array([[[i // block] + [-1] * 2] * Hkv for i in range(N)], np.int32)
    O, LSE, _ = oracle.attn_fwd(Q, K, V, only_local, Lkv=Lkv, block=block, scale=0.5)
    for i in (0, 128, 256):
        for h in range(Hq):
            g = h // G
            assert np.array_equal(O[i, h], V[i, g])
            assert abs(LSE[i, h] - 0.5 * float(Q[i, h] @ K[i, g])) < 1e-13


def test_merge_identity():
    """Per-part softmax results merged by LSE weighting equal the whole (P3 Ch. 5 combine)."""
    rng = np.random.default_rng(6)
    N = Lkv = 512
    Hq, Hkv, D, block = 2, 1, 16, 64
    Q, K, V = rnd(rng, N, Hq, D) * 3, rnd(rng, Lkv, Hkv, D), rnd(rng, Lkv, Hkv, D)
    i = 450  # lb = 7
    whole = np.full((N, 1, 8), -1, np.int32)
    whole[i, 0] = [7, 0, 3, 5, 1, 6, 2, 4]
    Ow, Lw, _ = oracle.attn_fwd(Q, K, V, whole, Lkv=Lkv, block=block, scale=0.4, qids=[i])
    parts = [[7, 3], [0], [5, 1, 6], [2, 4]]
    Op, Lp = [], []
    for p in parts:
        lst = np.full((N, 1, 8), -1, np.int32)
        lst[i, 0, : len(p)] = p
        o, l, _ = oracle.attn_fwd(Q, K, V, lst, Lkv=Lkv, block=block, scale=0.4, qids=[i])
        Op.append(o[0]); Lp.append(l[0])
    for h in range(Hq):
        O, L = oracle.lse_merge(np.stack([o[h] for o in Op]), np.array([l[h] for l in Lp]))
        assert np.max(np.abs(O - Ow[0, h])) < 1e-12
        assert abs(L - Lw[0, h]) < 1e-12
    # a plain average is not the merge
    avg = np.mean([o[0] for o in Op], axis=0)
    assert np.max(np.abs(avg - Ow[0, 0])) > 1e-3


def test_worked_example_reverse_index():
    with open(os.path.join(GOLDEN, "worked_example_reverse_index.json")) as f:
        ex = json.load(f)
    N, Hkv, topK = ex["N"], ex["Hkv"], ex["topK"]
    idx = np.full((N, Hkv, topK), -1, np.int32)
    idx[ex["query"], 0] = ex["list"]
    s = oracle.schedule(idx, Lkv=ex["Lkv"], block=ex["block"])
    nonempty = [r for r in range(len(s["counts"])) if s["counts"][r] > 0]
    assert nonempty == ex["expected_rows"]
    for r, k in zip(ex["expected_rows"], ex["expected_slots"]):
        p = s["offsets"][r]
        assert s["qlist"][p] == ex["query"] and s["slot"][p] == k
        assert s["cmap"][ex["query"], 0, k] == p
    assert s["E"] == 3 and s["nsb"] == 3


def brute_schedule(idx, Lkv, block):
    N, Hkv, topK = idx.shape
    nb = Lkv // block
    rows = []
    for g in range(Hkv):
        for b in range(nb):
            ent = []
            for i in range(N):
                lb = (Lkv - N + i) // block
                lst = [int(x) for x in idx[i, g]]
                if b <= lb and b in lst:
                    ent.append((i, lst.index(b)))
            rows.append(ent)
    return rows


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_schedule_bruteforce_and_invariants(seed):
    rng = np.random.default_rng(10 + seed)
    N, Lkv, Hkv, topK, block = 50, 80, 2, 6, 8
    nb = Lkv // block
    idx = rng.integers(-1, nb, size=(N, Hkv, topK)).astype(np.int32)
    s = oracle.schedule(idx, Lkv=Lkv, block=block)
    rows = brute_schedule(idx, Lkv, block)
    assert [len(r) for r in rows] == list(s["counts"])
    for r, ent in enumerate(rows):
        a, b = s["offsets"][r], s["offsets"][r + 1]
        assert list(zip(s["qlist"][a:b], s["slot"][a:b])) == ent
    E = s["E"]
    assert s["counts"].sum() == E == s["offsets"][-1]
    assert s["nsb"] == int((s["counts"] > 0).sum())
    cm = s["cmap"].reshape(-1)
    valid = cm[cm >= 0]
    assert sorted(valid.tolist()) == list(range(E))  # bijection onto [0, E)
    assert (s["cmap"] >= 0).sum(axis=2).max() <= topK
    for p in range(E):  # cmap inverts (qlist, slot)
        i, k = s["qlist"][p], s["slot"][p]
        r = np.searchsorted(s["offsets"], p, side="right") - 1
        g = r // nb
        assert s["cmap"][i, g, k] == p
    assert s["status"] == 0


def test_schedule_invalid_ids_flagged():
    idx = np.array([[[0, 9, -2]]], np.int32)  # nblocks = 2
    s = oracle.schedule(idx, Lkv=16, block=8)
    assert s["status"] == 1 and s["E"] == 1


def test_worklist_golden_windows():
    """The window-ordered work list against a hand-derived example: a short last
    window, a row whose entries span both windows, an empty segment and segments cut
    into tiles of 8 with a ragged last tile (tests/golden/worklist_windows.json)."""
    with open(os.path.join(GOLDEN, "worklist_windows.json")) as f:
        ex = json.load(f)
    N, Lkv, block = ex["N"], ex["Lkv"], ex["block"]
    lb = (Lkv - N + np.arange(N)) // block
    idx = np.full((N, ex["Hkv"], ex["topK"]), -1, np.int32)
    idx[:, 0, 0] = lb
    idx[ex["second_block_zero_queries"], 0, 1] = 0
    s = oracle.schedule(idx, Lkv=Lkv, block=block)
    assert s["E"] == ex["expected_E"] and s["offsets"].tolist() == ex["expected_offsets"]
    tiles, wt = oracle.worklist(s["offsets"], s["qlist"], N, window=ex["window"], tile_rows=ex["tile"])
    assert wt.tolist() == ex["expected_window_tiles"]
    assert tiles.tolist() == ex["expected_tiles"]


@pytest.mark.parametrize("seed,N,Lkv,Hkv,window", [(0, 700, 1024, 2, 256), (1, 256, 512, 1, 256), (2, 97, 2048, 3, 32),
                                                   (3, 1, 128, 1, 256)])
def test_worklist_invariants(seed, N, Lkv, Hkv, window):
    """Every CSR entry in exactly one tile; a tile holds 1..8 consecutive entries of one
    row whose queries all lie in its window; only a segment's last tile is short; tiles
    ordered by (window, row, first); window_tiles brackets each window's tiles."""
    rng = np.random.default_rng(40 + seed)
    nb, topK = Lkv // 128, 5
    idx = rng.integers(-1, nb, size=(N, Hkv, topK)).astype(np.int32)
    s = oracle.schedule(idx, Lkv=Lkv)
    tiles, wt = oracle.worklist(s["offsets"], s["qlist"], N, window=window)
    E, R, nW = s["E"], len(s["counts"]), (N + window - 1) // window
    assert len(wt) == nW + 1 and wt[0] == 0 and wt[-1] == len(tiles)
    seen = np.zeros(E, np.int64)
    row_of = np.repeat(np.arange(R), s["counts"])
    seg_len = {}
    for t, (r, first, cnt, w) in enumerate(tiles.tolist()):
        assert wt[w] <= t < wt[w + 1] and 1 <= cnt <= 8
        assert s["offsets"][r] <= first and first + cnt <= s["offsets"][r + 1]
        for p in range(first, first + cnt):
            seen[p] += 1
            assert row_of[p] == r and s["qlist"][p] // window == w
        seg_len.setdefault((w, r), []).append(cnt)
    assert np.all(seen == 1)
    for lens in seg_len.values():
        assert all(c == 8 for c in lens[:-1])
    keys = [(w, r, f) for r, f, _, w in tiles.tolist()]
    assert keys == sorted(keys) and len(set(keys)) == len(keys)


def test_dispatch_threshold():
    """KV-outer when 10 E - 13 nsb > 35000, evaluated by hand at and around the boundary."""
    assert oracle.dispatch(3500, 0) == 2 and oracle.dispatch(3501, 0) == 1  # 35000 is not above
    assert oracle.dispatch(3536, 28) == 2 and oracle.dispatch(3537, 28) == 1  # 34996 / 35006
    assert oracle.dispatch(4600, 1000) == 2 and oracle.dispatch(4600, 846) == 1  # 33000 / 35002
    # the workloads: M3 (E 462848, nsb 256) and the low-reuse one (E 16384, nsb 9980: 34100)
    assert oracle.dispatch(462848, 256) == 1 and oracle.dispatch(16384, 9980) == 2
    # a larger nsb favours Q-outer, a larger E KV-outer (the signs of the two terms)
    assert oracle.dispatch(10_000, 4999) == 1 and oracle.dispatch(10_000, 4999 + 3848) == 2  # 35013 / -11


def test_e4m3_decoder_matches_library_cast():
    """The spec-written E4M3 decoder agrees with torch's float8_e4m3fn on all 256 codes."""
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    lib = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    ours = np.array([oracle.e4m3_decode(i) for i in range(256)])
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(ours)) and nan.sum() == 2
    assert np.array_equal(lib[~nan], ours[~nan])
    assert oracle.e4m3_decode(0x7E) == 448.0 and oracle.e4m3_decode(0x01) == 2.0 ** -9


def test_bf16_decoder_matches_library_cast():
    """The bf16 decoder agrees with torch's bfloat16 -> float64 cast on all 65,536 codes."""
    codes = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    lib = torch.from_numpy(codes.view(np.int16).copy()).view(torch.bfloat16).to(torch.float64).numpy()
    ours = np.array([oracle.bf16_decode(int(u)) for u in codes])
    nan = np.isnan(lib)
    assert np.array_equal(nan, np.isnan(ours)) and nan.sum() == 2 * 127
    assert np.array_equal(lib[~nan], ours[~nan])
    assert np.array_equal(np.signbit(lib[~nan]), np.signbit(ours[~nan]))


def test_fp8_path_equals_decoded_f64():
    """e4m3 bytes + descales give the same result as their decoded values in float64."""
    rng = np.random.default_rng(8)
    N = Lkv = 256
    Hq, Hkv, D, block = 4, 2, 16, 64
    qb = torch.from_numpy(rng.standard_normal((N, Hq, D)).astype(np.float32)).to(torch.float8_e4m3fn)
    kb = torch.from_numpy(rng.standard_normal((Lkv, Hkv, D)).astype(np.float32)).to(torch.float8_e4m3fn)
    vb = torch.from_numpy(rng.standard_normal((Lkv, Hkv, D)).astype(np.float32)).to(torch.float8_e4m3fn)
    idx = full_lists(N, Lkv, Hkv, block, topK=3)
    dq, dk, dv = 0.5, 0.25, 2.0
    O8, L8, _ = oracle.attn_fwd(qb.view(torch.uint8).numpy(), kb.view(torch.uint8).numpy(),
                                vb.view(torch.uint8).numpy(), idx, Lkv=Lkv, block=block,
                                scale=0.3, q_descale=dq, k_descale=dk, v_descale=dv)
    Qf, Kf, Vf = (t.to(torch.float64).numpy() for t in (qb, kb, vb))
    O, L, _ = oracle.attn_fwd(Qf * dq, Kf * dk, Vf * dv, idx, Lkv=Lkv, block=block, scale=0.3)
    np.testing.assert_allclose(O8, O, atol=1e-12)
    np.testing.assert_allclose(L8, L, atol=1e-12)


def test_bf16_path_equals_decoded_f64():
    rng = np.random.default_rng(9)
    N = Lkv = 256
    Hq, Hkv, D, block = 4, 1, 16, 64
    ts = [torch.from_numpy(rng.standard_normal(s).astype(np.float32)).to(torch.bfloat16)
          for s in ((N, Hq, D), (Lkv, Hkv, D), (Lkv, Hkv, D))]
    bits = [t.view(torch.int16).numpy().view(np.uint16) for t in ts]
    idx = full_lists(N, Lkv, Hkv, block, topK=2)
    Ob, Lb, _ = oracle.attn_fwd(*bits, idx, Lkv=Lkv, block=block, scale=0.3)
    O, L, _ = oracle.attn_fwd(*(t.to(torch.float64).numpy() for t in ts), idx, Lkv=Lkv,
                              block=block, scale=0.3)
    assert np.array_equal(Ob, O) and np.array_equal(Lb, L)


# ---------------------------------------------------------------------------------
# Block selector R1 ("Sparse Attention", Chapter 4, "R1: One Representative"): pinned
# by closed forms on inputs built for them, by an invariance, and by the list rules.

def _r1(Q, K, Lkv, topK, block=32, tile=32):
    return oracle.select_r1(Q, K, Lkv=Lkv, topK=topK, block=block, tile=tile)


def test_select_r1_zero_queries_tie_rule():
    """Q = 0: every candidate scores 0, so after the forced own block the list is the
    candidates in ascending id order, padded with -1 when they run out."""
    N = Lkv = 128
    Q = np.zeros((N, 4, 8))
    K = np.random.default_rng(1).standard_normal((Lkv, 2, 8))
    idx, sc = _r1(Q, K, Lkv, topK=3)
    for t in range(4):  # tile t holds block t
        assert np.all(idx[32 * t:32 * t + 32, :, 0] == t)
        rest = [b for b in range(t)][:2]
        want = rest + [-1] * (2 - len(rest))
        assert np.all(idx[32 * t:32 * t + 32, :, 1:] == np.array(want))
        assert np.all(sc[t, :, :t] == 0.0) and np.all(np.isposinf(sc[t, :, t]))
        assert np.all(np.isneginf(sc[t, :, t + 1:]))


def test_select_r1_block_mean_and_head_max_closed_form():
    """Keys of block b of group 0 are j * (b + 1) * e0 (j = 0..31): the block mean is
    15.5 * (b + 1) * e0.  Only head 1 of the group has queries, all equal to 2 * e0, so
    its tile mean is 2 * e0 and the block score is max(0 (the other heads),
    31 * (b + 1)); group 1 has negative keys, so its scores are all 0."""
    N = Lkv = 128
    D, block = 4, 32
    Q = np.zeros((N, 4, D))
    Q[:, 1, 0] = 2.0
    K = np.zeros((Lkv, 2, D))
    for b in range(4):
        for j in range(32):
            K[b * 32 + j, 0, 0] = j * (b + 1)
            K[b * 32 + j, 1, 0] = -j * (b + 1)
    idx, sc = _r1(Q, K, Lkv, topK=4, block=block)
    t = 3  # the last tile sees blocks 0..2 as candidates
    np.testing.assert_allclose(sc[t, 0, :3], [31.0, 62.0, 93.0], rtol=0, atol=1e-12)
    np.testing.assert_allclose(sc[t, 1, :3], [0.0, 0.0, 0.0], atol=1e-12)
    assert list(idx[100, 0]) == [3, 2, 1, 0]
    assert list(idx[100, 1]) == [3, 0, 1, 2]


def test_select_r1_planted_block_is_chosen():
    """A block whose keys all equal a large multiple of the tile's mean query is chosen
    right after the forced own block, whatever the other blocks hold."""
    rng = np.random.default_rng(2)
    N = Lkv = 256
    D = 8
    Q = rng.standard_normal((N, 2, D)) * 0.1
    Q[192:224, 0, :] += 1.0  # tile 6: head 0 mean ~ ones
    K = rng.standard_normal((Lkv, 1, D)) * 0.1
    K[64:96, 0, :] = 10.0  # block 2
    idx, _ = _r1(Q, K, Lkv, topK=3)
    assert list(idx[200, 0, :2]) == [6, 2]


def test_select_r1_block_swap_equivariance():
    """Exchanging the keys of two candidate blocks exchanges their ids in every list."""
    rng = np.random.default_rng(3)
    N = Lkv = 256
    Q = rng.standard_normal((N, 4, 8))
    K = rng.standard_normal((Lkv, 2, 8))
    idx, _ = _r1(Q, K, Lkv, topK=5)
    K2 = K.copy()
    K2[32:64], K2[96:128] = K[96:128].copy(), K[32:64].copy()  # blocks 1 and 3
    idx2, _ = _r1(Q, K2, Lkv, topK=5)
    sw = idx.copy()
    sw[idx == 1], sw[idx == 3] = 3, 1
    # tiles 4.. see both blocks as candidates: the lists must match after the exchange
    assert np.array_equal(idx2[128:], sw[128:])


def test_select_r1_tail_queries_and_two_own_blocks():
    """Queries at the tail (N < Lkv) with a tile straddling two blocks: both blocks are
    forced, later blocks are never listed, a partial last tile uses its own mean."""
    rng = np.random.default_rng(4)
    N, Lkv = 80, 256  # positions 176..255; tiles of 32: [176..207] holds blocks 5 and 6
    Q = rng.standard_normal((N, 2, 8))
    K = rng.standard_normal((Lkv, 1, 8))
    idx, sc = _r1(Q, K, Lkv, topK=4)
    assert set(idx[0, 0, :2]) == {5, 6} and np.all(idx[0, 0] <= 6)
    assert np.all(np.isneginf(sc[0, 0, 7:]))
    # the last tile (queries 64..79, 16 queries) sees blocks 0..7
    assert idx[79, 0, 0] == 7 and np.all(idx[64:80] == idx[79])


# ----------------------------------------------------------------------------- selector R4
# "Sparse Attention", Chapter 4, "R4: Four Representatives": consecutive quarters of a query
# tile and of a key block are each summarised by their mean; the block score is the largest
# of the 16 quarter-pair dot products over the group's heads.

def _grid(rng, shape):
    """Small multiples of 1/8: sums and means of a few of them are exact in float64."""
    return rng.integers(-8, 9, size=shape).astype(np.float64) / 8


def test_select_r4_equals_r1_when_blocks_are_constant():
    rng = np.random.default_rng(21)
    N, Lkv, Hq, Hkv, D = 512, 1024, 4, 2, 8
    qv = _grid(rng, (N // 128, Hq, D))
    kv = _grid(rng, (Lkv // 128, Hkv, D))
    Q = np.repeat(qv, 128, axis=0)
    K = np.repeat(kv, 128, axis=0)
    i1, s1 = oracle.select_r1(Q, K, Lkv=Lkv, topK=5)
    i4, s4 = oracle.select_r4(Q, K, Lkv=Lkv, topK=5)
    assert np.array_equal(s1, s4) and np.array_equal(i1, i4)


def test_select_r4_closed_form_quarter_constants_and_short_tile():
    """Q constant over each 32-query quarter, K over each 32-key quarter: the representatives
    are those constants, so the score is a maximum of explicit dot products.  N = 296: the
    last tile holds 40 queries (quarters 0 and 1, the second with 8 queries)."""
    rng = np.random.default_rng(22)
    N, Lkv, Hq, Hkv, D, G = 296, 768, 4, 2, 8, 2
    nq, nk = -(-N // 32), Lkv // 32
    qv = _grid(rng, (nq, Hq, D))
    kv = _grid(rng, (nk, Hkv, D))
    Q = np.repeat(qv, 32, axis=0)[:N]
    K = np.repeat(kv, 32, axis=0)
    _, sc = oracle.select_r4(Q, K, Lkv=Lkv, topK=3)
    for t in range(-(-N // 128)):
        i0, i1 = 128 * t, min(128 * t + 128, N)
        quarters = [i0 // 32 + q for q in range(4) if i0 + 32 * q < i1]
        lb_first, lb_last = (Lkv - N + i0) // 128, (Lkv - N + i1 - 1) // 128
        for g in range(Hkv):
            for b in range(Lkv // 128):
                if b > lb_last:
                    assert sc[t, g, b] == -np.inf
                elif b >= lb_first:
                    assert sc[t, g, b] == np.inf
                else:
                    want = max(float(qv[q, h] @ kv[4 * b + r, g])
                               for h in range(g * G, (g + 1) * G) for q in quarters for r in range(4))
                    assert sc[t, g, b] == want, (t, g, b)


def test_select_r4_finds_a_quarter_that_r1_averages_away():
    """Block 2's mean key is zero, but its first 32 keys point along the queries: R1 scores it
    0 and misses it, R4 scores it highest."""
    rng = np.random.default_rng(23)
    N, Lkv, Hq, Hkv, D = 128, 1024, 2, 1, 8
    Q = np.zeros((N, Hq, D)); Q[:, :, 0] = 1.0
    K = 0.01 * rng.standard_normal((Lkv, Hkv, D))
    K[:, :, 0] = 0.1 * np.abs(rng.standard_normal((Lkv, Hkv)))  # every block mildly aligned
    K[256:288, :, 0] = 6.0
    K[288:384, :, 0] = -2.0                                       # block 2: mean 0 along e0
    K[256:384, :, 1:] = 0.0
    i1, _ = oracle.select_r1(Q, K, Lkv=Lkv, topK=3)
    i4, s4 = oracle.select_r4(Q, K, Lkv=Lkv, topK=3)
    assert 2 not in i1[0, 0].tolist()
    assert i4[0, 0, 1] == 2 and abs(s4[0, 0, 2] - 6.0) < 1e-12  # after the forced own block 7
