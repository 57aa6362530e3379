"""Shared helpers for the parity tests (no method arithmetic here)."""
import numpy as np

# Tolerances for bf16 inputs (fp32 accumulation) against the fp64 oracle.
BF16_REL_L2 = 1e-2
BF16_MAX_ABS = 2e-2
LSE_MAX_ABS = 1e-3
FP8_REL_L2 = 5e-2
WINDOW = 2048  # queries per work-list window of the library
TILE = 8      # CSR entries per tile


def compare_outputs(O_gpu, LSE_gpu, O_ref, LSE_ref):
    """rel-L2 and max-abs of O, max-abs of finite LSE; -inf LSE must match exactly."""
    Og = np.asarray(O_gpu, np.float64)
    Lg = np.asarray(LSE_gpu, np.float64)
    rel = np.linalg.norm(Og - O_ref) / max(np.linalg.norm(O_ref), 1e-30)
    mabs = float(np.abs(Og - O_ref).max()) if Og.size else 0.0
    inf_ref = np.isneginf(LSE_ref)
    assert np.array_equal(np.isneginf(Lg), inf_ref), "LSE -inf pattern differs"
    lerr = float(np.abs(Lg[~inf_ref] - LSE_ref[~inf_ref]).max()) if (~inf_ref).any() else 0.0
    return float(rel), mabs, lerr


def check_worklist(exp, ref, N):
    """The windowed work list: every CSR entry exactly once, tiles of <= 8 entries of
    one row whose queries all lie in the tile's window, ordered (window, row, first),
    and as many tiles as the sum over (window, row) of ceil(count / 8)."""
    tiles = np.asarray(exp["tiles"], np.int64).reshape(-1, 4)
    wt = np.asarray(exp["window_tiles"], np.int64)
    offsets = np.asarray(ref["offsets"], np.int64)
    qlist = np.asarray(ref["qlist"], np.int64)
    counts = np.asarray(ref["counts"], np.int64)
    E, R = int(ref["E"]), len(counts)
    nW = (N + WINDOW - 1) // WINDOW
    T = len(tiles)
    assert len(wt) == nW + 1 and wt[0] == 0 and wt[-1] == T
    win_of_q = qlist // WINDOW
    row_of_p = np.repeat(np.arange(R), counts)
    _, seg_counts = np.unique(row_of_p * nW + win_of_q, return_counts=True)
    assert T == int(((seg_counts + TILE - 1) // TILE).sum())
    if T == 0:
        return
    row, first, cnt, w = tiles[:, 0], tiles[:, 1], tiles[:, 2], tiles[:, 3]
    t = np.arange(T)
    assert np.all((wt[w] <= t) & (t < wt[w + 1]))
    assert np.all((cnt >= 1) & (cnt <= TILE))
    assert np.all((offsets[row] <= first) & (first + cnt <= offsets[row + 1]))
    ent = np.repeat(first, cnt) + (np.arange(int(cnt.sum())) - np.repeat(np.cumsum(cnt) - cnt, cnt))
    assert np.all(np.bincount(ent, minlength=E) == 1)
    assert np.all(win_of_q[ent] == np.repeat(w, cnt))
    key = (w * (R + 1) + row) * (E + 1) + first
    assert np.all(np.diff(key) > 0)

# Backward (bf16 inputs and outputs, fp32 accumulation, bf16 P / dS operands and bf16
# per-block dQ contributions) against the fp64 oracle: relative L2 per gradient tensor.
BWD_REL_L2 = 2e-2


def rel_l2(x, ref):
    x = np.asarray(x, np.float64)
    return float(np.linalg.norm(x - ref) / max(np.linalg.norm(ref), 1e-30))
