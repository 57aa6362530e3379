"""Oracle for block-sparse GQA attention: a plain fp64 CPU statement of the method.

TEST INFRASTRUCTURE.  Only the test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  It shares no code with
the CUDA library (``block_sparse_gqa_gb300``) and neither imports the other.

The arithmetic lives in ``msa_oracle.c`` (compiled with gcc, no fast-math); this
module only builds it and marshals numpy arrays.  See that file's header for the
passages each function follows and the readings taken where the pages are silent.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "msa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

FMT_BF16, FMT_E4M3, FMT_F64 = 0, 1, 2
DISPATCH_KV_OUTER, DISPATCH_Q_OUTER = 1, 2

_lib = None


def build(force: bool = False) -> str:
    """Compile msa_oracle.c into liboracle.so next to it (IEEE double, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fPIC", "-shared", "-fno-fast-math",
                               "-ffp-contract=off", "-o", tmp, _SRC, "-lm", "-lpthread"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        i32, i64, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_double
        lib.oracle_attn_fwd.restype = i32
        lib.oracle_attn_fwd.argtypes = [P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32,
                                        f64, f64, f64, f64, P, i32, P, P, i32]
        lib.oracle_schedule.restype = i32
        lib.oracle_schedule.argtypes = [P, i32, i32, i32, i32, i32, P, P, P, P, P, P, P]
        lib.oracle_worklist.restype = ctypes.c_long
        lib.oracle_worklist.argtypes = [P, P, i32, i32, i32, i32, P, P, ctypes.c_long]
        lib.oracle_lse_merge.restype = None
        lib.oracle_lse_merge.argtypes = [i32, i32, P, P, P, P]
        lib.oracle_bf16_decode.restype = f64
        lib.oracle_bf16_decode.argtypes = [ctypes.c_uint16]
        lib.oracle_e4m3_decode.restype = f64
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.oracle_dispatch.restype = i32
        lib.oracle_dispatch.argtypes = [ctypes.c_int64, ctypes.c_int32]
        lib.oracle_attn_bwd.restype = i32
        lib.oracle_attn_bwd.argtypes = [P, P, P, P, i32, P, i32, i32, i32, i32, i32, i32, i32, f64,
                                        P, i32, P, P, i32, P, P, i32]
        lib.oracle_select_r1.restype = i32
        lib.oracle_select_r1.argtypes = [P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32, P, P]
        lib.oracle_select_r4.restype = i32
        lib.oracle_select_r4.argtypes = [P, P, i32, i32, i32, i32, i32, i32, i32, i32, i32, P, P]
        _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _fmt_of(a: np.ndarray) -> int:
    if a.dtype == np.uint16:
        return FMT_BF16
    if a.dtype == np.uint8:
        return FMT_E4M3
    if a.dtype == np.float64:
        return FMT_F64
    raise TypeError(f"oracle inputs are bf16 bits (uint16), e4m3 bytes (uint8) or float64, got {a.dtype}")


def attn_fwd(Q, K, V, indices, *, Lkv, block=128, scale, q_descale=1.0, k_descale=1.0,
             v_descale=1.0, qids=None, nthreads=None):
    """O [nq,Hq,D] and LSE [nq,Hq] (float64) for the queries ``qids`` (default: all).

    Q [N,Hq,D], K/V [Lkv,Hkv,D] as bf16 bit patterns (uint16), e4m3 bytes (uint8) or
    float64; indices [N,Hkv,topK] int32.  Returns (O, LSE, status) with status 1 when
    an invalid block id (>= nblocks or < -1) was seen and ignored.
    """
    lib = _load()
    Q = np.ascontiguousarray(Q); K = np.ascontiguousarray(K); V = np.ascontiguousarray(V)
    fmt = _fmt_of(Q)
    if _fmt_of(K) != fmt or _fmt_of(V) != fmt:
        raise TypeError("Q, K and V must share one storage format")
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    N, Hq, D = Q.shape
    Hkv = K.shape[1]
    topK = indices.shape[2]
    assert K.shape == (Lkv, Hkv, D) and V.shape == K.shape and indices.shape == (N, Hkv, topK)
    if qids is None:
        qids = np.arange(N, dtype=np.int32)
    qids = np.ascontiguousarray(qids, dtype=np.int32)
    nq = len(qids)
    O = np.zeros((nq, Hq, D), np.float64)
    LSE = np.zeros((nq, Hq), np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    st = lib.oracle_attn_fwd(_ptr(Q), _ptr(K), _ptr(V), fmt, _ptr(indices), N, Lkv, Hq, Hkv, D,
                             topK, block, float(scale), float(q_descale), float(k_descale),
                             float(v_descale), _ptr(qids), nq, _ptr(O), _ptr(LSE), int(nthreads))
    if st < 0:
        raise ValueError("oracle_attn_fwd rejected its arguments")
    return O, LSE, st


def attn_bwd(Q, K, V, dO, indices, *, Lkv, block=128, scale, qids=None, rows=None, nthreads=None):
    """Gradients of the forward's O contracted with dO (float64).

    Q, dO [N,Hq,D], K/V [Lkv,Hkv,D] as bf16 bit patterns (uint16) or float64;
    indices [N,Hkv,topK] int32.  Returns (dQ, dK, dV, status): dQ [nq,Hq,D] for the
    queries ``qids`` (default all; ``qids=()`` skips dQ); dK and dV for the schedule
    rows ``rows`` (row r = g * nblocks + b, default all; ``rows=()`` skips them) as
    [nrows, block, D], or as [Lkv, Hkv, D] when ``rows`` is None.
    """
    lib = _load()
    Q, K, V, dO = (np.ascontiguousarray(a) for a in (Q, K, V, dO))
    fmt = _fmt_of(Q)
    if any(_fmt_of(a) != fmt for a in (K, V, dO)) or fmt == FMT_E4M3:
        raise TypeError("Q, K, V and dO must share one storage format (bf16 bits or float64)")
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    N, Hq, D = Q.shape
    Hkv = K.shape[1]
    topK = indices.shape[2]
    nblocks = Lkv // block
    assert K.shape == (Lkv, Hkv, D) and V.shape == K.shape and dO.shape == Q.shape
    assert indices.shape == (N, Hkv, topK)
    full_rows = rows is None
    qids = np.arange(N, dtype=np.int32) if qids is None else np.ascontiguousarray(qids, dtype=np.int32)
    rows = np.arange(Hkv * nblocks, dtype=np.int32) if rows is None else np.ascontiguousarray(rows, dtype=np.int32)
    nq, nr = len(qids), len(rows)
    dQ = np.zeros((nq, Hq, D), np.float64)
    dK = np.zeros((nr, block, D), np.float64)
    dV = np.zeros((nr, block, D), np.float64)
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    st = lib.oracle_attn_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), fmt, _ptr(indices), N, Lkv, Hq, Hkv, D,
                             topK, block, float(scale), _ptr(qids), nq, _ptr(dQ) if nq else None,
                             _ptr(rows), nr, _ptr(dK) if nr else None, _ptr(dV) if nr else None,
                             int(nthreads))
    if st < 0:
        raise ValueError("oracle_attn_bwd rejected its arguments")
    if full_rows:
        # row r = g * nblocks + b holds keys b*block.. of group g
        dK = dK.reshape(Hkv, nblocks, block, D).transpose(1, 2, 0, 3).reshape(Lkv, Hkv, D)
        dV = dV.reshape(Hkv, nblocks, block, D).transpose(1, 2, 0, 3).reshape(Lkv, Hkv, D)
    return dQ, dK, dV, st


def schedule(indices, *, Lkv, block=128):
    """Reverse index of the lists: dict with counts, offsets, qlist, slot, cmap, E, nsb, status."""
    lib = _load()
    indices = np.ascontiguousarray(indices, dtype=np.int32)
    N, Hkv, topK = indices.shape
    nblocks = Lkv // block
    R = Hkv * nblocks
    cap = max(N * Hkv * topK, 1)
    counts = np.zeros(R, np.int32)
    offsets = np.zeros(R + 1, np.int32)
    qlist = np.zeros(cap, np.int32)
    slot = np.zeros(cap, np.int32)
    cmap = np.zeros((N, Hkv, topK), np.int32)
    E = ctypes.c_int64(0)
    nsb = ctypes.c_int32(0)
    st = lib.oracle_schedule(_ptr(indices), N, Lkv, Hkv, topK, block, _ptr(counts), _ptr(offsets),
                             _ptr(qlist), _ptr(slot), _ptr(cmap), ctypes.byref(E), ctypes.byref(nsb))
    E = int(E.value)
    return dict(counts=counts, offsets=offsets, qlist=qlist[:E].copy(), slot=slot[:E].copy(),
                cmap=cmap, E=E, nsb=int(nsb.value), status=int(st))


def worklist(offsets, qlist, N, window=256, tile_rows=8):
    """Window-ordered tiles of a schedule's CSR: (tiles [T, 4] as (row, first, count,
    window), window_tiles [nW + 1])."""
    lib = _load()
    offsets = np.ascontiguousarray(offsets, dtype=np.int32)
    qlist = np.ascontiguousarray(qlist, dtype=np.int32)
    R = len(offsets) - 1
    nW = (N + window - 1) // window
    E = int(offsets[-1])
    cap = E + R * nW + 1
    tiles = np.zeros((cap, 4), np.int32)
    wt = np.zeros(nW + 1, np.int32)
    T = lib.oracle_worklist(_ptr(offsets), _ptr(qlist if len(qlist) else np.zeros(1, np.int32)), R, N, window,
                            tile_rows, _ptr(tiles), _ptr(wt), cap)
    assert T >= 0
    return tiles[:T].copy(), wt


def lse_merge(O_parts, lse_parts):
    """Merge n partial (O_k [n,D], lse_k [n]) results of one (query, head)."""
    lib = _load()
    O_parts = np.ascontiguousarray(O_parts, dtype=np.float64)
    lse_parts = np.ascontiguousarray(lse_parts, dtype=np.float64)
    n, D = O_parts.shape
    O = np.zeros(D, np.float64)
    lse = ctypes.c_double(0.0)
    lib.oracle_lse_merge(n, D, _ptr(O_parts), _ptr(lse_parts), _ptr(O), ctypes.byref(lse))
    return O, lse.value


def bf16_decode(bits: int) -> float:
    return _load().oracle_bf16_decode(int(bits))


def e4m3_decode(byte: int) -> float:
    return _load().oracle_e4m3_decode(int(byte))


def dispatch(E: int, nsb: int) -> int:
    """1 = KV-outer, 2 = Q-outer: KV-outer when 10 E - 13 nsb > 35000 (E CSR entries, nsb
    distinct (group, block) pairs; the GB300 re-derivation of the pages' crossover)."""
    return _load().oracle_dispatch(int(E), int(nsb))


def select_r4(Q, K, *, Lkv, topK, block=128, tile=128):
    """Block selector R4 ("Sparse Attention", Chapter 4): as select_r1 with four
    representatives (means of consecutive quarters) per query tile and per KV block."""
    return _select(_load().oracle_select_r4, "oracle_select_r4", Q, K, Lkv, topK, block, tile)


def select_r1(Q, K, *, Lkv, topK, block=128, tile=128):
    """Block selector R1 ("Sparse Attention", Chapter 4): (indices [N, Hkv, topK] int32,
    scores [ntiles, Hkv, nblocks] float64 with +inf for the tile's own blocks and -inf
    for blocks after the tile).  Q [N, Hq, D], K [Lkv, Hkv, D] as bf16 bit patterns
    (uint16) or float64."""
    return _select(_load().oracle_select_r1, "oracle_select_r1", Q, K, Lkv, topK, block, tile)


def _select(fn, name, Q, K, Lkv, topK, block, tile):
    Q = np.ascontiguousarray(Q); K = np.ascontiguousarray(K)
    fmt = _fmt_of(Q)
    if _fmt_of(K) != fmt:
        raise TypeError("Q and K must share one storage format")
    N, Hq, D = Q.shape
    Hkv = K.shape[1]
    assert K.shape == (Lkv, Hkv, D)
    nblocks = Lkv // block
    ntiles = -(-N // tile)
    idx = np.zeros((N, Hkv, topK), np.int32)
    scores = np.zeros((ntiles, Hkv, nblocks), np.float64)
    st = fn(_ptr(Q), _ptr(K), fmt, N, Lkv, Hq, Hkv, D, block, tile, topK, _ptr(idx), _ptr(scores))
    if st < 0:
        raise ValueError(f"{name} rejected its arguments")
    return idx, scores
