"""block_sparse_gqa_gb300: ctypes binding over libmsa (see include/msa.h).

Argument marshalling only: every step of the forward (schedule, attention,
combine) runs in the CUDA kernels of libmsa.so.  PyTorch supplies device memory
and streams.  There is no CPU fallback: if libmsa.so is missing or CUDA is not
available, the calls raise.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
# MSA_LIBRARY=debug selects the bounds-checked build (same entry points; see msa_debug_build)
LIB_PATH = os.path.join(_HERE, "libmsa_debug.so" if os.environ.get("MSA_LIBRARY") == "debug" else "libmsa.so")

MSA_OK = 0
STATUS_NAMES = {0: "MSA_OK", 1: "MSA_ERR_INVALID_ARG", 2: "MSA_ERR_UNSUPPORTED", 3: "MSA_ERR_CUDA",
                4: "MSA_ERR_OOM", 5: "MSA_ERR_BAD_INDEX", 6: "MSA_ERR_TIMEOUT", 7: "MSA_ERR_CAPACITY",
                8: "MSA_ERR_BOUNDS"}
DTYPE_BF16, DTYPE_FP8_E4M3 = 0, 1
PATHS = {"auto": 0, "kv_outer": 1, "q_outer": 2}
EXPORTED = ["msa_fwd_opts_init", "msa_build_schedule", "msa_sparse_attn_fwd", "msa_schedule_destroy",
            "msa_schedule_query", "msa_schedule_export", "msa_status_string", "msa_last_cuda_error",
            "msa_version", "msa_debug_build"]


class MsaError(RuntimeError):
    def __init__(self, status: int, what: str, text: str = ""):
        self.status = status
        super().__init__(f"{what}: {STATUS_NAMES.get(status, status)} ({text})")


class Tensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int), ("n", ctypes.c_int64),
                ("h", ctypes.c_int64), ("d", ctypes.c_int64)]


class FwdOpts(ctypes.Structure):
    _fields_ = [("stream", ctypes.c_void_p), ("path", ctypes.c_int), ("q_descale", ctypes.c_float),
                ("k_descale", ctypes.c_float), ("v_descale", ctypes.c_float),
                ("stage_events", ctypes.c_void_p * 3), ("num_ctas", ctypes.c_int), ("partials_fp32", ctypes.c_int),
                ("debug_flags", ctypes.c_int)]


class ScheduleInfo(ctypes.Structure):
    _fields_ = [("entries", ctypes.c_int64), ("nsb", ctypes.c_int32), ("ntiles", ctypes.c_int32),
                ("path", ctypes.c_int32), ("status", ctypes.c_int32), ("rows", ctypes.c_int32),
                ("windows", ctypes.c_int32)]


_lib = None


def lib() -> ctypes.CDLL:
    """Load libmsa.so (built by __graft_entry__.build()); raise if it is not there."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is not built; run `python -c 'import __graft_entry__ as g; g.build()'`")
        L = ctypes.CDLL(LIB_PATH)
        P, I = ctypes.c_void_p, ctypes.c_int
        L.msa_fwd_opts_init.restype = None
        L.msa_fwd_opts_init.argtypes = [ctypes.POINTER(FwdOpts)]
        L.msa_build_schedule.restype = I
        L.msa_build_schedule.argtypes = [P, I, I, I, I, P, ctypes.POINTER(P)]
        L.msa_sparse_attn_fwd.restype = I
        L.msa_sparse_attn_fwd.argtypes = [Tensor, Tensor, Tensor, P, P, P, ctypes.c_float, ctypes.POINTER(FwdOpts)]
        L.msa_sparse_attn_bwd.restype = I
        L.msa_sparse_attn_bwd.argtypes = [Tensor, Tensor, Tensor, P, P, P, P, P, P, P, ctypes.c_float,
                                          ctypes.POINTER(FwdOpts)]
        L.msa_schedule_destroy.restype = I
        L.msa_schedule_destroy.argtypes = [P]
        L.msa_schedule_query.restype = I
        L.msa_schedule_query.argtypes = [P, ctypes.POINTER(ScheduleInfo)]
        L.msa_schedule_status.restype = I
        L.msa_schedule_status.argtypes = [P]
        L.msa_schedule_export.restype = I
        L.msa_schedule_export.argtypes = [P] + [P] * 7
        L.msa_status_string.restype = ctypes.c_char_p
        L.msa_status_string.argtypes = [I]
        L.msa_last_cuda_error.restype = I
        L.msa_last_cuda_error.argtypes = []
        L.msa_version.restype = I
        L.msa_version.argtypes = []
        L.msa_select_workspace_bytes.restype = ctypes.c_size_t
        L.msa_select_workspace_bytes.argtypes = [I, I, I, I]
        L.msa_sparse_attn_fwd_tiles.restype = I
        L.msa_sparse_attn_fwd_tiles.argtypes = [Tensor, Tensor, Tensor, P, I, I, P, P, ctypes.c_float, P,
                                                ctypes.POINTER(FwdOpts)]
        L.msa_select_blocks_r4.restype = I
        L.msa_select_blocks_r4.argtypes = [Tensor, Tensor, I, P, P, ctypes.c_size_t, P]
        L.msa_select_blocks_r1.restype = I
        L.msa_select_blocks_r1.argtypes = [Tensor, Tensor, I, P, P, ctypes.c_size_t, P]
        _lib = L
    return _lib


def _check(st: int, what: str):
    if st != MSA_OK:
        raise MsaError(st, what, lib().msa_status_string(st).decode())


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    if t.dtype in (torch.float8_e4m3fn, torch.uint8):
        return DTYPE_FP8_E4M3
    raise TypeError(f"unsupported dtype {t.dtype}")


def _tensor(t: torch.Tensor) -> Tensor:
    if not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
        raise ValueError("Q/K/V must be contiguous 3-D CUDA tensors [n, h, d]")
    return Tensor(t.data_ptr(), _dtype_code(t), t.shape[0], t.shape[1], t.shape[2])


@dataclass
class Schedule:
    """Handle to a device schedule (reverse index + work list) built from one indices tensor."""
    handle: int | None  # the msa_schedule_t pointer value
    N: int
    Hkv: int
    topK: int
    nblocks: int

    def query(self) -> dict:
        info = ScheduleInfo()
        st = lib().msa_schedule_query(self.handle, ctypes.byref(info))
        d = {k: getattr(info, k) for k, _ in ScheduleInfo._fields_}
        d["status_code"] = st
        return d

    def status(self) -> int:
        """msa_schedule_status: the sticky device status as an msa_status_t code (synchronises)."""
        return lib().msa_schedule_status(self.handle)

    def export(self) -> dict:
        """Host copies of the schedule arrays (synchronises)."""
        import numpy as np
        info = self.query()
        E, T, R, W = info["entries"], info["ntiles"], info["rows"], info["windows"]
        out = dict(counts=np.zeros(R, np.int32), offsets=np.zeros(R + 1, np.int32),
                   qlist=np.zeros(max(E, 1), np.int32), slot=np.zeros(max(E, 1), np.int32),
                   cmap=np.zeros((self.N, self.Hkv, self.topK), np.int32),
                   tiles=np.zeros((max(T, 1), 4), np.int32), window_tiles=np.zeros(W + 1, np.int32))
        ptrs = [out[k].ctypes.data_as(ctypes.c_void_p) for k in
                ("counts", "offsets", "qlist", "slot", "cmap", "tiles", "window_tiles")]
        st = lib().msa_schedule_export(self.handle, *ptrs)
        if st not in (MSA_OK, 5):
            _check(st, "msa_schedule_export")
        out["qlist"], out["slot"], out["tiles"] = out["qlist"][:E], out["slot"][:E], out["tiles"][:T]
        out.update(E=E, nsb=info["nsb"], ntiles=T, path=info["path"], status=info["status"])
        return out

    def close(self):
        if self.handle:
            _check(lib().msa_schedule_destroy(self.handle), "msa_schedule_destroy")
            self.handle = None

    def __del__(self):
        try:
            if self.handle:
                lib().msa_schedule_destroy(self.handle)
        except Exception:
            pass


def build_schedule(indices: torch.Tensor, nblocks: int, schedule: Schedule | None = None,
                   stream=None) -> Schedule:
    """msa_build_schedule on an int32 CUDA tensor [N, Hkv, topK]; reuses `schedule` if given."""
    if indices.dtype != torch.int32 or not indices.is_cuda or not indices.is_contiguous() or indices.dim() != 3:
        raise ValueError("indices must be a contiguous int32 CUDA tensor [N, Hkv, topK]")
    N, Hkv, topK = indices.shape
    h = ctypes.c_void_p(schedule.handle if schedule is not None else None)
    st = lib().msa_build_schedule(indices.data_ptr(), N, Hkv, topK, nblocks, _stream_ptr(stream), ctypes.byref(h))
    _check(st, "msa_build_schedule")
    if schedule is not None:
        return schedule
    return Schedule(h.value, N, Hkv, topK, nblocks)


def sparse_attn_bwd(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, O: torch.Tensor, dO: torch.Tensor,
                    LSE: torch.Tensor, schedule: Schedule, scale: float | None = None, dQ: torch.Tensor | None = None,
                    dK: torch.Tensor | None = None, dV: torch.Tensor | None = None, num_ctas: int = 0,
                    stage_events=None, stream=None):
    """msa_sparse_attn_bwd; returns (dQ bf16 [N,Hq,D], dK bf16 [Lkv,Hkv,D], dV bf16 [Lkv,Hkv,D])."""
    N, Hq, D = Q.shape
    if scale is None:
        scale = D ** -0.5
    for name, t, shape, dt in (("O", O, Q.shape, torch.bfloat16), ("dO", dO, Q.shape, torch.bfloat16),
                               ("LSE", LSE, (N, Hq), torch.float32)):
        if not t.is_cuda or not t.is_contiguous() or tuple(t.shape) != tuple(shape) or t.dtype != dt:
            raise ValueError(f"{name} must be a contiguous {dt} CUDA tensor of shape {tuple(shape)}")
    if dQ is None:
        dQ = torch.empty_like(Q, dtype=torch.bfloat16)
    if dK is None:
        dK = torch.empty(K.shape, dtype=torch.bfloat16, device=K.device)
    if dV is None:
        dV = torch.empty(V.shape, dtype=torch.bfloat16, device=V.device)
    opts = FwdOpts()
    lib().msa_fwd_opts_init(ctypes.byref(opts))
    opts.stream = _stream_ptr(stream)
    opts.num_ctas = int(num_ctas)
    if stage_events is not None:
        for k, ev in enumerate(stage_events[:3]):
            opts.stage_events[k] = ev
    st = lib().msa_sparse_attn_bwd(_tensor(Q), _tensor(K), _tensor(V), O.data_ptr(), dO.data_ptr(), LSE.data_ptr(),
                                   schedule.handle, dQ.data_ptr(), dK.data_ptr(), dV.data_ptr(), float(scale),
                                   ctypes.byref(opts))
    _check(st, "msa_sparse_attn_bwd")
    return dQ, dK, dV


def sparse_attn_fwd(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, schedule: Schedule, scale: float | None = None,
                    O: torch.Tensor | None = None, LSE: torch.Tensor | None = None, path: str = "auto",
                    descales=(1.0, 1.0, 1.0), stage_events=None, num_ctas: int = 0, partials_fp32: bool = False,
                    debug_flags: int = 0, stream=None):
    """msa_sparse_attn_fwd; returns (O bf16 [N,Hq,D], LSE fp32 [N,Hq])."""
    N, Hq, D = Q.shape
    if scale is None:
        scale = D ** -0.5
    if O is None:
        O = torch.empty((N, Hq, D), dtype=torch.bfloat16, device=Q.device)
    if LSE is None:
        LSE = torch.empty((N, Hq), dtype=torch.float32, device=Q.device)
    opts = FwdOpts()
    lib().msa_fwd_opts_init(ctypes.byref(opts))
    opts.stream = _stream_ptr(stream)
    opts.path = PATHS[path]
    opts.q_descale, opts.k_descale, opts.v_descale = (float(x) for x in descales)
    opts.num_ctas = int(num_ctas)
    opts.partials_fp32 = 1 if partials_fp32 else 0
    opts.debug_flags = int(debug_flags)
    if stage_events is not None:
        for k, ev in enumerate(stage_events[:3]):
            opts.stage_events[k] = ev
    st = lib().msa_sparse_attn_fwd(_tensor(Q), _tensor(K), _tensor(V), schedule.handle, O.data_ptr(),
                                   LSE.data_ptr(), float(scale), ctypes.byref(opts))
    _check(st, "msa_sparse_attn_fwd")
    return O, LSE


def select_blocks_r4(Q: torch.Tensor, K: torch.Tensor, topK: int, indices: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """msa_select_blocks_r4: as select_blocks_r1 with four quarter-mean representatives."""
    return select_blocks_r1(Q, K, topK, indices, workspace, stream, _entry="msa_select_blocks_r4")


def select_blocks_r1(Q: torch.Tensor, K: torch.Tensor, topK: int, indices: torch.Tensor | None = None,
                     workspace: torch.Tensor | None = None, stream=None,
                     _entry: str = "msa_select_blocks_r1") -> torch.Tensor:
    """msa_select_blocks_r1: int32 block lists [N, Hkv, topK] (device) for bf16 Q [N, Hq, 128]
    and K [Lkv, Hkv, 128]; the workspace is allocated here unless given."""
    N, Hq, _ = Q.shape
    Lkv, Hkv, _ = K.shape
    if indices is None:
        indices = torch.empty((N, Hkv, topK), dtype=torch.int32, device=Q.device)
    need = lib().msa_select_workspace_bytes(N, Hq, Hkv, Lkv // 128)
    if workspace is None:
        workspace = torch.empty(need + 256, dtype=torch.uint8, device=Q.device)
    ptr = workspace.data_ptr()
    aligned = (ptr + 255) // 256 * 256
    usable = max(0, workspace.numel() * workspace.element_size() - (aligned - ptr))
    st = getattr(lib(), _entry)(_tensor(Q), _tensor(K), int(topK), indices.data_ptr(), aligned, usable,
                                _stream_ptr(stream))
    _check(st, _entry)
    return indices


def sparse_attn_fwd_tiles(Q: torch.Tensor, K: torch.Tensor, V: torch.Tensor, tile_lists: torch.Tensor, tile: int,
                          scale: float | None = None, O: torch.Tensor | None = None, LSE: torch.Tensor | None = None,
                          status: torch.Tensor | None = None, num_ctas: int = 0, stream=None):
    """msa_sparse_attn_fwd_tiles: (O bf16 [N,Hq,D], LSE fp32 [N,Hq]) for int32 lists
    [ceil(N / tile), Hkv, topK] shared by `tile` consecutive queries."""
    N, Hq, D = Q.shape
    if scale is None:
        scale = D ** -0.5
    if O is None:
        O = torch.empty((N, Hq, D), dtype=torch.bfloat16, device=Q.device)
    if LSE is None:
        LSE = torch.empty((N, Hq), dtype=torch.float32, device=Q.device)
    if tile_lists.dtype != torch.int32 or not tile_lists.is_contiguous() or tile_lists.dim() != 3:
        raise ValueError("tile_lists must be a contiguous int32 tensor [ceil(N / tile), Hkv, topK]")
    opts = FwdOpts()
    lib().msa_fwd_opts_init(ctypes.byref(opts))
    opts.stream = _stream_ptr(stream)
    opts.num_ctas = int(num_ctas)
    st = lib().msa_sparse_attn_fwd_tiles(_tensor(Q), _tensor(K), _tensor(V), tile_lists.data_ptr(), int(tile),
                                         int(tile_lists.shape[2]), O.data_ptr(), LSE.data_ptr(), float(scale),
                                         status.data_ptr() if status is not None else None, ctypes.byref(opts))
    _check(st, "msa_sparse_attn_fwd_tiles")
    return O, LSE


def version() -> int:
    return lib().msa_version()
