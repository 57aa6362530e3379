"""Seeded synthetic inputs for block-sparse GQA attention.

This module is shared by the tests, the benchmark and the smoke check; it feeds both
the CUDA library and the oracle and holds none of the method's arithmetic: only
random draws, round-to-nearest-even casts of the drawn values to the storage types,
and per-tensor fp8 quantisation of the inputs.

Workloads (one per named configuration, seed = 1000 + its index):

  tiny      N = Lkv = 1024 (8 blocks), Hq 16, Hkv 1, topK 4; own block + up to 3
            distinct uniform earlier blocks.
  m3        N = Lkv = 8192 (64 blocks), Hq 64, Hkv 4, topK 16 (the MiniMax M3 shape of
            "Kernel optimization for MiniMax M3 on NVIDIA Blackwell"); own block + up
            to 15 distinct uniform earlier blocks per (query, group).
  long      N = 32768 queries at the tail of Lkv = 131072; lists shared by runs of 64
            consecutive queries; 15 distinct earlier blocks drawn without replacement
            with P(b) proportional to (b + 1)^-1.2 (Zipf, s = 1.2, rank = block id + 1).
  lowreuse  N = 256 queries at the tail of Lkv = 524288; 15 distinct uniform earlier
            blocks per (query, group), independent.
  fp8       N = Lkv = 65536 (512 blocks); own block + 15 distinct picks
            b = round(lb + 32 z), z ~ N(0, 1), kept only in [0, lb); Q/K/V quantised
            per tensor to OCP E4M3 with fp32 descales (descale = amax / 448, RNE,
            saturating).

Q, K, V ~ N(0, 1) drawn in fp32 and rounded to bf16.  Every list starts with the
query's own block, then the picks in draw order, padded with -1.  Draws without
replacement use the Efraimidis-Spirakis exponential-key method (keys log(U)/w, largest
first), which reproduces successive weighted draws with duplicates rejected.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

BLOCK = 128
FP8_MAX = 448.0


@dataclass(frozen=True)
class Config:
    name: str
    N: int
    Lkv: int
    Hq: int
    Hkv: int
    D: int
    topK: int
    picks: str  # 'uniform' | 'zipf' | 'gauss'
    seed: int
    run: int = 1  # consecutive queries sharing one list
    dtype: str = "bf16"  # 'bf16' | 'e4m3'
    extra: dict = field(default_factory=dict)

    @property
    def nblocks(self) -> int:
        return self.Lkv // BLOCK

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def nominal_flops(self) -> float:
        """Useful FLOPs as 4 * N * Hq * topK * 128 * D (QK and PV, multiply-add = 2)."""
        return 4.0 * self.N * self.Hq * self.topK * BLOCK * self.D


CONFIGS = {
    "tiny": Config("tiny", 1024, 1024, 16, 1, 128, 4, "uniform", 1000),
    "m3": Config("m3", 8192, 8192, 64, 4, 128, 16, "uniform", 1001),
    "long": Config("long", 32768, 131072, 64, 4, 128, 16, "zipf", 1002, run=64),
    "lowreuse": Config("lowreuse", 256, 524288, 64, 4, 128, 16, "uniform", 1003),
    "fp8": Config("fp8", 65536, 65536, 64, 4, 128, 16, "gauss", 1004, dtype="e4m3",
                  extra={"sigma": 32.0}),
    # not one of the five configured workloads: one decode step (a single query at the tail
    # of a 128K-token context) for the decode-size study
    "decode": Config("decode", 1, 131072, 64, 4, 128, 16, "uniform", 1005),
}


def _ndtr(x: np.ndarray) -> np.ndarray:
    from scipy.special import ndtr
    return ndtr(x)


def _pick_weights(cfg: Config, lb: int) -> np.ndarray:
    b = np.arange(lb, dtype=np.float64)
    if cfg.picks == "uniform":
        return np.ones(lb)
    if cfg.picks == "zipf":
        return (b + 1.0) ** -1.2
    if cfg.picks == "gauss":
        s = cfg.extra["sigma"]
        return _ndtr((b + 0.5 - lb) / s) - _ndtr((b - 0.5 - lb) / s)
    raise ValueError(cfg.picks)


def make_indices(cfg: Config, seed: int | None = None) -> np.ndarray:
    """int32 [N, Hkv, topK]: own block first, then distinct earlier picks, -1 padded."""
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence(
        cfg.seed if seed is None else seed).spawn(4)[0]))
    N, Hkv, topK = cfg.N, cfg.Hkv, cfg.topK
    out = np.full((N, Hkv, topK), -1, np.int32)
    off = cfg.Lkv - N
    q = np.arange(N)
    lbs = (off + q) // BLOCK
    run = cfg.run
    for lb in np.unique(lbs):
        lb = int(lb)
        qs = q[lbs == lb]
        # one list per (run, group); runs never straddle a block (run divides 128 and
        # the tail offset is a multiple of 128 in every workload)
        runs = np.unique(qs // run)
        nl = len(runs) * Hkv
        npick = min(topK - 1, lb)
        lists = np.full((nl, topK), -1, np.int32)
        lists[:, 0] = lb
        if npick > 0:
            w = _pick_weights(cfg, lb)
            u = rng.random((nl, lb))
            with np.errstate(divide="ignore"):
                keys = np.log(u) / w[None, :]
            order = np.argsort(-keys, axis=1, kind="stable")[:, :npick]
            lists[:, 1:1 + npick] = order.astype(np.int32)
        lists = lists.reshape(len(runs), Hkv, topK)
        run_of = {int(r): k for k, r in enumerate(runs)}
        ridx = np.array([run_of[int(i // run)] for i in qs])
        out[qs] = lists[ridx]
    return out


def _normal(seed_seq, shape) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(seed_seq))
    return rng.standard_normal(shape, dtype=np.float32)


def quantize_e4m3(x: torch.Tensor):
    """Per-tensor E4M3 quantisation of a float32 tensor: (bytes uint8, descale float)."""
    amax = float(x.abs().max())
    descale = amax / FP8_MAX if amax > 0 else 1.0
    q = (x / descale).clamp_(-FP8_MAX, FP8_MAX).to(torch.float8_e4m3fn)
    return q.view(torch.uint8), descale


@dataclass
class Workload:
    cfg: Config
    indices: torch.Tensor  # int32 [N,Hkv,topK] (CPU)
    Q: torch.Tensor        # bf16 [N,Hq,D] or uint8 e4m3 bytes (CPU)
    K: torch.Tensor        # [Lkv,Hkv,D]
    V: torch.Tensor
    q_descale: float = 1.0
    k_descale: float = 1.0
    v_descale: float = 1.0

    def np_inputs(self):
        """Q, K, V as the oracle reads them: bf16 bit patterns (uint16) or e4m3 bytes."""
        if self.cfg.dtype == "bf16":
            return tuple(t.view(torch.int16).numpy().view(np.uint16) for t in (self.Q, self.K, self.V))
        return tuple(t.numpy() for t in (self.Q, self.K, self.V))


def make_workload(cfg: Config | str, seed: int | None = None, with_qkv: bool = True) -> Workload:
    if isinstance(cfg, str):
        cfg = CONFIGS[cfg]
    s = cfg.seed if seed is None else seed
    ss = np.random.SeedSequence(s).spawn(4)
    idx = torch.from_numpy(make_indices(cfg, s))
    if not with_qkv:
        e = torch.empty(0)
        return Workload(cfg, idx, e, e, e)
    shapes = [(cfg.N, cfg.Hq, cfg.D), (cfg.Lkv, cfg.Hkv, cfg.D), (cfg.Lkv, cfg.Hkv, cfg.D)]
    xs = [torch.from_numpy(_normal(ss[1 + t], shapes[t])) for t in range(3)]
    if cfg.dtype == "bf16":
        Q, K, V = (x.to(torch.bfloat16) for x in xs)
        return Workload(cfg, idx, Q, K, V)
    (Q, dq), (K, dk), (V, dv) = (quantize_e4m3(x) for x in xs)
    return Workload(cfg, idx, Q, K, V, dq, dk, dv)


def sample_queries(cfg: Config, n: int, seed: int = 7) -> np.ndarray:
    """Seeded sorted query subset including the first and last 128-query blocks' edges."""
    rng = np.random.Generator(np.random.PCG64(seed))
    chosen = {0, 1, min(127, cfg.N - 1), cfg.N - 1, max(cfg.N - 128, 0)}
    want = max(n, len(chosen))
    for x in rng.choice(cfg.N, size=min(n, cfg.N), replace=False):
        if len(chosen) >= want:
            break
        chosen.add(int(x))
    return np.array(sorted(chosen), np.int32)
