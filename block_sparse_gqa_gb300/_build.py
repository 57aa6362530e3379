"""Builds libmsa.so in-tree with nvcc for sm_103a (one -gencode, parallel TUs)."""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
BUILD = os.path.join(HERE, "_build")
LIB = os.path.join(HERE, "libmsa.so")
LIB_DEBUG = os.path.join(HERE, "libmsa_debug.so")  # bounds-checked build (MSA_DEBUG=1)
SOURCES = ["msa_api.cu", "schedule.cu", "attn_kv_outer.cu", "combine.cu", "attn_q_outer.cu", "msa_noalloc.cu",
           "select.cu", "attn_tiles.cu", "attn_bwd.cu"]
HEADERS = [os.path.join(CSRC, h) for h in ("ptx.cuh", "msa_internal.h")] + [os.path.join(ROOT, "include", "msa.h")]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
FLAGS = ARCH + ["-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr",
                "-I" + os.path.join(ROOT, "include")]


def _nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found")


def _stale(target: str, deps) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def _build_one(lib: str, objdir: str, defines, force: bool, verbose: bool, extra_flags) -> str:
    os.makedirs(objdir, exist_ok=True)
    nvcc = _nvcc()
    objs, jobs = [], []
    for src in SOURCES:
        s = os.path.join(CSRC, src)
        o = os.path.join(objdir, src.replace(".cu", ".o"))
        objs.append(o)
        if force or _stale(o, [s] + HEADERS):
            jobs.append([nvcc, *FLAGS, *defines, *extra_flags, "-c", s, "-o", o])
    return lib, objs, jobs


def build(force: bool = False, verbose: bool = False, extra_flags=()) -> str:
    """Compile libmsa.so and its bounds-checked twin libmsa_debug.so (MSA_DEBUG=1), all
    translation units of both in parallel."""
    targets = [_build_one(LIB, BUILD, [], force, verbose, extra_flags),
               _build_one(LIB_DEBUG, BUILD + "_debug", ["-DMSA_DEBUG=1"], force, verbose, extra_flags)]
    jobs = [j for _, _, js in targets for j in js]
    if jobs:
        with cf.ThreadPoolExecutor(max_workers=len(jobs)) as ex:
            futs = [ex.submit(subprocess.run, j, capture_output=True, text=True) for j in jobs]
            for j, f in zip(jobs, futs):
                r = f.result()
                if verbose and r.stderr:
                    print(r.stderr)
                if r.returncode != 0:
                    raise RuntimeError(f"nvcc failed: {' '.join(j)}\n{r.stdout}\n{r.stderr}")
    for lib, objs, js in targets:
        if force or js or _stale(lib, objs):
            tmp = lib + f".tmp{os.getpid()}"
            r = subprocess.run([_nvcc(), *ARCH, "-shared", "-o", tmp, *objs], capture_output=True, text=True)
            if r.returncode != 0:
                raise RuntimeError(f"link failed\n{r.stdout}\n{r.stderr}")
            os.replace(tmp, lib)
    return LIB


if __name__ == "__main__":
    print(build(verbose=True))
