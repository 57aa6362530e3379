"""The bounds-checked build (libmsa_debug.so, compiled with MSA_DEBUG=1) on the tiny
workload: every device-side gather index and TMA coordinate is checked, so a clean run
reports no status bit, and its outputs match the oracle like the release build's.

The library is selected per process (MSA_LIBRARY=debug), so the check runs in a child
interpreter.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import numpy as np, torch
import block_sparse_gqa_gb300 as msa, oracle, workloads
from tests.util import BF16_MAX_ABS, BF16_REL_L2, LSE_MAX_ABS, compare_outputs
assert msa.lib().msa_debug_build() == 1, "the bounds-checked library was not loaded"
wl = workloads.make_workload("tiny")
cfg = wl.cfg
dev = torch.device("cuda")
Q, K, V = (t.to(dev) for t in (wl.Q, wl.K, wl.V))
s = msa.build_schedule(wl.indices.to(dev), cfg.nblocks)
Qn, Kn, Vn = wl.np_inputs()
Or, Lr, _ = oracle.attn_fwd(Qn, Kn, Vn, wl.indices.numpy(), Lkv=cfg.Lkv, scale=cfg.scale)
for path in ("auto", "kv_outer", "q_outer"):
    O, LSE = msa.sparse_attn_fwd(Q, K, V, s, scale=cfg.scale, path=path)
    torch.cuda.synchronize()
    assert s.status() == 0, (path, s.query())
    rel, mabs, lerr = compare_outputs(O.float().cpu().numpy(), LSE.cpu().numpy(), Or, Lr)
    assert rel <= BF16_REL_L2 and mabs <= BF16_MAX_ABS and lerr <= LSE_MAX_ABS, (path, rel, mabs, lerr)
gen = torch.Generator().manual_seed(3)
dO = torch.randn((cfg.N, cfg.Hq, cfg.D), generator=gen).to(torch.bfloat16).to(dev)
msa.sparse_attn_bwd(Q, K, V, O, dO, LSE, s, scale=cfg.scale)
torch.cuda.synchronize()
assert s.status() == 0, s.query()
s.close()
print("debug build clean")
"""


def test_bounds_checked_build_runs_tiny_clean():
    env = dict(os.environ, MSA_LIBRARY="debug", PYTHONPATH=ROOT + os.pathsep + os.environ.get("PYTHONPATH", ""))
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "debug build clean" in r.stdout
