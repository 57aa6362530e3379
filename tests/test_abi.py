"""The C ABI without a GPU: libmsa.so builds, loads, exports every symbol that
include/msa.h declares, and host-side argument checks return before any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from block_sparse_gqa_gb300 import _build
    _build.build()
    import block_sparse_gqa_gb300 as msa
    return msa.lib()


def declared_functions():
    names = []
    for header in os.listdir(os.path.join(ROOT, "include")):
        if header.endswith(".h"):
            text = open(os.path.join(ROOT, "include", header)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(msa_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for required in ("msa_build_schedule", "msa_sparse_attn_fwd", "msa_schedule_destroy",
                     "msa_schedule_status", "msa_schedule_query", "msa_schedule_export", "msa_status_string"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_host_validation_without_gpu(lib):
    import block_sparse_gqa_gb300 as msa
    h = ctypes.c_void_p(None)
    assert lib.msa_build_schedule(None, 8, 1, 4, 1, None, ctypes.byref(h)) == 1      # null indices
    assert lib.msa_build_schedule(ctypes.c_void_p(16), 0, 1, 4, 1, None, ctypes.byref(h)) == 1
    assert lib.msa_build_schedule(ctypes.c_void_p(16), 300, 1, 4, 2, None, ctypes.byref(h)) == 1  # N > Lkv
    assert lib.msa_build_schedule(ctypes.c_void_p(16), 8, 1, 65, 1, None, ctypes.byref(h)) == 2   # topK > 64
    assert h.value is None
    t = msa.Tensor(None, 0, 1, 16, 128)
    assert lib.msa_sparse_attn_fwd(t, t, t, None, None, None, 1.0, None) == 1
    assert lib.msa_schedule_destroy(None) == 1
    assert lib.msa_schedule_query(None, None) == 1
    assert lib.msa_schedule_status(None) == 1
    assert lib.msa_status_string(6) == b"bounded device wait expired"
    assert lib.msa_version() >= 100
    opts = msa.FwdOpts()
    lib.msa_fwd_opts_init(ctypes.byref(opts))
    assert opts.path == 0 and opts.q_descale == 1.0 and opts.num_ctas == 0


def test_struct_layouts_match_header(tmp_path):
    """ctypes mirrors of the C structs agree with gcc's layout of include/msa.h."""
    import shutil
    import subprocess
    import block_sparse_gqa_gb300 as msa
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    fields = {"msa_tensor_t": (msa.Tensor, ["ptr", "dtype", "n", "h", "d"]),
              "msa_fwd_opts_t": (msa.FwdOpts, ["stream", "path", "q_descale", "k_descale", "v_descale",
                                               "stage_events", "num_ctas"]),
              "msa_schedule_info_t": (msa.ScheduleInfo, ["entries", "nsb", "ntiles", "path", "status",
                                                         "rows", "windows"])}
    lines = ['#include <stdio.h>', '#include <stddef.h>', '#include "msa.h"', "int main(void) {"]
    for st, (_, names) in fields.items():
        lines.append(f'printf("{st} %zu\\n", sizeof({st}));')
        for f in names:
            lines.append(f'printf("{st}.{f} %zu\\n", offsetof({st}, {f}));')
    lines.append("return 0; }")
    src = tmp_path / "layout.c"
    src.write_text("\n".join(lines))
    exe = tmp_path / "layout"
    cuda_inc = "/usr/local/cuda/include"
    subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc, str(src), "-o", str(exe)])
    got = dict(l.split() for l in subprocess.check_output([str(exe)], text=True).splitlines())
    for st, (cls, names) in fields.items():
        assert int(got[st]) == ctypes.sizeof(cls), st
        for f in names:
            assert int(got[f"{st}.{f}"]) == getattr(cls, f).offset, (st, f)
