"""The Python binding's constants and enum values are the C header's: a small C program
that includes include/mt_norm.h prints every bound and enumerator, and each must equal
the binding's copy (a binding that drifted from the header would pass the wrong bounds
and codes to callers)."""
import os
import shutil
import subprocess

import pytest

import row_wise_rmsnorm_gb300 as mt

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
NAMES = ["MT_OK", "MT_ERR_INVALID_ARG", "MT_ERR_UNSUPPORTED", "MT_ERR_CUDA",
         "MT_OP_RMSNORM", "MT_OP_LAYERNORM", "MT_OP_ADD_RMSNORM",
         "MT_DTYPE_F16", "MT_DTYPE_BF16", "MT_DTYPE_F32",
         "MT_REDUCTION_NONE", "MT_REDUCTION_SUM", "MT_REDUCTION_MEAN",
         "MT_MAX_COLS", "MT_MAX_SOFTMAX_COLS", "MT_MAX_CE_COLS",
         "MT_MAX_GEMV_ROWS", "MT_MAX_GEMV_K", "MT_NOALLOC_SCRATCH_BYTES", "MT_WAIT_ERR_CLUSTER"]


def test_header_constants_match_binding(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "consts.c"
    body = "\n".join(f'    printf("{n} %llu\\n", (unsigned long long)({n}));' for n in NAMES)
    src.write_text('#include <stdio.h>\n#include "mt_norm.h"\nint main(void) {\n' + body +
                   "\n    return 0;\n}\n")
    exe = tmp_path / "consts"
    subprocess.run([cc, "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)],
                   check=True, capture_output=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout
    got = {k: int(v) for k, v in (line.split() for line in out.splitlines())}
    assert set(got) == set(NAMES)
    for n in NAMES:
        assert getattr(mt, n, None) is not None or hasattr(mt._binding, n), n
        val = getattr(mt, n) if hasattr(mt, n) else getattr(mt._binding, n)
        assert got[n] == val, f"{n}: header {got[n]}, binding {val}"
