"""The C ABI on the host (no GPU): the library builds, exports every symbol that
include/mt_norm.h declares, and rejects bad arguments before any CUDA call.

Only calls whose arguments fail validation are made here, with fake addresses
that are never dereferenced: validation returns before any CUDA call.
"""
import ctypes
import os
import re
import subprocess

import pytest

import row_wise_rmsnorm_gb300 as mt
from row_wise_rmsnorm_gb300 import build as mtbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "mt_norm.h")
INV, UNS = mt.MT_ERR_INVALID_ARG, mt.MT_ERR_UNSUPPORTED

# fake, distinct, 16-byte-aligned addresses: validation never dereferences them
A, B, C, E, F, G, H, K, L = (0x10000 * (i + 1) for i in range(9))
BIG = 1 << 40


@pytest.fixture(scope="module")
def lib():
    mtbuild.build()
    return mt.load()


def declared_functions():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:mt_status_t|int|const char \*)\s*(mt_\w+)\(", text,
                                 re.M)))


def test_binding_loads_the_library_the_build_writes():
    assert mt.library_path() == mtbuild.LIB


def test_header_is_plain_c():
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only", "-x", "c", HEADER],
                   check=True)


def test_exports_every_declared_symbol(lib):
    decl = declared_functions()
    assert len(decl) == 23
    assert sorted(mt.EXPORTED) == decl
    out = subprocess.run(["nm", "-D", "--defined-only", mt.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT (mt_\w+)$", out, re.M))
    assert set(decl) <= exported
    for name in decl:
        assert getattr(lib, name) is not None


def test_library_targets_sm_103a_only():
    assert "arch=compute_103a,code=sm_103a" in " ".join(mtbuild.NVCC_FLAGS)
    assert not any("fast-math" in f or "use_fast_math" in f for f in mtbuild.NVCC_FLAGS)


def test_status_strings(lib):
    for code in range(4):
        assert lib.mt_status_string(code)
    assert lib.mt_norm_version() >= 100
    assert lib.mt_last_cuda_error() == 0


@pytest.mark.parametrize("case", ["null", "n0", "d0", "nneg", "dwide", "nhuge", "eps0", "epsneg",
                                  "epsnan", "epsinf", "alias", "overlap_stats"])
def test_rmsnorm_forward_validation(lib, case):
    args = dict(X=A, g=B, Y=C, r=E, N=4, D=64, eps=1e-5)
    expect = INV
    if case == "null": args["X"] = None
    if case == "n0": args["N"], expect = 0, mt.MT_OK  # an empty batch: no-op, no CUDA call
    if case == "d0": args["D"] = 0
    if case == "nneg": args["N"] = -3
    if case == "dwide": args["D"], expect = mt.MT_MAX_COLS + 1, UNS
    if case == "nhuge": args["N"], expect = 2 ** 31, UNS
    if case == "eps0": args["eps"] = 0.0
    if case == "epsneg": args["eps"] = -1e-5
    if case == "epsnan": args["eps"] = float("nan")
    if case == "epsinf": args["eps"] = float("inf")
    if case == "alias": args["Y"] = args["X"]
    if case == "overlap_stats": args["r"] = args["X"] + 8  # rstd inside X
    st = lib.mt_rmsnorm_forward(args["X"], args["g"], args["Y"], args["r"], args["N"],
                                args["D"], args["eps"], None)
    assert st == expect


def test_backward_validation(lib):
    N, D = 8, 64
    # RMSNorm backward: NULLs, shapes, dX aliasing dY, dgamma aliasing gamma
    assert lib.mt_rmsnorm_backward(A, B, C, E, F, None, N, D, None) == INV
    assert lib.mt_rmsnorm_backward(A, B, C, E, F, G, -1, D, None) == INV
    assert lib.mt_rmsnorm_backward(None, None, None, None, None, None, 0, D, None) == INV
    assert lib.mt_rmsnorm_backward(A, B, C, E, F, G, N, mt.MT_MAX_COLS + 1, None) == UNS
    assert lib.mt_rmsnorm_backward(A, B, C, E, C, G, N, D, None) == INV
    assert lib.mt_rmsnorm_backward(A, B, C, E, F, B, N, D, None) == INV
    # _ws: NULL / misaligned / overlapping workspace
    assert lib.mt_rmsnorm_backward_ws(A, B, C, E, F, G, N, D, None, 1 << 20, None) == INV
    assert lib.mt_rmsnorm_backward_ws(A, B, C, E, F, G, N, D, H + 4, 1 << 20, None) == INV
    assert lib.mt_rmsnorm_backward_ws(A, B, C, E, F, G, N, D, A, 1 << 20, None) == INV
    # LayerNorm
    assert lib.mt_layernorm_backward(A, B, C, E, F, G, H, None, N, D, None) == INV
    assert lib.mt_layernorm_backward(A, B, C, E, F, G, H, H, N, D, None) == INV  # dgamma == dbeta
    assert lib.mt_layernorm_backward_ws(A, B, C, E, F, G, H, K, N, D, None, 0, None) == INV
    # fused op: dS is nullable, others are not; dX may not alias dS
    assert lib.mt_add_rmsnorm_backward(None, B, C, None, E, F, G, N, D, None) == INV
    assert lib.mt_add_rmsnorm_backward(A, B, C, K, E, K, G, N, D, None) == INV
    assert lib.mt_add_rmsnorm_backward_ws(A, B, C, None, E, F, G, N, D, None, 0, None) == INV


def test_forward_validation_other_ops(lib):
    N, D = 8, 64
    assert lib.mt_layernorm_forward(A, B, None, C, E, F, N, D, 1e-5, None) == INV
    assert lib.mt_layernorm_forward(A, B, C, E, F, F, N, D, 1e-5, None) == INV  # mean == rstd
    assert lib.mt_layernorm_forward(A, B, C, E, F, G, N, D, 0.0, None) == INV
    assert lib.mt_add_rmsnorm_forward(A, B, C, E, E, F, N, D, 1e-6, None) == INV  # S == Y
    assert lib.mt_add_rmsnorm_forward(A, B, C, B, E, F, N, D, 1e-6, None) == INV  # S == R
    assert lib.mt_add_rmsnorm_forward(A, B, C, E, F, G, N, 0, 1e-6, None) == INV


def test_explicit_dtype_validation(lib):
    """mt_norm_forward_ex / mt_norm_backward_ex: codes, required pointers by op, and
    overlap checks sized by the storage type."""
    N, D = 8, 64
    F16, BF16, F32 = mt.MT_DTYPE_F16, mt.MT_DTYPE_BF16, mt.MT_DTYPE_F32
    RMS, LN, ADD = mt.MT_OP_RMSNORM, mt.MT_OP_LAYERNORM, mt.MT_OP_ADD_RMSNORM
    fwd, bwd = lib.mt_norm_forward_ex, lib.mt_norm_backward_ex
    # unknown op or dtype code
    assert fwd(5, F16, F16, A, None, B, None, None, C, None, E, N, D, 1e-5, None) == INV
    assert fwd(RMS, 3, F16, A, None, B, None, None, C, None, E, N, D, 1e-5, None) == INV
    assert fwd(RMS, F16, -1, A, None, B, None, None, C, None, E, N, D, 1e-5, None) == INV
    assert bwd(RMS, F16, F16, 9, A, B, C, None, None, E, F, G, None, N, D, None, 0, None) == INV
    # required pointers depend on the op; unused ones are ignored
    assert fwd(LN, F32, F32, A, None, B, None, None, C, E, F, N, D, 1e-5, None) == INV  # beta
    assert fwd(ADD, BF16, F32, A, None, B, None, E, C, None, F, N, D, 1e-5, None) == INV  # R
    assert bwd(LN, BF16, BF16, F32, A, B, C, None, E, F, G, H, None, N, D, None, 0, None) == INV
    # an fp32 activation spans 4 bytes per element: Y placed 2*N*D bytes after X overlaps
    # X for fp32 (invalid) but not for fp16 (then only eps decides: 0 is invalid too,
    # so use a valid eps and an invalid shape to stay away from CUDA)
    half = 2 * N * D
    assert fwd(RMS, F32, F32, A, None, B, None, None, A + half, None, E, N, D, 1e-5, None) == INV
    assert fwd(RMS, F16, F16, A, None, B, None, None, A + half, None, E, N,
               mt.MT_MAX_COLS + 1, 1e-5, None) == UNS
    # dY in fp32 overlapping dX placed right after an fp16-sized dY
    assert bwd(RMS, F16, F16, F32, A, B, C, None, None, E, C + half, G, None, N, D, None, 0,
               None) == INV
    assert lib.mt_last_cuda_error() == 0  # nothing reached CUDA


def test_softmax_and_cross_entropy_validation(lib):
    N, D = 8, 64
    F16, F32 = mt.MT_DTYPE_F16, mt.MT_DTYPE_F32
    NONE, SUM, MEAN = mt.MT_REDUCTION_NONE, mt.MT_REDUCTION_SUM, mt.MT_REDUCTION_MEAN
    assert lib.mt_softmax_forward(F16, None, B, N, D, 0, None) == INV
    assert lib.mt_softmax_forward(5, A, B, N, D, 0, None) == INV
    assert lib.mt_softmax_forward(F16, A, A, N, D, 1, None) == INV          # in place
    assert lib.mt_softmax_forward(F16, A, B, N, mt.MT_MAX_SOFTMAX_COLS + 1, 0, None) == UNS
    assert lib.mt_softmax_forward(F16, None, None, 0, D, 0, None) == mt.MT_OK      # empty batch
    assert lib.mt_softmax_backward(F16, None, None, None, 0, D, 1, None) == mt.MT_OK
    assert lib.mt_softmax_forward(F16, A, B, -1, D, 0, None) == INV
    assert lib.mt_softmax_backward(F32, A, None, C, N, D, 0, None) == INV
    assert lib.mt_softmax_backward(F32, A, B, B, N, D, 0, None) == INV      # dX aliases dY
    ce_f, ce_b = lib.mt_cross_entropy_forward, lib.mt_cross_entropy_backward
    assert ce_f(F16, A, B, N, D, -100, 0.0, 0.0, SUM, C, E, None, G, None) == INV  # loss_out
    assert ce_f(F16, A, B, N, D, -100, 1.5, 0.0, NONE, C, E, None, None, None) == INV
    assert ce_f(F16, A, B, N, D, -100, 0.0, -1.0, NONE, C, E, None, None, None) == INV
    assert ce_f(F16, A, B, N, D, -100, 0.0, float("nan"), NONE, C, E, None, None, None) == INV
    assert ce_f(F16, A, B, N, D, -100, 0.0, 0.0, 3, C, E, F, G, None) == INV         # reduction
    assert ce_f(F16, A, B, N, mt.MT_MAX_CE_COLS + 1, -100, 0.0, 0.0, NONE, C, E, None, None,
                None) == UNS
    assert ce_f(F16, A, B, N, D, -100, 0.0, 0.0, NONE, C, C, None, None, None) == INV  # lse==rows
    assert ce_b(F16, A, B, C, N, D, -100, 0.0, 0.0, MEAN, E, None, G, None) == INV    # n_valid
    assert ce_b(F16, A, B, C, N, D, -100, 0.0, 0.0, NONE, E, None, A, None) == INV    # dX == X
    # empty batch: NONE and the backward are no-ops (no CUDA call); SUM/MEAN still need
    # their two distinct scalar outputs
    assert ce_f(F16, None, None, 0, D, -100, 0.0, 0.0, NONE, None, None, None, None, None) == 0
    assert ce_b(F16, None, None, None, 0, D, -100, 0.0, 0.0, MEAN, None, None, None, None) == 0
    assert ce_f(F16, None, None, 0, D, -100, 0.0, 0.0, SUM, None, None, None, G, None) == INV
    assert ce_f(F16, None, None, 0, D, -100, 0.0, 0.0, SUM, None, None, G, G, None) == INV
    assert lib.mt_last_cuda_error() == 0  # nothing reached CUDA


def test_norm_gemv_validation(lib):
    """mt_fused_rmsnorm_gemv / mt_fused_layernorm_gemv: argument errors before any CUDA
    call; M = 0 and N = 0 are no-ops."""
    f_rms, f_ln = lib.mt_fused_rmsnorm_gemv, lib.mt_fused_layernorm_gemv
    M, N, K = 4, 64, 128
    assert f_rms(None, B, C, E, M, N, K, 1e-5, None) == INV
    assert f_ln(A, B, None, C, E, M, N, K, 1e-5, None) == INV        # beta
    assert f_rms(A, B, C, E, -1, N, K, 1e-5, None) == INV
    assert f_rms(A, B, C, E, M, N, 0, 1e-5, None) == INV
    assert f_rms(A, B, C, E, M, N, K, 0.0, None) == INV
    assert f_rms(A, B, C, E, mt.MT_MAX_GEMV_ROWS + 1, N, K, 1e-5, None) == UNS
    assert f_rms(A, B, C, E, M, N, mt.MT_MAX_GEMV_K + 1, 1e-5, None) == UNS
    assert f_rms(A, B, C, C + 8, M, N, K, 1e-5, None) == INV          # Y inside W
    assert f_rms(None, None, None, None, 0, N, K, 1e-5, None) == mt.MT_OK
    assert f_ln(None, None, None, None, None, M, 0, K, 1e-5, None) == mt.MT_OK
    assert lib.mt_last_cuda_error() == 0  # nothing reached CUDA


def test_workspace_size_validation(lib):
    out = ctypes.c_size_t(0)
    assert lib.mt_norm_backward_workspace_size(0, 8, 64, 0, None) == INV
    assert lib.mt_norm_backward_workspace_size(7, 8, 64, 0, ctypes.byref(out)) == INV
    assert lib.mt_norm_backward_workspace_size(0, -1, 64, 0, ctypes.byref(out)) == INV
    assert lib.mt_norm_backward_workspace_size(1, 8, mt.MT_MAX_COLS + 1, 0, ctypes.byref(out)) == UNS
    out.value = 7
    assert lib.mt_norm_backward_workspace_size(0, 0, 64, 0, ctypes.byref(out)) == mt.MT_OK
    assert out.value == 0  # an empty batch needs no workspace
    assert lib.mt_norm_backward_workspace_size(2, 8, 64, -1, ctypes.byref(out)) == INV
    assert lib.mt_last_cuda_error() == 0  # nothing reached CUDA


def test_product_path_does_not_import_oracle():
    """The binding and the kernels never reach the oracle (test infrastructure)."""
    pkg = os.path.join(ROOT, "row_wise_rmsnorm_gb300")
    for dirpath, _, files in os.walk(pkg):
        if "_build" in dirpath:
            continue
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in text.lower(), f"{f} mentions the oracle"
