"""fp64 CPU oracle for row-wise normalization, row softmax and per-row cross-entropy --
TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline leg
(``cpu_baseline`` and ``--impl reference``) may import this package. The CUDA
library and its Python binding never import it, and it imports nothing from
them: the two share no code.

The arithmetic lives in ``norm_oracle.c`` (plain single-threaded C, fp64, built
with ``-ffp-contract=off``); this module only compiles it with gcc, widens the
fp16 inputs to fp64 (exact) and marshals numpy arrays through ctypes. Every
output is fp64 and unrounded.

Sources for the formulas (page title, section):
  * meTile, "Kernel coverage and training scope", "Exact native normalization
    contract" -- RMSNorm, LayerNorm (centred population variance), fused
    residual-add + RMSNorm (unrounded sum normalised; residual-output cotangent
    added to both input gradients), backward at the saved statistics.
  * tensorcore, "Training kernels", "RMSnorm -- Llama-style" (Math) and
    "LayerNorm -- standard"; "Softmax -- standalone, row-wise".
  * meTile reduction and loss checklists: softmax / log-softmax with input
    gradients; cross-entropy with ignore-index, none/sum/mean, label smoothing,
    z-loss. "Metal subgroup LayerNorm and cross-entropy report", "Structural
    repair exercised by cross-entropy": the per-row loss formula.
  * tensorcore, "Training kernels", "Fused Norm + GEMV": Y = Norm(X) @ W with the
    normalized rows kept unrounded.

Parity pins: tests/test_oracle_pins.py pins every function here against finite
differences, closed forms, invariants, the worked LayerNorm example of the
meTile contract and torch's fp64 CPU layer_norm / rms_norm with autograd.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "norm_oracle.c")
BUILD_DIR = os.path.join(_HERE, "_build")
LIB_PATH = os.path.join(BUILD_DIR, "liboracle.so")
CFLAGS = ["-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def compile_oracle(source: str = SOURCE, out: str = LIB_PATH) -> str:
    """Compile the C oracle with gcc; return the path of the shared object."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, "-o", tmp, source, "-lm"], check=True)
    os.replace(tmp, out)
    return out


def _declare(lib):
    lib.oracle_rmsnorm_forward.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, ctypes.c_double]
    lib.oracle_rmsnorm_backward.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _dp, _i64, _i64]
    lib.oracle_layernorm_forward.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64, _i64, ctypes.c_double]
    lib.oracle_layernorm_backward.argtypes = [_dp] * 10 + [_i64, _i64]
    lib.oracle_add_rmsnorm_forward.argtypes = [_dp] * 6 + [_i64, _i64, ctypes.c_double]
    lib.oracle_add_rmsnorm_backward.argtypes = [_dp] * 8 + [_i64, _i64]
    _lp = ctypes.POINTER(ctypes.c_int64)
    lib.oracle_softmax_forward.argtypes = [_dp, _dp, _i64, _i64, ctypes.c_int]
    lib.oracle_softmax_backward.argtypes = [_dp, _dp, _dp, _i64, _i64, ctypes.c_int]
    lib.oracle_cross_entropy_forward.argtypes = [_dp, _lp, _i64, _i64, _i64, ctypes.c_double,
                                                 ctypes.c_double, _dp, _dp]
    lib.oracle_cross_entropy_backward.argtypes = [_dp, _lp, _dp, _dp, _i64, _i64, _i64,
                                                  ctypes.c_double, ctypes.c_double, _dp]
    lib.oracle_norm_gemv.argtypes = [ctypes.c_int] + [_dp] * 7 + [_i64, _i64, _i64,
                                                                   ctypes.c_double]
    for name in ("oracle_norm_gemv", "oracle_rmsnorm_forward", "oracle_rmsnorm_backward",
                 "oracle_layernorm_forward", "oracle_layernorm_backward",
                 "oracle_add_rmsnorm_forward", "oracle_add_rmsnorm_backward",
                 "oracle_softmax_forward", "oracle_softmax_backward",
                 "oracle_cross_entropy_forward", "oracle_cross_entropy_backward"):
        getattr(lib, name).restype = None
    return lib


def load_library(path: str | None = None):
    """Load a compiled oracle. With no path: the default build, compiled on first use."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            stale = (not os.path.exists(LIB_PATH)
                     or os.path.getmtime(LIB_PATH) < os.path.getmtime(SOURCE))
            if stale:
                compile_oracle()
            _lib = _declare(ctypes.CDLL(LIB_PATH))
    return _lib


def _f64(a) -> np.ndarray:
    """Widen to a C-contiguous fp64 array (exact for fp16 and fp32 inputs)."""
    if hasattr(a, "detach"):  # a torch CPU tensor
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _p(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _shape(X) -> tuple[int, int]:
    if X.ndim != 2:
        raise ValueError("expected a 2-D [N, D] array")
    return int(X.shape[0]), int(X.shape[1])


def rmsnorm_forward(X, gamma, eps, lib=None):
    """RMSNorm forward -> (Y [N,D], rstd [N]), fp64."""
    lib = lib or load_library()
    X, gamma = _f64(X), _f64(gamma)
    N, D = _shape(X)
    Y = np.empty((N, D)); rstd = np.empty(N)
    lib.oracle_rmsnorm_forward(_p(X), _p(gamma), _p(Y), _p(rstd), N, D, float(eps))
    return Y, rstd


def rmsnorm_backward(X, gamma, dY, rstd, lib=None):
    """RMSNorm backward -> (dX [N,D], dgamma [D], dgamma_abs [D]), fp64."""
    lib = lib or load_library()
    X, gamma, dY, rstd = _f64(X), _f64(gamma), _f64(dY), _f64(rstd)
    N, D = _shape(X)
    dX = np.empty((N, D)); dg = np.empty(D); dga = np.empty(D)
    lib.oracle_rmsnorm_backward(_p(X), _p(gamma), _p(dY), _p(rstd), _p(dX), _p(dg), _p(dga), N, D)
    return dX, dg, dga


def layernorm_forward(X, gamma, beta, eps, lib=None):
    """LayerNorm forward -> (Y [N,D], mean [N], rstd [N]), fp64."""
    lib = lib or load_library()
    X, gamma, beta = _f64(X), _f64(gamma), _f64(beta)
    N, D = _shape(X)
    Y = np.empty((N, D)); mean = np.empty(N); rstd = np.empty(N)
    lib.oracle_layernorm_forward(_p(X), _p(gamma), _p(beta), _p(Y), _p(mean), _p(rstd),
                                 N, D, float(eps))
    return Y, mean, rstd


def layernorm_backward(X, gamma, dY, mean, rstd, lib=None):
    """LayerNorm backward -> (dX, dgamma, dbeta, dgamma_abs, dbeta_abs), fp64."""
    lib = lib or load_library()
    X, gamma, dY, mean, rstd = _f64(X), _f64(gamma), _f64(dY), _f64(mean), _f64(rstd)
    N, D = _shape(X)
    dX = np.empty((N, D)); dg = np.empty(D); db = np.empty(D)
    dga = np.empty(D); dba = np.empty(D)
    lib.oracle_layernorm_backward(_p(X), _p(gamma), _p(dY), _p(mean), _p(rstd), _p(dX),
                                  _p(dg), _p(db), _p(dga), _p(dba), N, D)
    return dX, dg, db, dga, dba


def add_rmsnorm_forward(X, R, gamma, eps, lib=None):
    """Fused residual-add + RMSNorm forward -> (Y [N,D], S_exact [N,D], rstd [N]), fp64.

    S_exact is the exact sum X + R; the stored residual output is its
    round-to-nearest-even fp16 value, which the caller forms.
    """
    lib = lib or load_library()
    X, R, gamma = _f64(X), _f64(R), _f64(gamma)
    N, D = _shape(X)
    if R.shape != X.shape:
        raise ValueError("R must match X")
    Y = np.empty((N, D)); S = np.empty((N, D)); rstd = np.empty(N)
    lib.oracle_add_rmsnorm_forward(_p(X), _p(R), _p(gamma), _p(S), _p(Y), _p(rstd),
                                   N, D, float(eps))
    return Y, S, rstd


def add_rmsnorm_backward(S, gamma, dY, dS, rstd, lib=None):
    """Fused residual-add + RMSNorm backward -> (dX [N,D], dgamma [D], dgamma_abs [D]).

    dX is both d(source) and d(residual). dS may be None (treated as zero).
    """
    lib = lib or load_library()
    S, gamma, dY, rstd = _f64(S), _f64(gamma), _f64(dY), _f64(rstd)
    N, D = _shape(S)
    dS_arr = None if dS is None else _f64(dS)
    dX = np.empty((N, D)); dg = np.empty(D); dga = np.empty(D)
    lib.oracle_add_rmsnorm_backward(_p(S), _p(gamma), _p(dY),
                                    None if dS_arr is None else _p(dS_arr),
                                    _p(rstd), _p(dX), _p(dg), _p(dga), N, D)
    return dX, dg, dga


# ------------------------------------------------ row softmax, cross-entropy ---

def softmax_forward(X, log_softmax=False, lib=None):
    """Row softmax (or log-softmax) of X [N, D] -> Y fp64. tensorcore "Training kernels",
    "Softmax -- standalone, row-wise"; meTile softmax / log-softmax."""
    lib = lib or load_library()
    X = _f64(X)
    N, D = _shape(X)
    Y = np.empty((N, D))
    lib.oracle_softmax_forward(_p(X), _p(Y), N, D, int(bool(log_softmax)))
    return Y


def softmax_backward(Y, dY, log_softmax=False, lib=None):
    """Input gradient of the row softmax (log-softmax) from its output Y and dY."""
    lib = lib or load_library()
    Y, dY = _f64(Y), _f64(dY)
    N, D = _shape(Y)
    dX = np.empty((N, D))
    lib.oracle_softmax_backward(_p(Y), _p(dY), _p(dX), N, D, int(bool(log_softmax)))
    return dX


def _targets(T) -> np.ndarray:
    if hasattr(T, "detach"):
        T = T.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(T, dtype=np.int64))


def cross_entropy_forward(X, T, ignore_index=-100, label_smoothing=0.0, z_loss=0.0, lib=None):
    """Per-row cross-entropy of logits X [N, D] with integer targets T [N] (meTile losses;
    LuisaCompute report formula) -> (loss [N], lse [N]) fp64; ignored rows have loss 0."""
    lib = lib or load_library()
    X = _f64(X)
    N, D = _shape(X)
    T = _targets(T)
    loss, lse = np.empty(N), np.empty(N)
    lib.oracle_cross_entropy_forward(_p(X), T.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                     N, D, int(ignore_index), float(label_smoothing),
                                     float(z_loss), _p(loss), _p(lse))
    return loss, lse


def cross_entropy_reduce(loss, T, ignore_index, reduction):
    """The plain reductions: "none" -> loss [N]; "sum" -> sum; "mean" -> sum / number of
    rows whose target is not ignore_index (0 if there is none). Returns (value, n_valid)."""
    n_valid = float(np.sum(_targets(T) != ignore_index))
    if reduction == "none":
        return np.asarray(loss, dtype=np.float64), n_valid
    total = float(np.sum(loss))
    if reduction == "sum":
        return total, n_valid
    return (total / n_valid if n_valid > 0 else 0.0), n_valid


def cross_entropy_row_grad(dloss, N, n_valid, reduction):
    """Upstream gradient per row g_i: none -> dloss_i; sum -> dloss; mean -> dloss / n_valid
    (0 if no row is valid)."""
    if reduction == "none":
        return _f64(dloss).reshape(N)
    d = float(np.asarray(dloss, dtype=np.float64).reshape(-1)[0])
    if reduction == "sum":
        return np.full(N, d)
    return np.full(N, d / n_valid if n_valid > 0 else 0.0)


def cross_entropy_backward(X, T, lse, g, ignore_index=-100, label_smoothing=0.0, z_loss=0.0,
                           lib=None):
    """Gradient of sum_i g_i * loss_i with respect to the logits, at the saved lse."""
    lib = lib or load_library()
    X, lse, g = _f64(X), _f64(lse), _f64(g)
    N, D = _shape(X)
    T = _targets(T)
    dX = np.empty((N, D))
    lib.oracle_cross_entropy_backward(_p(X), T.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                                      _p(lse), _p(g), N, D, int(ignore_index),
                                      float(label_smoothing), float(z_loss), _p(dX))
    return dX


def norm_gemv(op, X, gamma, beta, W, eps, lib=None):
    """Fused normalization + GEMV (tensorcore "Fused Norm + GEMV"): Y = Norm(X) @ W with the
    normalized rows unrounded. op "rmsnorm" or "layernorm" (beta ignored for RMSNorm);
    X [M, K], W [K, N]. -> (Y [M, N], Y_abs [M, N] = sum_k |xn_mk W_kn|), fp64."""
    lib = lib or load_library()
    code = {"rmsnorm": 0, "layernorm": 1}[op]
    X, gamma, W = _f64(X), _f64(gamma), _f64(W)
    beta = _f64(beta) if beta is not None else np.zeros_like(gamma)
    M, K = _shape(X)
    if W.ndim != 2 or W.shape[0] != K:
        raise ValueError("W must be [K, N]")
    N = int(W.shape[1])
    Y, Ya, xn = np.empty((M, N)), np.empty((M, N)), np.empty(K)
    lib.oracle_norm_gemv(code, _p(X), _p(gamma), _p(beta), _p(W), _p(Y), _p(Ya), _p(xn), M, N,
                         K, float(eps))
    return Y, Ya


BF16_MAX = (2.0 - 2.0 ** -7) * 2.0 ** 127  # largest finite bfloat16


def round_fp16(a) -> np.ndarray:
    """Round fp64 values to IEEE binary16, round-to-nearest-even (numpy's conversion)."""
    return np.asarray(a, dtype=np.float64).astype(np.float16)


def round_bf16(a) -> np.ndarray:
    """Round fp64 values to bfloat16 (7 fraction bits, the fp32 exponent range), round to
    nearest even, returned as fp64.

    Direct rounding from fp64 (not through fp32, which would round twice): with
    e = max(floor(log2|x|), -126) the bf16 grid step near x is 2^(e-7); |x| / step is
    exact (a power-of-two scaling), numpy's rint rounds it to the nearest integer with
    ties to even, and the product with the step is exact. Past the largest finite bf16
    the result is infinity; NaN stays NaN.
    """
    x = np.asarray(a, dtype=np.float64)
    ax = np.abs(x)
    with np.errstate(invalid="ignore"):
        _, E = np.frexp(ax)
        step = np.ldexp(1.0, np.maximum(E - 1, -126) - 7)
        r = np.rint(ax / step) * step
    r = np.where(r > BF16_MAX, np.inf, r)
    return np.copysign(r, x)


def round_f32(a) -> np.ndarray:
    """Round fp64 values to IEEE binary32, round-to-nearest-even, returned as fp64."""
    return np.asarray(a, dtype=np.float64).astype(np.float32).astype(np.float64)


def round_storage(a, dtype: str) -> np.ndarray:
    """Round to a storage type named "f16", "bf16" or "f32" (returned as fp64)."""
    if dtype == "f16":
        return round_fp16(a).astype(np.float64)
    if dtype == "bf16":
        return round_bf16(a)
    if dtype == "f32":
        return round_f32(a)
    raise ValueError(dtype)
