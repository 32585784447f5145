"""ctypes binding of libmt_norm.so (the C ABI in include/mt_norm.h).

Two layers, both argument marshalling only -- every step of the computation runs in
the CUDA kernels behind the C ABI:

* ``mt_*`` functions with the C names and the C argument order. Tensor arguments may
  be torch tensors (their ``data_ptr()`` is passed) or raw integer addresses; the
  stream may be a ``torch.cuda.Stream``, a raw ``cudaStream_t`` integer, or None for
  torch's current stream. A non-zero status raises ``MtNormError``.
* ``rmsnorm_forward`` & co.: allocate outputs (and the backward workspace) with
  torch on the input's device and call the ``mt_*`` function on the current stream.

There is no fallback: if the library has not been built, or is loaded without a
CUDA device, the calls fail loudly.
"""
from __future__ import annotations

import ctypes
import os


# the library build.py writes (build.LIB; not imported here, so that
# `python -m row_wise_rmsnorm_gb300.build` runs a module nothing has imported yet)
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libmt_norm.so")

MT_OK, MT_ERR_INVALID_ARG, MT_ERR_UNSUPPORTED, MT_ERR_CUDA = 0, 1, 2, 3
MT_OP_RMSNORM, MT_OP_LAYERNORM, MT_OP_ADD_RMSNORM = 0, 1, 2
MT_DTYPE_F16, MT_DTYPE_BF16, MT_DTYPE_F32 = 0, 1, 2
MT_REDUCTION_NONE, MT_REDUCTION_SUM, MT_REDUCTION_MEAN = 0, 1, 2
MT_MAX_CE_COLS = 262144
MT_MAX_COLS = 131072
MT_MAX_SOFTMAX_COLS = 262144
MT_MAX_GEMV_ROWS = 8
MT_MAX_GEMV_K = 32768

# Every exported symbol of include/mt_norm.h.
EXPORTED = (
    "mt_rmsnorm_forward", "mt_rmsnorm_backward", "mt_rmsnorm_backward_ws",
    "mt_layernorm_forward", "mt_layernorm_backward", "mt_layernorm_backward_ws",
    "mt_add_rmsnorm_forward", "mt_add_rmsnorm_backward", "mt_add_rmsnorm_backward_ws",
    "mt_norm_forward_ex", "mt_norm_backward_ex",
    "mt_softmax_forward", "mt_softmax_backward",
    "mt_cross_entropy_forward", "mt_cross_entropy_backward",
    "mt_fused_rmsnorm_gemv", "mt_fused_layernorm_gemv",
    "mt_rmsnorm_backward_noalloc",
    "mt_norm_backward_workspace_size", "mt_last_cuda_error", "mt_status_string",
    "mt_norm_version", "mt_device_wait_errors",
)
MT_WAIT_ERR_CLUSTER = 1
MT_NOALLOC_SCRATCH_BYTES = 16 << 20


class MtNormError(RuntimeError):
    def __init__(self, status: int, func: str, lib):
        self.status = status
        msg = lib.mt_status_string(status).decode()
        if status == MT_ERR_CUDA:
            msg += f" (cudaError {lib.mt_last_cuda_error()})"
        super().__init__(f"{func}: {msg}")


_lib = None

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_F = ctypes.c_float
_SZ = ctypes.c_size_t
_SIGS = {
    "mt_rmsnorm_forward": [_P, _P, _P, _P, _I64, _I64, _F, _P],
    "mt_rmsnorm_backward": [_P, _P, _P, _P, _P, _P, _I64, _I64, _P],
    "mt_rmsnorm_backward_ws": [_P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, _P],
    "mt_layernorm_forward": [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P],
    "mt_layernorm_backward": [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P],
    "mt_layernorm_backward_ws": [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, _P],
    "mt_add_rmsnorm_forward": [_P, _P, _P, _P, _P, _P, _I64, _I64, _F, _P],
    "mt_add_rmsnorm_backward": [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P],
    "mt_add_rmsnorm_backward_ws": [_P, _P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, _P],
    "mt_norm_forward_ex": [ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P, _P, _P, _P, _P,
                           _P, _I64, _I64, _F, _P],
    "mt_norm_backward_ex": [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int, _P, _P, _P,
                            _P, _P, _P, _P, _P, _P, _I64, _I64, _P, _SZ, _P],
    "mt_softmax_forward": [ctypes.c_int, _P, _P, _I64, _I64, ctypes.c_int, _P],
    "mt_softmax_backward": [ctypes.c_int, _P, _P, _P, _I64, _I64, ctypes.c_int, _P],
    "mt_cross_entropy_forward": [ctypes.c_int, _P, _P, _I64, _I64, _I64, _F, _F, ctypes.c_int,
                                 _P, _P, _P, _P, _P],
    "mt_fused_rmsnorm_gemv": [_P, _P, _P, _P, _I64, _I64, _I64, _F, _P],
    "mt_fused_layernorm_gemv": [_P, _P, _P, _P, _P, _I64, _I64, _I64, _F, _P],
    "mt_cross_entropy_backward": [ctypes.c_int, _P, _P, _P, _I64, _I64, _I64, _F, _F,
                                  ctypes.c_int, _P, _P, _P, _P],
    "mt_rmsnorm_backward_noalloc": [_P, _P, _P, _P, _P, _P, _I64, _I64, _P],
    "mt_norm_backward_workspace_size": [ctypes.c_int, _I64, _I64, ctypes.c_int,
                                        ctypes.POINTER(_SZ)],
    "mt_last_cuda_error": [],
    "mt_device_wait_errors": [ctypes.c_int, ctypes.POINTER(ctypes.c_uint), ctypes.c_int],
    "mt_status_string": [ctypes.c_int],
    "mt_norm_version": [],
}


def library_path() -> str:
    return LIB_PATH


def load():
    """Load libmt_norm.so (built by ``row_wise_rmsnorm_gb300.build``); raise if absent."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"CUDA library not built: {LIB_PATH} is missing. Build it with "
                "`python -m row_wise_rmsnorm_gb300.build` (needs nvcc); there is no "
                "CPU fallback.")
        lib = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            fn = getattr(lib, name)
            fn.argtypes = args
            fn.restype = ctypes.c_int
        lib.mt_status_string.restype = ctypes.c_char_p
        _lib = lib
    return _lib


def _ptr(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(s):
    if s is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(s, int):
        return s
    return s.cuda_stream


def _check(status: int, func: str):
    if status != MT_OK:
        raise MtNormError(status, func, load())


# ------------------------------------------------------------ C-named calls ---

def mt_rmsnorm_forward(X, gamma, Y, rstd, N, D, eps, stream=None):
    _check(load().mt_rmsnorm_forward(_ptr(X), _ptr(gamma), _ptr(Y), _ptr(rstd), N, D, eps,
                                     _stream(stream)), "mt_rmsnorm_forward")


def mt_rmsnorm_backward(X, gamma, dY, rstd, dX, dgamma, N, D, stream=None):
    _check(load().mt_rmsnorm_backward(_ptr(X), _ptr(gamma), _ptr(dY), _ptr(rstd), _ptr(dX),
                                      _ptr(dgamma), N, D, _stream(stream)), "mt_rmsnorm_backward")


def mt_rmsnorm_backward_ws(X, gamma, dY, rstd, dX, dgamma, N, D, workspace, workspace_bytes,
                           stream=None):
    _check(load().mt_rmsnorm_backward_ws(_ptr(X), _ptr(gamma), _ptr(dY), _ptr(rstd), _ptr(dX),
                                         _ptr(dgamma), N, D, _ptr(workspace), workspace_bytes,
                                         _stream(stream)), "mt_rmsnorm_backward_ws")


def mt_layernorm_forward(X, gamma, beta, Y, mean, rstd, N, D, eps, stream=None):
    _check(load().mt_layernorm_forward(_ptr(X), _ptr(gamma), _ptr(beta), _ptr(Y), _ptr(mean),
                                       _ptr(rstd), N, D, eps, _stream(stream)),
           "mt_layernorm_forward")


def mt_layernorm_backward(X, gamma, dY, mean, rstd, dX, dgamma, dbeta, N, D, stream=None):
    _check(load().mt_layernorm_backward(_ptr(X), _ptr(gamma), _ptr(dY), _ptr(mean), _ptr(rstd),
                                        _ptr(dX), _ptr(dgamma), _ptr(dbeta), N, D,
                                        _stream(stream)), "mt_layernorm_backward")


def mt_layernorm_backward_ws(X, gamma, dY, mean, rstd, dX, dgamma, dbeta, N, D, workspace,
                             workspace_bytes, stream=None):
    _check(load().mt_layernorm_backward_ws(_ptr(X), _ptr(gamma), _ptr(dY), _ptr(mean),
                                           _ptr(rstd), _ptr(dX), _ptr(dgamma), _ptr(dbeta), N, D,
                                           _ptr(workspace), workspace_bytes, _stream(stream)),
           "mt_layernorm_backward_ws")


def mt_add_rmsnorm_forward(X, R, gamma, S, Y, rstd, N, D, eps, stream=None):
    _check(load().mt_add_rmsnorm_forward(_ptr(X), _ptr(R), _ptr(gamma), _ptr(S), _ptr(Y),
                                         _ptr(rstd), N, D, eps, _stream(stream)),
           "mt_add_rmsnorm_forward")


def mt_add_rmsnorm_backward(S, gamma, dY, dS, rstd, dX, dgamma, N, D, stream=None):
    _check(load().mt_add_rmsnorm_backward(_ptr(S), _ptr(gamma), _ptr(dY), _ptr(dS), _ptr(rstd),
                                          _ptr(dX), _ptr(dgamma), N, D, _stream(stream)),
           "mt_add_rmsnorm_backward")


def mt_add_rmsnorm_backward_ws(S, gamma, dY, dS, rstd, dX, dgamma, N, D, workspace,
                               workspace_bytes, stream=None):
    _check(load().mt_add_rmsnorm_backward_ws(_ptr(S), _ptr(gamma), _ptr(dY), _ptr(dS),
                                             _ptr(rstd), _ptr(dX), _ptr(dgamma), N, D,
                                             _ptr(workspace), workspace_bytes, _stream(stream)),
           "mt_add_rmsnorm_backward_ws")


def mt_norm_forward_ex(op, x_dtype, w_dtype, X, R, gamma, beta, S, Y, mean, rstd, N, D, eps,
                       stream=None):
    _check(load().mt_norm_forward_ex(op, x_dtype, w_dtype, _ptr(X), _ptr(R), _ptr(gamma),
                                     _ptr(beta), _ptr(S), _ptr(Y), _ptr(mean), _ptr(rstd), N, D,
                                     eps, _stream(stream)), "mt_norm_forward_ex")


def mt_norm_backward_ex(op, x_dtype, w_dtype, g_dtype, X, gamma, dY, dS, mean, rstd, dX, dgamma,
                        dbeta, N, D, workspace=None, workspace_bytes=0, stream=None):
    _check(load().mt_norm_backward_ex(op, x_dtype, w_dtype, g_dtype, _ptr(X), _ptr(gamma),
                                      _ptr(dY), _ptr(dS), _ptr(mean), _ptr(rstd), _ptr(dX),
                                      _ptr(dgamma), _ptr(dbeta), N, D, _ptr(workspace),
                                      workspace_bytes, _stream(stream)), "mt_norm_backward_ex")


def mt_softmax_forward(dtype, X, Y, N, D, log_softmax=0, stream=None):
    _check(load().mt_softmax_forward(dtype, _ptr(X), _ptr(Y), N, D, int(log_softmax),
                                     _stream(stream)), "mt_softmax_forward")


def mt_softmax_backward(dtype, Y, dY, dX, N, D, log_softmax=0, stream=None):
    _check(load().mt_softmax_backward(dtype, _ptr(Y), _ptr(dY), _ptr(dX), N, D, int(log_softmax),
                                      _stream(stream)), "mt_softmax_backward")


def mt_cross_entropy_forward(dtype, logits, targets, N, D, ignore_index, label_smoothing, z_loss,
                             reduction, loss_rows, lse, loss_out, n_valid, stream=None):
    _check(load().mt_cross_entropy_forward(dtype, _ptr(logits), _ptr(targets), N, D, ignore_index,
                                           label_smoothing, z_loss, reduction, _ptr(loss_rows),
                                           _ptr(lse), _ptr(loss_out), _ptr(n_valid),
                                           _stream(stream)), "mt_cross_entropy_forward")


def mt_cross_entropy_backward(dtype, logits, targets, lse, N, D, ignore_index, label_smoothing,
                              z_loss, reduction, dloss, n_valid, dlogits, stream=None):
    _check(load().mt_cross_entropy_backward(dtype, _ptr(logits), _ptr(targets), _ptr(lse), N, D,
                                            ignore_index, label_smoothing, z_loss, reduction,
                                            _ptr(dloss), _ptr(n_valid), _ptr(dlogits),
                                            _stream(stream)), "mt_cross_entropy_backward")


def mt_fused_rmsnorm_gemv(X, gamma, W, Y, M, N, K, eps, stream=None):
    _check(load().mt_fused_rmsnorm_gemv(_ptr(X), _ptr(gamma), _ptr(W), _ptr(Y), M, N, K, eps,
                                        _stream(stream)), "mt_fused_rmsnorm_gemv")


def mt_fused_layernorm_gemv(X, gamma, beta, W, Y, M, N, K, eps, stream=None):
    _check(load().mt_fused_layernorm_gemv(_ptr(X), _ptr(gamma), _ptr(beta), _ptr(W), _ptr(Y), M, N,
                                          K, eps, _stream(stream)), "mt_fused_layernorm_gemv")


def mt_rmsnorm_backward_noalloc(X, gamma, dY, rstd, dX, dgamma, N, D, stream=None):
    """RMSNorm backward with the library's fixed scratch array (no allocation).

    For callers that may not allocate device memory; see include/mt_norm.h. The
    first call on a device must come before any stream capture; calls must not
    overlap on the GPU.
    """
    _check(load().mt_rmsnorm_backward_noalloc(_ptr(X), _ptr(gamma), _ptr(dY), _ptr(rstd),
                                              _ptr(dX), _ptr(dgamma), N, D, _stream(stream)),
           "mt_rmsnorm_backward_noalloc")


def mt_norm_backward_workspace_size(op, N, D, device=0) -> int:
    out = _SZ(0)
    _check(load().mt_norm_backward_workspace_size(op, N, D, device, ctypes.byref(out)),
           "mt_norm_backward_workspace_size")
    return int(out.value)


def mt_last_cuda_error() -> int:
    return load().mt_last_cuda_error()


def mt_device_wait_errors(device: int = 0, clear: bool = False) -> int:
    """Error bits of the device's bounded waits (0: none has given up); see the header."""
    v = ctypes.c_uint(0)
    _check(load().mt_device_wait_errors(int(device), ctypes.byref(v), 1 if clear else 0),
           "mt_device_wait_errors")
    return v.value


def mt_status_string(status: int) -> str:
    return load().mt_status_string(status).decode()


def mt_norm_version() -> int:
    return load().mt_norm_version()


# ---------------------------------------------------- allocating wrappers ---

def _new(like, shape, dtype):
    import torch
    return torch.empty(shape, dtype=dtype, device=like.device)


def _workspace(op, x):
    import torch
    n, d = x.shape
    nbytes = mt_norm_backward_workspace_size(op, n, d, x.device.index or 0)
    return torch.empty(nbytes, dtype=torch.uint8, device=x.device), nbytes


def rmsnorm_forward(x, gamma, eps=1e-5):
    """-> (y fp16 [N,D], rstd fp32 [N])"""
    import torch
    n, d = x.shape
    y = _new(x, (n, d), torch.float16)
    rstd = _new(x, (n,), torch.float32)
    mt_rmsnorm_forward(x, gamma, y, rstd, n, d, eps)
    return y, rstd


def rmsnorm_backward(x, gamma, dy, rstd):
    """-> (dx fp16 [N,D], dgamma fp32 [D])"""
    import torch
    n, d = x.shape
    dx = _new(x, (n, d), torch.float16)
    dgamma = _new(x, (d,), torch.float32)
    ws, nbytes = _workspace(MT_OP_RMSNORM, x)
    mt_rmsnorm_backward_ws(x, gamma, dy, rstd, dx, dgamma, n, d, ws, nbytes)
    return dx, dgamma


def layernorm_forward(x, gamma, beta, eps=1e-5):
    """-> (y fp16 [N,D], mean fp32 [N], rstd fp32 [N])"""
    import torch
    n, d = x.shape
    y = _new(x, (n, d), torch.float16)
    mean = _new(x, (n,), torch.float32)
    rstd = _new(x, (n,), torch.float32)
    mt_layernorm_forward(x, gamma, beta, y, mean, rstd, n, d, eps)
    return y, mean, rstd


def layernorm_backward(x, gamma, dy, mean, rstd):
    """-> (dx fp16 [N,D], dgamma fp32 [D], dbeta fp32 [D])"""
    import torch
    n, d = x.shape
    dx = _new(x, (n, d), torch.float16)
    dgamma = _new(x, (d,), torch.float32)
    dbeta = _new(x, (d,), torch.float32)
    ws, nbytes = _workspace(MT_OP_LAYERNORM, x)
    mt_layernorm_backward_ws(x, gamma, dy, mean, rstd, dx, dgamma, dbeta, n, d, ws, nbytes)
    return dx, dgamma, dbeta


def add_rmsnorm_forward(x, r, gamma, eps=1e-5):
    """-> (y fp16 [N,D], s fp16 [N,D] residual sum, rstd fp32 [N])"""
    import torch
    n, d = x.shape
    y = _new(x, (n, d), torch.float16)
    s = _new(x, (n, d), torch.float16)
    rstd = _new(x, (n,), torch.float32)
    mt_add_rmsnorm_forward(x, r, gamma, s, y, rstd, n, d, eps)
    return y, s, rstd


def add_rmsnorm_backward(s, gamma, dy, ds, rstd):
    """-> (dx fp16 [N,D] (= d source = d residual), dgamma fp32 [D]); ds may be None."""
    import torch
    n, d = s.shape
    dx = _new(s, (n, d), torch.float16)
    dgamma = _new(s, (d,), torch.float32)
    ws, nbytes = _workspace(MT_OP_ADD_RMSNORM, s)
    mt_add_rmsnorm_backward_ws(s, gamma, dy, ds, rstd, dx, dgamma, n, d, ws, nbytes)
    return dx, dgamma


# ------------------------------------------------ wrappers for any storage type ---

def dtype_code(torch_dtype) -> int:
    """mt_dtype_t of a torch dtype (float16, bfloat16 or float32)."""
    import torch
    codes = {torch.float16: MT_DTYPE_F16, torch.bfloat16: MT_DTYPE_BF16,
             torch.float32: MT_DTYPE_F32}
    if torch_dtype not in codes:
        raise TypeError(f"unsupported storage type {torch_dtype}")
    return codes[torch_dtype]


def norm_forward(op, x, gamma, beta=None, residual=None, eps=1e-5):
    """Forward of `op` for any storage types; the output (and residual sum) take x's type.

    Returns (y, rstd) for RMSNorm, (y, mean, rstd) for LayerNorm and (y, s, rstd) for the
    fused residual-add + RMSNorm.
    """
    import torch
    n, d = x.shape
    y = _new(x, (n, d), x.dtype)
    rstd = _new(x, (n,), torch.float32)
    mean = _new(x, (n,), torch.float32) if op == MT_OP_LAYERNORM else None
    s = _new(x, (n, d), x.dtype) if op == MT_OP_ADD_RMSNORM else None
    mt_norm_forward_ex(op, dtype_code(x.dtype), dtype_code(gamma.dtype), x, residual, gamma,
                       beta, s, y, mean, rstd, n, d, eps)
    if op == MT_OP_LAYERNORM:
        return y, mean, rstd
    if op == MT_OP_ADD_RMSNORM:
        return y, s, rstd
    return y, rstd


def norm_backward(op, x, gamma, dy, rstd, mean=None, ds=None):
    """Backward of `op` for any storage types (x is the saved S for the fused op).

    dx takes x's type; dgamma (and dbeta) are fp32. Returns (dx, dgamma) or, for
    LayerNorm, (dx, dgamma, dbeta).
    """
    import torch
    n, d = x.shape
    dx = _new(x, (n, d), x.dtype)
    dgamma = _new(x, (d,), torch.float32)
    dbeta = _new(x, (d,), torch.float32) if op == MT_OP_LAYERNORM else None
    ws, nbytes = _workspace(op, x)
    mt_norm_backward_ex(op, dtype_code(x.dtype), dtype_code(gamma.dtype), dtype_code(dy.dtype),
                        x, gamma, dy, ds, mean, rstd, dx, dgamma, dbeta, n, d, ws, nbytes)
    return (dx, dgamma, dbeta) if op == MT_OP_LAYERNORM else (dx, dgamma)


# ------------------------------------------------ row softmax, cross-entropy ---

_REDUCTIONS = {"none": MT_REDUCTION_NONE, "sum": MT_REDUCTION_SUM, "mean": MT_REDUCTION_MEAN}


def softmax_forward(x, log_softmax=False):
    """Row softmax (or log-softmax) of x [N, D]; the output takes x's type."""
    n, d = x.shape
    y = _new(x, (n, d), x.dtype)
    mt_softmax_forward(dtype_code(x.dtype), x, y, n, d, log_softmax)
    return y


def softmax_backward(y, dy, log_softmax=False):
    """Input gradient of the row softmax (log-softmax) from its output y and dy (same type)."""
    n, d = y.shape
    dx = _new(y, (n, d), y.dtype)
    mt_softmax_backward(dtype_code(y.dtype), y, dy, dx, n, d, log_softmax)
    return dx


def cross_entropy_forward(logits, targets, ignore_index=-100, label_smoothing=0.0, z_loss=0.0,
                          reduction="mean"):
    """-> (loss, lse, n_valid): loss [N] fp32 for "none", else a 1-element fp32 tensor;
    lse [N] fp32 (saved for the backward); n_valid a 1-element fp32 tensor (or None for
    "none"). targets: int64 [N] on the device."""
    import torch
    n, d = logits.shape
    rows = _new(logits, (n,), torch.float32)
    lse = _new(logits, (n,), torch.float32)
    red = _REDUCTIONS[reduction]
    out = _new(logits, (1,), torch.float32) if red else None
    nv = _new(logits, (1,), torch.float32) if red else None
    mt_cross_entropy_forward(dtype_code(logits.dtype), logits, targets, n, d, ignore_index,
                             label_smoothing, z_loss, red, rows, lse, out, nv)
    return (rows if red == MT_REDUCTION_NONE else out), lse, nv


def cross_entropy_backward(logits, targets, lse, dloss, n_valid=None, ignore_index=-100,
                           label_smoothing=0.0, z_loss=0.0, reduction="mean"):
    """Gradient of the reduced loss with respect to the logits (logits' type)."""
    n, d = logits.shape
    dx = _new(logits, (n, d), logits.dtype)
    mt_cross_entropy_backward(dtype_code(logits.dtype), logits, targets, lse, n, d, ignore_index,
                              label_smoothing, z_loss, _REDUCTIONS[reduction], dloss, n_valid, dx)
    return dx


def norm_gemv(x, gamma, w, beta=None, eps=1e-5):
    """Y = Norm(x, gamma[, beta]) @ w for a decode batch: RMSNorm when beta is None, else
    LayerNorm. x [M, K], w [K, N], all fp16 on the device -> Y [M, N] fp16."""
    import torch
    m, k = x.shape
    n = w.shape[1]
    y = _new(x, (m, n), torch.float16)
    if beta is None:
        mt_fused_rmsnorm_gemv(x, gamma, w, y, m, n, k, eps)
    else:
        mt_fused_layernorm_gemv(x, gamma, beta, w, y, m, n, k, eps)
    return y
