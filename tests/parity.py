"""Run one op on the GPU (through the C ABI) and on the fp64 oracle, and compare.

Tolerances (GPU vs oracle, every element checked):
  * fp16 outputs Y, dX:    |gpu - ref| <= 2e-3 + 2e-3 |ref|   (about 4 half-ulps of fp16)
  * bf16 outputs Y, dX:    |gpu - ref| <= 8e-3 + 8e-3 |ref|   (the same 4 half-ulps of bf16,
                           whose half-ulp 2^-9 is 4x fp16's 2^-11)
  * fp32 outputs Y, dX:    |gpu - ref| <= 1e-5 + 1e-5 |ref|   (fp32 arithmetic: rounding of
                           the row sums, about (32 + log2 D) * 2^-24 relative, and rsqrtf's
                           2 ulp, with a margin of 5 or more)
  * rstd:                  |gpu - ref| <= 1e-5 |ref|
  * mean (LayerNorm):      |gpu - ref| <= 1e-5 mean_j|x_ij| + 1e-7 (a mean near zero has no
                           relative accuracy; the sum's natural scale is mean|x|)
  * dgamma_j, dbeta_j:     |gpu - ref| <= 1e-4 sum_i |term_ij| + 1e-7
  * S (fused op):          bit-exact: x + r rounded once to the storage type, nearest even
                           (the kernel rounds the fp32 sum; fp32 keeps 24 >= 2p + 2 bits of a
                           sum of two p-bit values, so that second rounding is innocuous)
NaN must sit in the same places on both sides.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import row_wise_rmsnorm_gb300 as mt
import workloads as W

FP16_ATOL = 2e-3
FP16_RTOL = 2e-3
# (atol, rtol) of an output stored in each type
OUT_TOL = {torch.float16: (2e-3, 2e-3), torch.bfloat16: (8e-3, 8e-3), torch.float32: (1e-5, 1e-5)}
STORAGE = {torch.float16: "f16", torch.bfloat16: "bf16", torch.float32: "f32"}
STAT_RTOL = 1e-5
PARAM_RTOL = 1e-4


def f64(t) -> np.ndarray:
    if isinstance(t, torch.Tensor):
        return t.detach().cpu().double().numpy()
    return np.asarray(t, dtype=np.float64)


def _same_nans(got, ref, what):
    gn, rn = np.isnan(got), np.isnan(ref)
    assert np.array_equal(gn, rn), f"{what}: NaN positions differ ({gn.sum()} vs {rn.sum()})"
    return ~rn


def _report(err, bound, what):
    bad = ~(err <= bound)
    if bad.any():
        idx = np.argwhere(bad)[:5].tolist()
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; "
                             f"max err {np.max(err):.3e}, max err/bound "
                             f"{np.max(err / bound):.3f}; first at {idx}")


def check_fp16(got, ref, what):
    got, ref = f64(got), f64(ref)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    m = _same_nans(got, ref, what)
    err = np.abs(got[m] - ref[m])
    _report(err, FP16_ATOL + FP16_RTOL * np.abs(ref[m]), what)


def check_out(got, ref, dtype, what):
    """An output stored as `dtype` against the oracle, with that type's tolerance."""
    atol, rtol = OUT_TOL[dtype]
    got, ref = f64(got), f64(ref)
    assert got.shape == ref.shape, f"{what}: shape {got.shape} vs {ref.shape}"
    m = _same_nans(got, ref, what)
    err = np.abs(got[m] - ref[m])
    _report(err, atol + rtol * np.abs(ref[m]), what)


def check_rstd(got, ref, what="rstd"):
    got, ref = f64(got), f64(ref)
    m = _same_nans(got, ref, what)
    _report(np.abs(got[m] - ref[m]), STAT_RTOL * np.abs(ref[m]), what)


def check_mean(got, ref, X, what="mean"):
    got, ref = f64(got), f64(ref)
    scale = np.mean(np.abs(f64(X)), axis=1)
    m = _same_nans(got, ref, what)
    _report(np.abs(got[m] - ref[m]), STAT_RTOL * scale[m] + 1e-7, what)


def check_param(got, ref, ref_abs, what):
    got, ref, ref_abs = f64(got), f64(ref), f64(ref_abs)
    m = _same_nans(got, ref, what)
    _report(np.abs(got[m] - ref[m]), PARAM_RTOL * ref_abs[m] + 1e-7, what)


# ---------------------------------------------------------------- GPU runs ---

def gpu_run(op: str, t: dict, eps: float, *, use_ds: bool = True, stream=None) -> dict:
    """Forward then backward of `op` on the GPU through the C-named binding.

    `t` holds fp16 CUDA tensors (X, gamma, dY, and R/dS or beta by op). Outputs are
    freshly allocated; the backward consumes the forward's saved tensors.
    """
    X, gamma, dY = t["X"], t["gamma"], t["dY"]
    N, D = X.shape
    dev = X.device
    out: dict[str, torch.Tensor] = {}
    h = dict(dtype=torch.float16, device=dev)
    f = dict(dtype=torch.float32, device=dev)
    Y = torch.empty((N, D), **h)
    rstd = torch.empty(N, **f)
    dX = torch.empty((N, D), **h)
    dg = torch.empty(D, **f)
    if op == W.RMSNORM:
        mt.mt_rmsnorm_forward(X, gamma, Y, rstd, N, D, eps, stream)
        ws_n = mt.mt_norm_backward_workspace_size(mt.MT_OP_RMSNORM, N, D, dev.index or 0)
        ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
        mt.mt_rmsnorm_backward_ws(X, gamma, dY, rstd, dX, dg, N, D, ws, ws_n, stream)
    elif op == W.LAYERNORM:
        mean = torch.empty(N, **f)
        db = torch.empty(D, **f)
        mt.mt_layernorm_forward(X, gamma, t["beta"], Y, mean, rstd, N, D, eps, stream)
        ws_n = mt.mt_norm_backward_workspace_size(mt.MT_OP_LAYERNORM, N, D, dev.index or 0)
        ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
        mt.mt_layernorm_backward_ws(X, gamma, dY, mean, rstd, dX, dg, db, N, D, ws, ws_n, stream)
        out.update(mean=mean, dbeta=db)
    else:
        S = torch.empty((N, D), **h)
        mt.mt_add_rmsnorm_forward(X, t["R"], gamma, S, Y, rstd, N, D, eps, stream)
        dS = t.get("dS") if use_ds else None
        ws_n = mt.mt_norm_backward_workspace_size(mt.MT_OP_ADD_RMSNORM, N, D, dev.index or 0)
        ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
        mt.mt_add_rmsnorm_backward_ws(S, gamma, dY, dS, rstd, dX, dg, N, D, ws, ws_n, stream)
        out.update(S=S)
    out.update(Y=Y, rstd=rstd, dX=dX, dgamma=dg)
    return out


def gpu_run_ex(op: str, t: dict, eps: float, *, use_ds: bool = True, stream=None) -> dict:
    """Forward then backward through mt_norm_forward_ex / mt_norm_backward_ex, the storage
    types taken from the tensors (X/R: activations, gamma/beta: parameters, dY/dS:
    cotangents). Outputs Y, S and dX take the activation type."""
    X, gamma, dY = t["X"], t["gamma"], t["dY"]
    N, D = X.shape
    dev = X.device
    xt, wt, gt = mt.dtype_code(X.dtype), mt.dtype_code(gamma.dtype), mt.dtype_code(dY.dtype)
    f = dict(dtype=torch.float32, device=dev)
    op_code = {W.RMSNORM: mt.MT_OP_RMSNORM, W.LAYERNORM: mt.MT_OP_LAYERNORM,
               W.ADD_RMSNORM: mt.MT_OP_ADD_RMSNORM}[op]
    Y = torch.empty((N, D), dtype=X.dtype, device=dev)
    rstd = torch.empty(N, **f)
    mean = torch.empty(N, **f) if op == W.LAYERNORM else None
    S = torch.empty((N, D), dtype=X.dtype, device=dev) if op == W.ADD_RMSNORM else None
    mt.mt_norm_forward_ex(op_code, xt, wt, X, t.get("R"), gamma, t.get("beta"), S, Y, mean, rstd,
                          N, D, eps, stream)
    dX = torch.empty((N, D), dtype=X.dtype, device=dev)
    dg = torch.empty(D, **f)
    db = torch.empty(D, **f) if op == W.LAYERNORM else None
    ws_n = mt.mt_norm_backward_workspace_size(op_code, N, D, dev.index or 0)
    ws = torch.empty(ws_n, dtype=torch.uint8, device=dev)
    dS = t.get("dS") if (use_ds and op == W.ADD_RMSNORM) else None
    mt.mt_norm_backward_ex(op_code, xt, wt, gt, S if op == W.ADD_RMSNORM else X, gamma, dY, dS,
                           mean, rstd, dX, dg, db, N, D, ws, ws_n, stream)
    out = dict(Y=Y, rstd=rstd, dX=dX, dgamma=dg)
    if mean is not None:
        out.update(mean=mean, dbeta=db)
    if S is not None:
        out.update(S=S)
    return out


def compare_ex(op: str, got: dict, ref: dict, X, tag=""):
    """Check every output of gpu_run_ex against oracle_run(..., x_storage=...)."""
    dt = got["Y"].dtype
    check_out(got["Y"], ref["Y"], dt, f"{tag} Y")
    check_rstd(got["rstd"], ref["rstd"], f"{tag} rstd")
    check_out(got["dX"], ref["dX"], dt, f"{tag} dX")
    check_param(got["dgamma"], ref["dgamma"], ref["dgamma_abs"], f"{tag} dgamma")
    if op == W.LAYERNORM:
        check_mean(got["mean"], ref["mean"], f64(X), f"{tag} mean")
        check_param(got["dbeta"], ref["dbeta"], ref["dbeta_abs"], f"{tag} dbeta")
    if op == W.ADD_RMSNORM:
        s_gpu = f64(got["S"])
        assert np.array_equal(s_gpu, ref["S_st"]), f"{tag} S not x + r rounded once"


# ------------------------------------------------------------- oracle runs ---

def oracle_run(op: str, t: dict, eps: float, *, use_ds: bool = True, rows=None,
               x_storage: str = "f16") -> dict:
    """The same forward + backward on the fp64 oracle from the same stored inputs.

    ``rows`` (an index array) restricts Y/dX/stats to those rows; dgamma/dbeta always
    cover every row. For the fused op the backward takes the oracle's own S, rounded to
    the activation storage type ``x_storage`` ("f16", "bf16" or "f32"; also in "S_st").
    """
    eps = float(np.float32(eps))  # the GPU receives eps as fp32
    X = f64(t["X"])
    gamma = f64(t["gamma"])
    dY = f64(t["dY"])
    ref: dict[str, np.ndarray] = {}
    if op == W.RMSNORM:
        Y, rstd = oracle.rmsnorm_forward(X, gamma, eps)
        dX, dg, dga = oracle.rmsnorm_backward(X, gamma, dY, rstd)
    elif op == W.LAYERNORM:
        beta = f64(t["beta"])
        Y, mean, rstd = oracle.layernorm_forward(X, gamma, beta, eps)
        dX, dg, db, dga, dba = oracle.layernorm_backward(X, gamma, dY, mean, rstd)
        ref.update(mean=mean, dbeta=db, dbeta_abs=dba)
    else:
        R = f64(t["R"])
        Y, S_exact, rstd = oracle.add_rmsnorm_forward(X, R, gamma, eps)
        S16 = oracle.round_fp16(S_exact)
        S_st = oracle.round_storage(S_exact, x_storage)
        dS = f64(t["dS"]) if (use_ds and "dS" in t) else None
        dX, dg, dga = oracle.add_rmsnorm_backward(S_st, gamma, dY, dS, rstd)
        ref.update(S16=S16, S_st=S_st)
    ref.update(Y=Y, rstd=rstd, dX=dX, dgamma=dg, dgamma_abs=dga)
    if rows is not None:
        for k in ("Y", "dX", "rstd", "mean", "S16", "S_st"):
            if k in ref:
                ref[k] = ref[k][rows]
    return ref


def compare(op: str, got: dict, ref: dict, X, rows=None, tag=""):
    """Check every output of `got` (GPU) against `ref` (oracle)."""
    def sel(a):
        if rows is None:
            return a
        if isinstance(a, torch.Tensor):
            return a[torch.as_tensor(rows, device=a.device)]
        return a[rows]
    check_fp16(sel(got["Y"]), ref["Y"], f"{tag} Y")
    check_rstd(sel(got["rstd"]), ref["rstd"], f"{tag} rstd")
    check_fp16(sel(got["dX"]), ref["dX"], f"{tag} dX")
    check_param(got["dgamma"], ref["dgamma"], ref["dgamma_abs"], f"{tag} dgamma")
    if op == W.LAYERNORM:
        check_mean(sel(got["mean"]), ref["mean"], sel(f64(X)), f"{tag} mean")
        check_param(got["dbeta"], ref["dbeta"], ref["dbeta_abs"], f"{tag} dbeta")
    if op == W.ADD_RMSNORM and "S" in got:
        s_gpu = sel(got["S"]).cpu().numpy()
        s_ref = ref["S16"]
        assert np.array_equal(s_gpu.view(np.uint16), s_ref.view(np.uint16)), \
            f"{tag} S not bit-exact fp16(x + r)"
