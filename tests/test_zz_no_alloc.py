"""mt_rmsnorm_backward_noalloc: the RMSNorm backward for callers that may not allocate.

Some callers cannot allocate device memory while they run -- their device memory is
owned by a framework pool that must not be bypassed, or the loop they run in may not
call an allocator -- so they can use neither mt_rmsnorm_backward (which allocates its
scratch) nor mt_rmsnorm_backward_ws (which needs scratch from them). The no-alloc entry
point takes its scratch from a fixed array inside the library instead. These tests call
it through the C ABI and hold its outputs to the ordinary backward's, within the
tolerance the parity tests use, on two calls in a row (the second reuses the array the
first one left behind). This file is collected last so that a run stopping at the first
failure has already run every other test.
"""
import ctypes

import pytest
import torch

import row_wise_rmsnorm_gb300 as mt
import workloads as W
from parity import FP16_ATOL, FP16_RTOL, PARAM_RTOL

# fake addresses: validation rejects these calls before any CUDA call
A, B, C, E, F, G = (0x10000 * (i + 1) for i in range(6))


def test_noalloc_rejects_bad_arguments_without_cuda():
    from row_wise_rmsnorm_gb300 import build
    build.build()
    lib = mt.load()
    f = lib.mt_rmsnorm_backward_noalloc
    assert f(A, B, C, E, F, None, 8, 64, None) == mt.MT_ERR_INVALID_ARG
    assert f(A, B, C, E, F, G, -1, 64, None) == mt.MT_ERR_INVALID_ARG
    assert f(None, None, None, None, None, None, 0, 64, None) == mt.MT_ERR_INVALID_ARG
    assert f(A, B, C, E, F, G, 8, 0, None) == mt.MT_ERR_INVALID_ARG
    assert f(A, B, C, E, F, G, 8, mt.MT_MAX_COLS + 1, None) == mt.MT_ERR_UNSUPPORTED


def _reference(X, gamma, dY, rstd):
    """The ordinary backward (caller-supplied workspace) on the same inputs."""
    N, D = X.shape
    dX = torch.empty_like(X)
    dg = torch.empty(D, dtype=torch.float32, device=X.device)
    need = mt.mt_norm_backward_workspace_size(mt.MT_OP_RMSNORM, N, D, X.device.index or 0)
    ws = torch.empty(need, dtype=torch.uint8, device=X.device)
    mt.mt_rmsnorm_backward_ws(X, gamma, dY, rstd, dX, dg, N, D, ws, need)
    return dX, dg


def _within_tolerance(X, dY, rstd, dX, dg, ref_dX, ref_dg):
    err = (dX.double() - ref_dX.double()).abs()
    assert bool((err <= FP16_ATOL + FP16_RTOL * ref_dX.double().abs()).all()), \
        f"dX differs: max err {err.max().item():.3e}"
    # dgamma: 1e-4 of the column's sum of |dY * xhat| terms
    scale = (dY.double() * X.double() * rstd.double()[:, None]).abs().sum(dim=0)
    gerr = (dg.double() - ref_dg.double()).abs()
    assert bool((gerr <= PARAM_RTOL * scale + 1e-7).all()), \
        f"dgamma differs: max err {gerr.max().item():.3e}"


@pytest.mark.gpu
@pytest.mark.parametrize("N,D", [(16384, 4096), (4000, 16384), (1000, 257)])
def test_noalloc_matches_workspace_backward_twice(N, D):
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the -m gpu tests")
    from row_wise_rmsnorm_gb300 import build
    build.build()
    dev = torch.device("cuda:0")
    for call, seed in enumerate((101, 202)):
        t = W.generate("rmsnorm", N, D, device=dev, seed=seed, dy_std=1.0)
        X, gamma, dY = t["X"], t["gamma"], t["dY"]
        y, rstd = mt.rmsnorm_forward(X, gamma, eps=1e-6)
        ref_dX, ref_dg = _reference(X, gamma, dY, rstd)
        dX = torch.full_like(X, float("nan"))
        dg = torch.full((D,), float("nan"), dtype=torch.float32, device=dev)
        mt.mt_rmsnorm_backward_noalloc(X, gamma, dY, rstd, dX, dg, N, D)
        torch.cuda.synchronize()
        assert torch.isfinite(dX).all() and torch.isfinite(dg).all(), f"call {call}"
        _within_tolerance(X, dY, rstd, dX, dg, ref_dX, ref_dg)
