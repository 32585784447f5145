"""mt_rmsnorm_backward_noalloc: the RMSNorm backward for callers that may not allocate.

Some callers cannot allocate device memory while they run -- their device memory is
owned by a framework pool that must not be bypassed, or the loop they run in may not
call an allocator -- so they can use neither mt_rmsnorm_backward (which allocates its
scratch) nor mt_rmsnorm_backward_ws (which needs scratch from them). The no-alloc entry
point takes its scratch from a fixed array inside the library instead.

These tests call it through the C ABI on two calls in a row (the second reuses the
array the first one left behind) and hold it to two references:
  * the ordinary backward with a caller-supplied workspace: the same kernels with the
    same number of partial rows, so every output must agree bit for bit;
  * the fp64 oracle: dX on sampled rows (every row for small shapes) within the fp16
    tolerance, dgamma on every column within 1e-4 of the column's sum of |terms|.
The shapes cover every kernel family the call can take: the pipelined vector backward
(4096 and 16384 columns), the scalar kernel (ragged widths up to 16383 columns, and
misaligned rows), and rows split across a thread-block cluster (vector and scalar, up
to the widest supported row). On a 152-SM GB300 the largest scratch any of them needs
is about 10 MB (16383-column rows on the scalar kernel: one partial row per SM; split
rows: one per cluster), below the array's MT_NOALLOC_SCRATCH_BYTES.

This file is collected last so that a run stopping at the first failure has already run
every other test.
"""
import numpy as np
import pytest
import torch

import row_wise_rmsnorm_gb300 as mt
import workloads as W
from parity import check_fp16, check_param, f64, oracle_run

# fake addresses: validation rejects these calls before any CUDA call
A, B, C, E, F, G = (0x10000 * (i + 1) for i in range(6))

EPS = 1e-6


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


def _workspace_backward(X, gamma, dY, rstd):
    """The ordinary backward (caller-supplied workspace) on the same inputs."""
    N, D = X.shape
    dX = torch.empty_like(X)
    dg = torch.empty(D, dtype=torch.float32, device=X.device)
    need = mt.mt_norm_backward_workspace_size(mt.MT_OP_RMSNORM, N, D, X.device.index or 0)
    ws = torch.empty(need, dtype=torch.uint8, device=X.device)
    mt.mt_rmsnorm_backward_ws(X, gamma, dY, rstd, dX, dg, N, D, ws, need)
    return dX, dg


def _misaligned(t, dev):
    """Copies of the tensors that start 2 bytes past a 16-byte boundary (scalar path)."""
    out = {}
    for k, v in t.items():
        buf = torch.empty(v.numel() + 8, dtype=v.dtype, device=dev)
        view = buf[1:1 + v.numel()].view(v.shape)
        view.copy_(v.to(dev))
        assert view.data_ptr() % 16 == 2
        out[k] = view
    return out


# (N, D, misaligned): the vector pipelined backward at 4096 and 16384 columns (the first
# is the Llama-7B activation shape); the scalar kernel at ragged widths; misaligned rows;
# split rows on a cluster (vector: 131072 and 100000 columns, the latter with a short last
# slice and clusters that loop over several rows; scalar: 131071).
SHAPES = [(16384, 4096, False), (4000, 16384, False), (1000, 257, False), (64, 4095, False),
          (64, 8191, False), (64, 16383, False), (37, 16384, True), (3, 131072, False),
          (40, 100000, False), (3, 131071, False)]


@pytest.mark.gpu
@pytest.mark.parametrize("N,D,misaligned", SHAPES)
def test_noalloc_matches_workspace_backward_and_oracle_twice(N, D, misaligned):
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for the -m gpu tests")
    from row_wise_rmsnorm_gb300 import build
    build.build()
    dev = torch.device("cuda:0")
    rng = np.random.default_rng(N + D)
    rows = np.arange(N) if N * D <= (1 << 22) else np.unique(
        np.concatenate([[0, N - 1], rng.integers(0, N, 62)]))
    for call, seed in enumerate((101, 202)):
        host = W.generate("rmsnorm", N, D, seed=seed, x_kind="row_scaled", dy_std=1.0)
        t = _misaligned(host, dev) if misaligned else {k: v.to(dev) for k, v in host.items()}
        X, gamma, dY = t["X"], t["gamma"], t["dY"]
        y, rstd = mt.rmsnorm_forward(X, gamma, eps=EPS)
        ref_dX, ref_dg = _workspace_backward(X, gamma, dY, rstd)
        dX = torch.full_like(X, float("nan"))
        dg = torch.full((D,), float("nan"), dtype=torch.float32, device=dev)
        mt.mt_rmsnorm_backward_noalloc(X, gamma, dY, rstd, dX, dg, N, D)
        torch.cuda.synchronize()
        tag = f"noalloc {N}x{D}{' misaligned' if misaligned else ''} call {call}"
        # same kernels, same partial rows: bit for bit
        assert torch.equal(dX.view(torch.int16), ref_dX.view(torch.int16)), f"{tag}: dX bits"
        assert torch.equal(dg.view(torch.int32), ref_dg.view(torch.int32)), f"{tag}: dgamma bits"
        # and the oracle
        ref = oracle_run(W.RMSNORM, host, EPS, rows=rows)
        sel = torch.as_tensor(rows, device=dev)
        check_fp16(dX[sel], ref["dX"], f"{tag} dX")
        check_param(dg, ref["dgamma"], ref["dgamma_abs"], f"{tag} dgamma")
        assert np.isfinite(f64(dg)).all(), tag
