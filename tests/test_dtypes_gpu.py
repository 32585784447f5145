"""bf16 and fp32 storage, and parameter/cotangent types independent of the activations,
through the explicit-dtype C entry points, against the fp64 oracle on the same stored
inputs (meTile "Kernel coverage and training scope", "Exact native normalization
contract": storage FP16 or FP32 with weight, bias and cotangents each in either type,
FP32 statistics and parameter gradients; bf16 is this library's addition).

The combinations cover every vector-kernel family (all three types equal; fp32
parameters and/or cotangents with fp16/bf16 activations; all fp32) and two that only
the scalar kernels serve. The shapes cover the scalar path (ragged width), narrow and
wide vector tables, a width with a ragged last tile, and 16384-wide rows, where an
all-fp32 backward ring does not fit and the scalar backward takes over.
"""
import numpy as np
import pytest
import torch

import row_wise_rmsnorm_gb300 as mt
import workloads as W
from parity import STORAGE, check_out, compare_ex, f64, gpu_run_ex, oracle_run

pytestmark = pytest.mark.gpu

F16, BF16, F32 = torch.float16, torch.bfloat16, torch.float32
COMBOS = [
    (BF16, BF16, BF16), (F32, F32, F32),                      # one type throughout
    (F16, F32, F16), (BF16, F32, BF16),                       # fp32 parameters
    (F16, F16, F32), (BF16, F32, F32),                        # fp32 cotangents
    (F32, F16, BF16), (BF16, F16, F16),                       # scalar kernels only
]
SHAPES = [(17, 257), (96, 1024), (40, 4104), (9, 16384)]
OPS = [W.RMSNORM, W.LAYERNORM, W.ADD_RMSNORM]


def _name(c):
    return "-".join(STORAGE[t] for t in c)


def _inputs(op, N, D, combo, seed=3, x_kind="normal"):
    x, w, g = combo
    return W.generate(op, N, D, device="cuda", seed=seed, x_kind=x_kind, dy_std=1.0,
                      x_dtype=x, w_dtype=w, g_dtype=g)


@pytest.mark.parametrize("combo", COMBOS, ids=_name)
@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("op", OPS)
def test_dtype_parity(op, shape, combo):
    N, D = shape
    t = _inputs(op, N, D, combo)
    eps = 1e-5
    got = gpu_run_ex(op, t, eps)
    torch.cuda.synchronize()
    ref = oracle_run(op, t, eps, x_storage=STORAGE[combo[0]])
    compare_ex(op, got, ref, t["X"], tag=f"{op} {N}x{D} {_name(combo)}")


@pytest.mark.parametrize("combo", COMBOS[:6], ids=_name)
def test_fused_without_residual_cotangent(combo):
    N, D = 64, 2048
    t = _inputs(W.ADD_RMSNORM, N, D, combo)
    got = gpu_run_ex(W.ADD_RMSNORM, t, 1e-6, use_ds=False)
    ref = oracle_run(W.ADD_RMSNORM, t, 1e-6, use_ds=False, x_storage=STORAGE[combo[0]])
    compare_ex(W.ADD_RMSNORM, got, ref, t["X"], tag=f"add noDS {_name(combo)}")


@pytest.mark.parametrize("combo", [(BF16, BF16, BF16), (F32, F32, F32), (BF16, F32, F32)],
                         ids=_name)
def test_layernorm_large_mean(combo):
    """X = 50 + N(0,1) in each storage type: the centred two-pass statistics hold."""
    N, D = 48, 4096
    t = _inputs(W.LAYERNORM, N, D, combo, x_kind="shifted")
    got = gpu_run_ex(W.LAYERNORM, t, 1e-5)
    ref = oracle_run(W.LAYERNORM, t, 1e-5, x_storage=STORAGE[combo[0]])
    compare_ex(W.LAYERNORM, got, ref, t["X"], tag=f"ln shifted {_name(combo)}")


@pytest.mark.parametrize("dtype", [BF16, F32], ids=lambda d: STORAGE[d])
def test_misaligned_rows_take_the_scalar_path(dtype):
    """Row bases one element off 16 bytes: the scalar kernels, same results."""
    N, D = 33, 1024
    combo = (dtype, dtype, dtype)
    t = _inputs(W.RMSNORM, N, D, combo)
    buf = torch.empty(N * D + 1, dtype=dtype, device="cuda")
    xs = buf[1:].view(N, D)
    xs.copy_(t["X"])
    t2 = dict(t, X=xs)
    got = gpu_run_ex(W.RMSNORM, t2, 1e-6)
    ref = oracle_run(W.RMSNORM, t, 1e-6, x_storage=STORAGE[dtype])
    compare_ex(W.RMSNORM, got, ref, t["X"], tag=f"misaligned {STORAGE[dtype]}")


def test_fp16_through_the_explicit_entry_points_is_bitwise_the_fp16_api():
    N, D = 256, 4096
    t = W.generate(W.LAYERNORM, N, D, device="cuda", seed=5, dy_std=1.0)
    a = gpu_run_ex(W.LAYERNORM, t, 1e-5)
    from parity import gpu_run
    b = gpu_run(W.LAYERNORM, t, 1e-5)
    for k in ("Y", "rstd", "mean", "dX", "dgamma", "dbeta"):
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("combo", [(BF16, BF16, BF16), (F32, F32, F32), (BF16, F32, F32)],
                         ids=_name)
def test_deterministic(combo):
    N, D = 512, 4096
    t = _inputs(W.ADD_RMSNORM, N, D, combo)
    a = gpu_run_ex(W.ADD_RMSNORM, t, 1e-6)
    b = gpu_run_ex(W.ADD_RMSNORM, t, 1e-6)
    for k in a:
        assert torch.equal(a[k], b[k]), k


@pytest.mark.parametrize("dtype", [BF16, F32], ids=lambda d: STORAGE[d])
def test_full_size_sampled(dtype):
    """RMSNorm at 16384 x 4096 in one storage type: sampled rows of Y and dX against the
    oracle (which computes those rows one by one), dgamma through the property that it
    equals the sum over rows of dY * xhat (checked against fp64 on the GPU outputs'
    own inputs for a column sample)."""
    N, D = 16384, 4096
    combo = (dtype, dtype, dtype)
    t = W.generate(W.RMSNORM, N, D, device="cuda", seed=0, x_kind="row_scaled", dy_std=0.01,
                   x_dtype=dtype, w_dtype=dtype, g_dtype=dtype)
    got = gpu_run_ex(W.RMSNORM, t, 1e-6)
    rows = np.array([0, 1, 777, 8191, 12345, N - 1])
    sub = {k: v[torch.as_tensor(rows, device="cuda")] if v.dim() == 2 else v
           for k, v in t.items()}
    ref = oracle_run(W.RMSNORM, sub, 1e-6, x_storage=STORAGE[dtype])
    check_out(got["Y"][torch.as_tensor(rows, device="cuda")], ref["Y"], dtype, "Y rows")
    check_out(got["dX"][torch.as_tensor(rows, device="cuda")], ref["dX"], dtype, "dX rows")
    cols = torch.as_tensor([0, 5, 1000, 4095], device="cuda")
    x = f64(t["X"][:, cols])
    dy = f64(t["dY"][:, cols])
    r = f64(got["rstd"])[:, None]
    want = (dy * x * r).sum(axis=0)
    tol = 1e-4 * np.abs(dy * x * r).sum(axis=0) + 1e-7
    assert np.all(np.abs(f64(got["dgamma"][cols]) - want) <= tol)
