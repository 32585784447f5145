"""Rows wider than 16384 columns and the empty batch, against the fp64 oracle on the
same stored inputs.

The pages bound a row to 8192 columns (meTile "Exact native normalization contract");
the library widens the bound to 131072. An aligned row of more than 16384 columns runs
its forward on one CTA in two passes (LayerNorm merging per-thread centred sums by
Chan's update); the backward, and the forward of misaligned or ragged rows, run on a
cluster of 2, 4 or 8 CTAs, each a slice of the row, adding the CTAs' row sums in a fixed
order. The oracle's definitions apply unchanged. The widths cover each cluster size
(16392 and 24576: 2 CTAs; 40000 and 65536: 4; 131072: 8) and each streaming shape,
ragged widths and misaligned rows (the scalar kernels, also split), every op, the
storage types, more rows than resident clusters (the persistent backward loops), rows
far from zero mean, and N = 0.
"""
import numpy as np
import pytest
import torch

import oracle
import row_wise_rmsnorm_gb300 as mt
import workloads as W
from parity import STORAGE, check_out, check_rstd, compare_ex, f64, gpu_run_ex, oracle_run

pytestmark = pytest.mark.gpu

F16, BF16, F32 = torch.float16, torch.bfloat16, torch.float32
OPS = [W.RMSNORM, W.LAYERNORM, W.ADD_RMSNORM]
SHAPES = [(7, 16392), (5, 24576), (3, 40000), (4, 65536), (2, 131072), (3, 20001), (2, 131071)]


def _inputs(op, N, D, combo=(F16, F16, F16), seed=3, x_kind="normal"):
    x, w, g = combo
    return W.generate(op, N, D, device="cuda", seed=seed, x_kind=x_kind, dy_std=1.0,
                      x_dtype=x, w_dtype=w, g_dtype=g)


def _name(c):
    return "-".join(STORAGE[t] for t in c)


@pytest.mark.parametrize("shape", SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("op", OPS)
def test_wide_parity(op, shape):
    N, D = shape
    t = _inputs(op, N, D)
    got = gpu_run_ex(op, t, 1e-5)
    torch.cuda.synchronize()
    ref = oracle_run(op, t, 1e-5, x_storage="f16")
    compare_ex(op, got, ref, t["X"], tag=f"{op} {N}x{D}")


COMBOS = [(BF16, BF16, BF16), (F32, F32, F32), (F16, F32, F32), (BF16, F32, BF16)]


@pytest.mark.parametrize("D", [32768, 131072])
@pytest.mark.parametrize("combo", COMBOS, ids=_name)
@pytest.mark.parametrize("op", OPS)
def test_wide_storage_types(op, combo, D):
    """Every family of the split kernels: matching 2-byte types, all fp32 (its backward
    slices are 8192 columns, so 131072 columns take 16-CTA clusters), fp32
    parameters or cotangents."""
    N = 3
    t = _inputs(op, N, D, combo)
    got = gpu_run_ex(op, t, 1e-5)
    torch.cuda.synchronize()
    ref = oracle_run(op, t, 1e-5, x_storage=STORAGE[combo[0]])
    compare_ex(op, got, ref, t["X"], tag=f"{op} {N}x{D} {_name(combo)}")


@pytest.mark.parametrize("D", [65544, 100000])
@pytest.mark.parametrize("op", OPS)
def test_wide_all_fp32_sixteen_cta_clusters(op, D):
    """All-fp32 backwards of rows wider than 65536 columns take 16-CTA clusters of
    8192-column slices. At these ragged widths the last slice is short (65544: slices of
    4104 columns, the last 3984; 100000: 6256, the last 6160), and with 40 rows every
    resident cluster runs several rows and sums them into its partial row. Every output
    against the oracle, and a second run bit for bit."""
    N = 40
    t = _inputs(op, N, D, (F32, F32, F32), seed=5)
    got = gpu_run_ex(op, t, 1e-5)
    again = gpu_run_ex(op, t, 1e-5)
    torch.cuda.synchronize()
    ref = oracle_run(op, t, 1e-5, x_storage="f32")
    compare_ex(op, got, ref, t["X"], tag=f"{op} {N}x{D} f32 16-CTA")
    for k in got:
        assert torch.equal(got[k].view(torch.int32), again[k].view(torch.int32)), k


def test_split_row_exchange_waits_never_give_up():
    """The split-row backward exchanges row sums by pushing them into the peers' shared
    memory and waiting, bounded, on the CTA's own mbarrier. Over every cluster size (2, 4,
    8 and the all-fp32 16) and many rows per cluster, the outputs match the oracle and the
    device's wait-error word stays 0."""
    mt.mt_device_wait_errors(0, clear=True)
    for op, N, D, combo in [(W.RMSNORM, 200, 24576, (F16, F16, F16)),
                            (W.LAYERNORM, 120, 65536, (BF16, BF16, BF16)),
                            (W.ADD_RMSNORM, 60, 131072, (F16, F16, F16)),
                            (W.LAYERNORM, 40, 131072, (F32, F32, F32))]:
        t = _inputs(op, N, D, combo, seed=9)
        got = gpu_run_ex(op, t, 1e-5)
        torch.cuda.synchronize()
        ref = oracle_run(op, t, 1e-5, x_storage=STORAGE[combo[0]])
        compare_ex(op, got, ref, t["X"], tag=f"{op} {N}x{D} {_name(combo)} exchange")
    assert mt.mt_device_wait_errors(0) == 0


@pytest.mark.parametrize("op", OPS)
def test_wide_many_rows(op):
    """More rows than resident clusters: every cluster of the persistent backward runs
    several rows and its partial row sums them; LayerNorm with a large mean."""
    N, D = 300, 32768
    t = _inputs(op, N, D, x_kind="shifted" if op == W.LAYERNORM else "normal")
    got = gpu_run_ex(op, t, 1e-5)
    torch.cuda.synchronize()
    ref = oracle_run(op, t, 1e-5, x_storage="f16")
    compare_ex(op, got, ref, t["X"], tag=f"{op} {N}x{D}")


@pytest.mark.parametrize("D", [40000, 131072])
def test_wide_layernorm_offset_rows(D):
    """fp32 rows with mean 1000 and standard deviation 0.1 through the streamed forward:
    the sum of squares minus the squared sum would lose every digit of the variance in
    fp32. rstd to the usual 1e-5, the saved mean to one fp32 rounding of |mean|, Y to the
    fp32 output tolerance. (The backward is not checked here: it takes x - mean with the
    fp32 mean the interface saves, which at |mean| / std = 1e4 moves x-hat by about
    ulp(1000) * rstd = 6e-4, beyond the fp32 tolerances.)"""
    N = 3
    t = _inputs(W.LAYERNORM, N, D, (F32, F32, F32))
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    t["X"] = 1000.0 + 0.1 * torch.randn(N, D, generator=g, device="cuda")
    got = gpu_run_ex(W.LAYERNORM, t, 1e-5)
    torch.cuda.synchronize()
    ref = oracle_run(W.LAYERNORM, t, 1e-5, x_storage="f32")
    check_rstd(got["rstd"], ref["rstd"], f"offset rows rstd {N}x{D}")
    mu, mref = f64(got["mean"]), f64(ref["mean"])
    assert np.all(np.abs(mu - mref) <= 2.0 ** -23 * np.abs(mref)), (mu - mref)
    check_out(got["Y"], ref["Y"], F32, f"offset rows Y {N}x{D}")


def test_wide_fused_without_residual_cotangent():
    N, D = 9, 49152
    t = _inputs(W.ADD_RMSNORM, N, D)
    got = gpu_run_ex(W.ADD_RMSNORM, t, 1e-6, use_ds=False)
    ref = oracle_run(W.ADD_RMSNORM, t, 1e-6, use_ds=False, x_storage="f16")
    compare_ex(W.ADD_RMSNORM, got, ref, t["X"], tag="add noDS wide")


def test_wide_misaligned_rows():
    """Row bases one element off 16 bytes at a width the vector kernels could take: the
    split scalar kernels, same results."""
    N, D = 5, 32768
    t = _inputs(W.LAYERNORM, N, D)
    buf = torch.empty(N * D + 1, dtype=F16, device="cuda")
    xs = buf[1:].view(N, D)
    xs.copy_(t["X"])
    got = gpu_run_ex(W.LAYERNORM, dict(t, X=xs), 1e-5)
    ref = oracle_run(W.LAYERNORM, t, 1e-5, x_storage="f16")
    compare_ex(W.LAYERNORM, got, ref, t["X"], tag="misaligned wide")


@pytest.mark.parametrize("op", OPS)
def test_wide_deterministic(op):
    N, D = 200, 65536
    t = _inputs(op, N, D)
    a = gpu_run_ex(op, t, 1e-5)
    b = gpu_run_ex(op, t, 1e-5)
    for k in a:
        assert torch.equal(a[k], b[k]), k


def test_wide_full_size_sampled():
    """RMSNorm 4096 x 32768 (the wide-row bench workload): sampled rows of Y and dX
    against the oracle, dgamma through its definition on a column sample."""
    w = W.WORKLOADS["rmsnorm_4096x32768"]
    N, D = w.N, w.D
    t = W.generate_workload(w.name, device="cuda")
    got = gpu_run_ex(W.RMSNORM, t, w.eps)
    rows = torch.as_tensor([0, 1, 1000, 2047, 4095], device="cuda")
    sub = {k: v[rows] if v.dim() == 2 else v for k, v in t.items()}
    ref = oracle_run(W.RMSNORM, sub, w.eps, x_storage="f16")
    check_out(got["Y"][rows], ref["Y"], F16, "Y rows")
    check_out(got["dX"][rows], ref["dX"], F16, "dX rows")
    cols = torch.as_tensor([0, 7, 16383, 16384, 30000, D - 1], device="cuda")
    x, dy = f64(t["X"][:, cols]), f64(t["dY"][:, cols])
    r = f64(got["rstd"])[:, None]
    want = (dy * x * r).sum(axis=0)
    tol = 1e-4 * np.abs(dy * x * r).sum(axis=0) + 1e-7
    assert np.all(np.abs(f64(got["dgamma"][cols]) - want) <= tol)


# ------------------------------------------------------------------ N = 0 ---

@pytest.mark.parametrize("D", [64, 4096, 40000])
@pytest.mark.parametrize("op", OPS)
def test_empty_batch(op, D):
    """N = 0: the forward returns without touching anything; the backward sets the
    parameter gradients to the empty sum, 0, and needs no workspace."""
    t = _inputs(op, 0, D)
    assert t["X"].shape == (0, D)
    code = {W.RMSNORM: mt.MT_OP_RMSNORM, W.LAYERNORM: mt.MT_OP_LAYERNORM,
            W.ADD_RMSNORM: mt.MT_OP_ADD_RMSNORM}[op]
    assert mt.mt_norm_backward_workspace_size(code, 0, D, 0) == 0
    got = gpu_run_ex(op, t, 1e-5)
    torch.cuda.synchronize()
    assert got["Y"].shape == (0, D) and got["dX"].shape == (0, D)
    assert torch.count_nonzero(got["dgamma"]).item() == 0
    if op == W.LAYERNORM:
        assert torch.count_nonzero(got["dbeta"]).item() == 0
    # the fp16 entry points, dgamma first filled with NaN
    x = torch.empty((0, D), dtype=F16, device="cuda")
    g = torch.ones(D, dtype=F16, device="cuda")
    dg = torch.full((D,), float("nan"), device="cuda")
    r = torch.empty(0, device="cuda")
    mt.mt_rmsnorm_backward(x, g, x, r, x, dg, 0, D)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dg).item() == 0


def test_empty_batch_softmax_and_cross_entropy():
    x = torch.empty((0, 1000), dtype=BF16, device="cuda")
    assert mt.softmax_forward(x).shape == (0, 1000)
    t = torch.empty(0, dtype=torch.int64, device="cuda")
    for red in ("sum", "mean"):
        loss, lse, nv = mt.cross_entropy_forward(x, t, -100, 0.1, 1e-4, red)
        assert loss.item() == 0.0 and nv.item() == 0.0 and lse.shape == (0,)
        dx = mt.cross_entropy_backward(x, t, lse, torch.ones(1, device="cuda"), nv, reduction=red)
        assert dx.shape == (0, 1000)
