"""Row softmax / log-softmax and per-row cross-entropy on the GPU against the fp64 oracle
(tensorcore "Training kernels", "Softmax -- standalone, row-wise"; meTile reduction and
loss checklists; "Metal subgroup LayerNorm and cross-entropy report", cross-entropy).

Inputs are seeded and synthetic: softmax rows N(0, 3^2) (peaked rows), cotangents N(0, 1);
logits N(0, 2^2) with uniform random targets and a few ignored rows. Shapes: the report's
cross-entropy shapes (1x127, 17x257, 128x1024, 64x4096), ragged widths for the scalar
paths, and rows up to the 262144-column bound for both softmax and cross-entropy.

Tolerances: softmax outputs and gradients use the storage type's output tolerance
(parity.OUT_TOL); cross-entropy losses and lse (fp32, computed from the stored logits)
|err| <= 1e-5 (1 + |ref|): the fp32 running sums of exp carry about
(elements per thread + log2 threads) * 2^-24 relative error and __expf about 2^-21, so
the log of the sum is good to a few 1e-6; reduced losses 1e-5 of sum_i |loss_i|; logit
gradients rtol * |ref| + atol * max_j |ref_ij| per row with the storage type's (atol,
rtol), since most entries are tiny probabilities next to the target's O(1) entry.
"""
import numpy as np
import pytest
import torch

import oracle
import row_wise_rmsnorm_gb300 as mt
from parity import OUT_TOL, check_out, f64

pytestmark = pytest.mark.gpu

F16, BF16, F32 = torch.float16, torch.bfloat16, torch.float32
DTYPES = [F16, BF16, F32]
NAMES = {F16: "f16", BF16: "bf16", F32: "f32"}


def _gen(shape, std, dtype, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    return (torch.randn(shape, generator=g, device="cuda") * std).to(dtype)


# -------------------------------------------------------------------- softmax ---

# up to 16384 columns the row stays in registers; wider rows (to the meTile bound of
# 262144) take the two-pass streaming kernels: one CTA per row, except the backward of
# rows wider than 65536, split over a cluster (65544 and 131072: 4 CTAs, 262144: 8); a
# ragged width on the scalar path
SM_SHAPES = [(1, 127), (17, 257), (96, 1024), (40, 4104), (9, 16384), (300, 64),
             (4, 16392), (6, 65536), (3, 65544), (5, 50001), (3, 131072), (2, 262144)]


@pytest.mark.parametrize("log", [False, True], ids=["softmax", "log_softmax"])
@pytest.mark.parametrize("shape", SM_SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("dtype", DTYPES, ids=lambda d: NAMES[d])
def test_softmax_parity(dtype, shape, log):
    N, D = shape
    x = _gen((N, D), 3.0, dtype, 1)
    dy = _gen((N, D), 1.0, dtype, 2)
    y = mt.softmax_forward(x, log)
    dx = mt.softmax_backward(y, dy, log)
    torch.cuda.synchronize()
    Y = oracle.softmax_forward(f64(x), log)
    check_out(y, Y, dtype, f"softmax(log={log}) Y {NAMES[dtype]} {N}x{D}")
    # the backward is checked from the GPU's own stored Y (its input)
    dX = oracle.softmax_backward(f64(y), f64(dy), log)
    check_out(dx, dX, dtype, f"softmax(log={log}) dX {NAMES[dtype]} {N}x{D}")
    if not log:
        s = f64(y).sum(axis=1)
        assert np.all(np.abs(s - 1.0) <= D * OUT_TOL[dtype][0] + 1e-6), "rows sum to one"


@pytest.mark.parametrize("D", [4096, 65536, 262144])
def test_softmax_masked_columns(D):
    """-inf logits (masked columns), a row whose maximum is its last element, and a
    row whose first columns are all masked: the running maximum starts at -inf and
    masked entries come out as exactly 0."""
    N = 3
    x = _gen((N, D), 3.0, F32, 6)
    x[0, ::3] = float("-inf")
    x[1, -1] = 40.0
    x[2, : D // 2] = float("-inf")
    for log in (False, True):
        y = mt.softmax_forward(x, log)
        torch.cuda.synchronize()
        Y, got = oracle.softmax_forward(f64(x), log), f64(y)
        fin = np.isfinite(Y)   # log-softmax of a masked column is -inf on both sides
        assert np.array_equal(np.isfinite(got), fin) and np.all(got[~fin] == -np.inf)
        check_out(got[fin], Y[fin], F32, f"masked softmax(log={log}) {D}")
        if not log:
            assert torch.all(y[0, ::3] == 0) and torch.all(y[2, : D // 2] == 0)


@pytest.mark.parametrize("D", [1024, 40000, 70000], ids=["regs", "stream", "stream_split"])
def test_softmax_misaligned_and_deterministic(D):
    N = 33 if D <= 16384 else 3
    x = _gen((N, D), 3.0, F16, 4)
    buf = torch.empty(N * D + 1, dtype=F16, device="cuda")
    xs = buf[1:].view(N, D)
    xs.copy_(x)
    a = mt.softmax_forward(xs)
    b = mt.softmax_forward(x)
    check_out(a, oracle.softmax_forward(f64(x)), F16, "misaligned softmax")
    assert torch.equal(mt.softmax_forward(x), b), "softmax not deterministic"
    dy = _gen((N, D), 1.0, F16, 5)
    dys = torch.empty(N * D + 1, dtype=F16, device="cuda")[1:].view(N, D)
    dys.copy_(dy)
    ys = torch.empty(N * D + 1, dtype=F16, device="cuda")[1:].view(N, D)
    ys.copy_(a)
    g = mt.softmax_backward(ys, dys)
    check_out(g, oracle.softmax_backward(f64(a), f64(dy)), F16, "misaligned softmax backward")
    assert torch.equal(mt.softmax_backward(a, dy), mt.softmax_backward(a, dy)), \
        "softmax backward not deterministic"


# -------------------------------------------------------------- cross-entropy ---

CE_SHAPES = [(1, 127), (17, 257), (128, 1024), (64, 4096), (8, 32768), (5, 50001),
             (3, 131072), (2, 262144)]


def _targets(N, D, seed, ignore=(-100,)):
    rng = np.random.default_rng(seed)
    t = rng.integers(0, D, N)
    if N >= 4:
        t[1] = ignore[0]
    return torch.tensor(t, dtype=torch.int64, device="cuda")


def _check_rows(got, ref, what):
    """Per-row fp32 values (losses, lse): |err| <= 1e-5 (1 + |ref|); NaN where ref is NaN."""
    g = f64(got)
    assert np.array_equal(np.isnan(g), np.isnan(ref)), f"{what}: NaN positions"
    m = ~np.isnan(ref)
    assert np.all(np.abs(g[m] - ref[m]) <= 1e-5 * (1 + np.abs(ref[m]))), (
        f"{what}: max err {np.max(np.abs(g[m] - ref[m])):.3e}")


def _check_grad(got, ref, dtype, what):
    atol, rtol = OUT_TOL[dtype]
    g, r = f64(got), f64(ref)
    scale = np.max(np.abs(r), axis=1, keepdims=True)
    bad = ~(np.abs(g - r) <= rtol * np.abs(r) + atol * scale + 1e-30)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} out of tolerance, max err "
                           f"{np.max(np.abs(g - r)):.3e}")


@pytest.mark.parametrize("opts", [(0.0, 0.0, "none"), (0.1, 0.0, "mean"), (0.0, 1e-4, "sum"),
                                  (0.05, 1e-3, "mean")], ids=lambda o: f"ls{o[0]}-z{o[1]}-{o[2]}")
@pytest.mark.parametrize("shape", CE_SHAPES, ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("dtype", DTYPES, ids=lambda d: NAMES[d])
def test_cross_entropy_parity(dtype, shape, opts):
    eps, z, red = opts
    N, D = shape
    x = _gen((N, D), 2.0, dtype, 3)
    t = _targets(N, D, 5)
    loss, lse, nv = mt.cross_entropy_forward(x, t, -100, eps, z, red)
    rng = np.random.default_rng(6)
    up = rng.standard_normal(N) if red == "none" else np.array([1.3])
    dloss = torch.tensor(up, dtype=torch.float32, device="cuda")
    dx = mt.cross_entropy_backward(x, t, lse, dloss, nv, -100, eps, z, red)
    torch.cuda.synchronize()
    X = f64(x)
    T = t.cpu().numpy()
    rows, ref_lse = oracle.cross_entropy_forward(X, T, -100, eps, z)
    val, n_valid = oracle.cross_entropy_reduce(rows, T, -100, red)
    tag = f"ce {NAMES[dtype]} {N}x{D} {opts}"
    _check_rows(lse, ref_lse, tag + " lse")
    if red == "none":
        _check_rows(loss, rows, tag + " loss rows")
    else:
        tol = 1e-5 * np.sum(np.abs(rows)) + 1e-6
        assert abs(float(loss.item()) - val) <= tol, f"{tag}: reduced loss {loss.item()} vs {val}"
        assert float(nv.item()) == n_valid, f"{tag}: n_valid"
    g = oracle.cross_entropy_row_grad(up, N, n_valid, red)
    ref_dx = oracle.cross_entropy_backward(X, T, f64(lse), g, -100, eps, z)
    _check_grad(dx, ref_dx, dtype, tag + " dlogits")


def test_cross_entropy_edge_cases():
    """All rows ignored (mean = 0, gradient 0), an out-of-range target (NaN in its row
    only), a custom ignore index, and bitwise determinism of the reduced loss."""
    N, D = 6, 1000
    x = _gen((N, D), 2.0, F32, 7)
    t = torch.full((N,), 7, dtype=torch.int64, device="cuda")
    loss, lse, nv = mt.cross_entropy_forward(x, t, 7, 0.0, 0.0, "mean")
    dx = mt.cross_entropy_backward(x, t, lse, torch.ones(1, device="cuda"), nv, 7, 0.0, 0.0, "mean")
    assert loss.item() == 0.0 and nv.item() == 0.0 and torch.count_nonzero(dx).item() == 0
    t = torch.tensor([3, D + 5, 2, -1, 9, 0], dtype=torch.int64, device="cuda")
    rows, _, _ = mt.cross_entropy_forward(x, t, -1, 0.0, 0.0, "none")
    r = rows.cpu().numpy()
    assert np.isnan(r[1]) and r[3] == 0.0 and np.all(np.isfinite(r[[0, 2, 4, 5]]))
    x = _gen((4096, 4096), 2.0, BF16, 8)
    t = _targets(4096, 4096, 9)
    a = mt.cross_entropy_forward(x, t, -100, 0.1, 1e-4, "mean")
    b = mt.cross_entropy_forward(x, t, -100, 0.1, 1e-4, "mean")
    assert torch.equal(a[0], b[0]) and torch.equal(a[1], b[1])


def test_cross_entropy_count_past_fp32_integers():
    """More rows than fp32 counts exactly (2^24): the valid rows are counted as an integer,
    so n_valid is that count rounded once to fp32, and the mean is the fp32 sum divided by
    the exact count (rounded once); both reductions match the oracle."""
    N, D = (1 << 24) + 4100, 2
    x = _gen((N, D), 2.0, F16, 11)
    t = torch.zeros(N, dtype=torch.int64, device="cuda")
    t[1::65536] = -100
    count = N - int((t == -100).sum().item())
    assert count > (1 << 24) and count % 2 == 1  # not an fp32 integer
    mean, _, nv = mt.cross_entropy_forward(x, t, -100, 0.0, 0.0, "mean")
    tot, _, nv_sum = mt.cross_entropy_forward(x, t, -100, 0.0, 0.0, "sum")
    torch.cuda.synchronize()
    assert float(nv.item()) == float(np.float32(count)) == float(nv_sum.item())
    assert float(mean.item()) == float(np.float32(float(tot.item()) / count))
    rows, _ = oracle.cross_entropy_forward(f64(x), t.cpu().numpy(), -100, 0.0, 0.0)
    ref_sum, n_valid = oracle.cross_entropy_reduce(rows, t.cpu().numpy(), -100, "sum")
    assert n_valid == count
    tol = 1e-5 * np.sum(np.abs(rows))
    assert abs(float(tot.item()) - ref_sum) <= tol, f"sum {tot.item()} vs {ref_sum}"
    assert abs(float(mean.item()) - ref_sum / count) <= tol / count, f"mean {mean.item()}"


@pytest.mark.parametrize("shape", [(64, 4096), (17, 1001), (4, 50000)],
                         ids=lambda s: f"{s[0]}x{s[1]}")
@pytest.mark.parametrize("dtype", [BF16, F32], ids=lambda d: NAMES[d])
def test_cross_entropy_masked_columns(dtype, shape):
    """Logits of -inf (a masked vocabulary: a leading and a trailing block of columns) add
    nothing to the row's sum of exponentials, also where a thread's first logits are all
    masked; with label smoothing the loss is +inf (mass placed on impossible classes)."""
    N, D = shape
    x = _gen((N, D), 2.0, dtype, 11)
    lead, tail = D // 4, D // 8
    x[:, :lead] = float("-inf")
    x[:, D - tail:] = float("-inf")
    rng = np.random.default_rng(12)
    t = torch.tensor(rng.integers(lead, D - tail, N), dtype=torch.int64, device="cuda")
    loss, lse, nv = mt.cross_entropy_forward(x, t, -100, 0.0, 1e-4, "none")
    up = rng.standard_normal(N)
    dloss = torch.tensor(up, dtype=torch.float32, device="cuda")
    dx = mt.cross_entropy_backward(x, t, lse, dloss, nv, -100, 0.0, 1e-4, "none")
    torch.cuda.synchronize()
    X, T = f64(x), t.cpu().numpy()
    rows, ref_lse = oracle.cross_entropy_forward(X, T, -100, 0.0, 1e-4)
    _check_rows(lse, ref_lse, "masked lse")
    _check_rows(loss, rows, "masked loss")
    ref_dx = oracle.cross_entropy_backward(X, T, f64(lse), up, -100, 0.0, 1e-4)
    _check_grad(dx, ref_dx, dtype, "masked dlogits")
    assert torch.count_nonzero(dx[:, :lead]).item() == 0
    smooth, _, _ = mt.cross_entropy_forward(x, t, -100, 0.1, 0.0, "none")
    assert torch.all(torch.isposinf(smooth)).item()
