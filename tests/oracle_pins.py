"""Pins for the fp64 oracle: checks that tie it to something other than itself.

Each ``pin_*`` function takes a loaded oracle library handle and raises
AssertionError when the oracle disagrees with a fact fixed by the mathematics or
the pages (finite differences, closed forms, invariants, the meTile worked
example, torch's fp64 CPU layer_norm / rms_norm with autograd). They are plain
functions so that test_oracle_mutations.py can run them against deliberately
broken copies of the oracle and show that each plausible mistake is caught.
"""
from __future__ import annotations

import json
import os

import numpy as np

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _close(a, b, atol, rtol, what):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} vs {b.shape}"
    err = np.abs(a - b)
    bound = atol + rtol * np.abs(b)
    bad = ~(err <= bound)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} out of tolerance; "
                           f"max err {np.max(np.where(np.isnan(err), np.inf, err)):.3e}")


def _fd(loss, arr, h_rel=1e-6):
    """Central finite-difference gradient of the scalar loss() w.r.t. arr (in place)."""
    g = np.zeros_like(arr)
    for idx in np.ndindex(arr.shape):
        v = arr[idx]
        h = h_rel * max(1.0, abs(v))
        arr[idx] = v + h
        fp = loss()
        arr[idx] = v - h
        fm = loss()
        arr[idx] = v
        g[idx] = (fp - fm) / (2.0 * h)
    return g


# --------------------------------------------------------------------------- #
# Finite differences on 4 x 8 inputs: every backward formula.
# --------------------------------------------------------------------------- #
def pin_fd_rmsnorm(lib):
    rng = np.random.default_rng(11)
    X = rng.standard_normal((4, 8))
    gamma = 1.0 + 0.3 * rng.standard_normal(8)
    dY = rng.standard_normal((4, 8))
    eps = 1e-2  # large enough that a misplaced eps changes the derivative

    def loss():
        Y, _ = oracle.rmsnorm_forward(X, gamma, eps, lib=lib)
        return float(np.sum(dY * Y))

    _, rstd = oracle.rmsnorm_forward(X, gamma, eps, lib=lib)
    dX, dg, _ = oracle.rmsnorm_backward(X, gamma, dY, rstd, lib=lib)
    _close(dX, _fd(loss, X), 1e-7, 1e-6, "rms dX vs finite differences")
    _close(dg, _fd(loss, gamma), 1e-7, 1e-6, "rms dgamma vs finite differences")


def pin_fd_layernorm(lib):
    rng = np.random.default_rng(12)
    X = rng.standard_normal((4, 8)) + 0.7
    gamma = 1.0 + 0.3 * rng.standard_normal(8)
    beta = 0.5 * rng.standard_normal(8)
    dY = rng.standard_normal((4, 8))
    eps = 1e-2

    def loss():
        Y, _, _ = oracle.layernorm_forward(X, gamma, beta, eps, lib=lib)
        return float(np.sum(dY * Y))

    _, mean, rstd = oracle.layernorm_forward(X, gamma, beta, eps, lib=lib)
    dX, dg, db, _, _ = oracle.layernorm_backward(X, gamma, dY, mean, rstd, lib=lib)
    _close(dX, _fd(loss, X), 1e-7, 1e-6, "ln dX vs finite differences")
    _close(dg, _fd(loss, gamma), 1e-7, 1e-6, "ln dgamma vs finite differences")
    _close(db, _fd(loss, beta), 1e-7, 1e-6, "ln dbeta vs finite differences")


def pin_fd_add_rmsnorm(lib):
    # Dyadic inputs (multiples of 1/8 in [-4, 4]) so that S = X + R is exact in
    # fp16 and the saved-S backward equals the derivative of the real formula.
    rng = np.random.default_rng(13)
    X = rng.integers(-32, 33, size=(4, 8)) / 8.0
    R = rng.integers(-32, 33, size=(4, 8)) / 8.0
    gamma = 1.0 + 0.3 * rng.standard_normal(8)
    dY = rng.standard_normal((4, 8))
    dS = rng.standard_normal((4, 8))
    eps = 1e-2
    S16 = oracle.round_fp16(X + R).astype(np.float64)
    assert np.array_equal(S16, X + R)

    for cot in (dS, None):
        def loss():
            Y, S, _ = oracle.add_rmsnorm_forward(X, R, gamma, eps, lib=lib)
            total = float(np.sum(dY * Y))
            if cot is not None:
                total += float(np.sum(cot * S))
            return total

        _, S, rstd = oracle.add_rmsnorm_forward(X, R, gamma, eps, lib=lib)
        dX, dg, _ = oracle.add_rmsnorm_backward(S16, gamma, dY, cot, rstd, lib=lib)
        tag = "with dS" if cot is not None else "dS absent"
        _close(dX, _fd(loss, X), 1e-7, 1e-6, f"add dX ({tag}) vs finite differences")
        _close(dX, _fd(loss, R), 1e-7, 1e-6, f"add dR ({tag}) vs finite differences")
        _close(dg, _fd(loss, gamma), 1e-7, 1e-6, f"add dgamma ({tag}) vs finite differences")


# --------------------------------------------------------------------------- #
# Textbook library routine: torch fp64 CPU layer_norm / rms_norm + autograd.
# --------------------------------------------------------------------------- #
def pin_torch_fp64(lib):
    import torch
    import torch.nn.functional as F

    rng = np.random.default_rng(14)
    N, D = 17, 257
    X = oracle.round_fp16(rng.standard_normal((N, D))).astype(np.float64)
    R = oracle.round_fp16(rng.standard_normal((N, D))).astype(np.float64)
    gamma = oracle.round_fp16(1 + 0.1 * rng.standard_normal(D)).astype(np.float64)
    beta = oracle.round_fp16(0.1 * rng.standard_normal(D)).astype(np.float64)
    dY = oracle.round_fp16(rng.standard_normal((N, D))).astype(np.float64)
    dS = oracle.round_fp16(rng.standard_normal((N, D))).astype(np.float64)
    tight = dict(atol=1e-12, rtol=1e-10)

    def T(a):
        return torch.tensor(a, dtype=torch.float64, requires_grad=True)

    # RMSNorm
    eps = 1e-6
    x, w = T(X), T(gamma)
    y = F.rms_norm(x, (D,), weight=w, eps=eps)
    (y * torch.tensor(dY)).sum().backward()
    Y, rstd = oracle.rmsnorm_forward(X, gamma, eps, lib=lib)
    dX, dg, _ = oracle.rmsnorm_backward(X, gamma, dY, rstd, lib=lib)
    _close(Y, y.detach().numpy(), what="rms Y vs torch", **tight)
    _close(rstd, 1.0 / np.sqrt(np.mean(X * X, axis=1) + eps), what="rms rstd vs numpy", **tight)
    _close(dX, x.grad.numpy(), what="rms dX vs torch autograd", **tight)
    _close(dg, w.grad.numpy(), what="rms dgamma vs torch autograd", **tight)

    # LayerNorm
    eps = 1e-5
    x, w, b = T(X), T(gamma), T(beta)
    y = F.layer_norm(x, (D,), weight=w, bias=b, eps=eps)
    (y * torch.tensor(dY)).sum().backward()
    Y, mean, rstd = oracle.layernorm_forward(X, gamma, beta, eps, lib=lib)
    dX, dg, db, _, _ = oracle.layernorm_backward(X, gamma, dY, mean, rstd, lib=lib)
    _close(Y, y.detach().numpy(), what="ln Y vs torch", **tight)
    _close(mean, np.mean(X, axis=1), what="ln mean vs numpy", **tight)
    _close(rstd, 1.0 / np.sqrt(np.var(X, axis=1) + eps), what="ln rstd vs numpy", **tight)
    _close(dX, x.grad.numpy(), what="ln dX vs torch autograd", **tight)
    _close(dg, w.grad.numpy(), what="ln dgamma vs torch autograd", **tight)
    _close(db, b.grad.numpy(), what="ln dbeta vs torch autograd", **tight)

    # Fused residual add + RMSNorm: L = sum(dY * Y) + sum(dS * S), S = X + R.
    # With X + R not fp16-exact the saved-S backward differs from the exact-s
    # derivative by the fp16 rounding of S, so compare the exact-S backward here.
    eps = 1e-6
    x, r, w = T(X), T(R), T(gamma)
    s = x + r
    y = F.rms_norm(s, (D,), weight=w, eps=eps)
    ((y * torch.tensor(dY)).sum() + (s * torch.tensor(dS)).sum()).backward()
    Y, S, rstd = oracle.add_rmsnorm_forward(X, R, gamma, eps, lib=lib)
    _close(S, (X + R), atol=0.0, rtol=0.0, what="add S exact sum")
    dX, dg, _ = oracle.add_rmsnorm_backward(S, gamma, dY, dS, rstd, lib=lib)
    _close(Y, y.detach().numpy(), what="add Y vs torch", **tight)
    _close(dX, x.grad.numpy(), what="add dX vs torch autograd", **tight)
    _close(dX, r.grad.numpy(), what="add dR vs torch autograd", **tight)
    _close(dg, w.grad.numpy(), what="add dgamma vs torch autograd", **tight)


# --------------------------------------------------------------------------- #
# Closed forms and invariants.
# --------------------------------------------------------------------------- #
def pin_closed_forms(lib):
    rng = np.random.default_rng(15)
    X = rng.standard_normal((6, 33)) * np.array([0.01, 0.1, 1, 3, 10, 100])[:, None]
    D = X.shape[1]
    ones = np.ones(D)
    for eps in (1e-6, 1e-2, 1.0):
        # RMS with gamma = 1: mean(y^2) = ms / (ms + eps)
        Y, _ = oracle.rmsnorm_forward(X, ones, eps, lib=lib)
        ms = np.mean(X ** 2, axis=1)
        _close(np.mean(Y ** 2, axis=1), ms / (ms + eps), 1e-15, 1e-12, "rms mean(y^2)")
        # LN with gamma = 1, beta = 0: mean(y) = 0, mean(y^2) = var / (var + eps)
        Y, mean, rstd = oracle.layernorm_forward(X, ones, np.zeros(D), eps, lib=lib)
        var = np.var(X, axis=1)
        _close(np.mean(Y, axis=1), np.zeros(6), 1e-12, 0.0, "ln mean(y)")
        _close(np.mean(Y ** 2, axis=1), var / (var + eps), 1e-15, 1e-12, "ln mean(y^2)")


def pin_invariants(lib):
    rng = np.random.default_rng(16)
    N, D = 5, 24
    X = rng.standard_normal((N, D)) * 2.0 + 0.5
    gamma = 1 + 0.2 * rng.standard_normal(D)
    beta = 0.1 * rng.standard_normal(D)
    dY = rng.standard_normal((N, D))
    # eps = 0: RMS  sum_k dX_k x_k = 0; LN  sum_k dX_k = 0 and sum_k dX_k xhat_k = 0.
    _, rstd = oracle.rmsnorm_forward(X, gamma, 0.0, lib=lib)
    dX, _, _ = oracle.rmsnorm_backward(X, gamma, dY, rstd, lib=lib)
    _close(np.sum(dX * X, axis=1), np.zeros(N), 1e-11, 0, "rms sum(dX*x) at eps=0")
    _, mean, rstd = oracle.layernorm_forward(X, gamma, beta, 0.0, lib=lib)
    dX, _, _, _, _ = oracle.layernorm_backward(X, gamma, dY, mean, rstd, lib=lib)
    xhat = (X - np.mean(X, axis=1, keepdims=True)) / np.std(X, axis=1, keepdims=True)
    _close(np.sum(dX, axis=1), np.zeros(N), 1e-11, 0, "ln sum(dX) at eps=0")
    _close(np.sum(dX * xhat, axis=1), np.zeros(N), 1e-11, 0, "ln sum(dX*xhat) at eps=0")
    # eps > 0, LN: sum_k dX_k = 0 still holds.
    _, mean, rstd = oracle.layernorm_forward(X, gamma, beta, 0.3, lib=lib)
    dX, _, _, _, _ = oracle.layernorm_backward(X, gamma, dY, mean, rstd, lib=lib)
    _close(np.sum(dX, axis=1), np.zeros(N), 1e-11, 0, "ln sum(dX) at eps>0")
    # Fused op, dS only (dY = 0): dX = dS exactly, dgamma = 0.
    dS = rng.standard_normal((N, D))
    _, S, rstd = oracle.add_rmsnorm_forward(X, -0.5 * X, gamma, 1e-6, lib=lib)
    dX, dg, _ = oracle.add_rmsnorm_backward(S, gamma, np.zeros((N, D)), dS, rstd, lib=lib)
    _close(dX, dS, 0, 0, "add dX with dY = 0")
    _close(dg, np.zeros(D), 0, 0, "add dgamma with dY = 0")
    # dgamma_abs is the sum of |terms|: equal to dgamma when every term is >= 0.
    Xp = np.abs(X) + 0.1
    dYp = np.abs(dY) + 0.1
    _, rstd = oracle.rmsnorm_forward(Xp, gamma, 1e-6, lib=lib)
    _, dg, dga = oracle.rmsnorm_backward(Xp, gamma, dYp, rstd, lib=lib)
    _close(dga, dg, 0, 1e-15, "dgamma_abs for positive terms")
    _, rstd = oracle.rmsnorm_forward(X, gamma, 1e-6, lib=lib)
    _, dg, dga = oracle.rmsnorm_backward(X, gamma, dY, rstd, lib=lib)
    assert np.all(dga >= np.abs(dg)) and np.all(dga > 0), "dgamma_abs >= |dgamma|"
    _, mean, rstd = oracle.layernorm_forward(X, gamma, beta, 1e-5, lib=lib)
    _, _, db, _, dba = oracle.layernorm_backward(X, gamma, dY, mean, rstd, lib=lib)
    _close(dba, np.sum(np.abs(dY), axis=0), 0, 1e-14, "dbeta_abs = sum |dY|")
    _close(db, np.sum(dY, axis=0), 1e-14, 1e-14, "dbeta = column sums of dY")


def pin_worked_example(lib):
    """meTile contract's LayerNorm example (3 x 7, arange/10, unit weight, zero bias)."""
    with open(os.path.join(GOLDEN, "metile_layernorm_worked_example.json")) as f:
        fx = json.load(f)
    rows, cols, eps = fx["rows"], fx["cols"], fx["epsilon"]
    X = (np.arange(rows * cols, dtype=np.float32).reshape(rows, cols) / 10).astype(np.float64)
    Y, mean, rstd = oracle.layernorm_forward(X, np.ones(cols), np.zeros(cols), eps, lib=lib)
    assert Y.shape == X.shape
    expect_row = (np.arange(cols) - 3) * 0.1 / np.sqrt(0.04 + eps)
    _close(Y, np.tile(expect_row, (rows, 1)), 1e-6, 1e-6, "worked example Y")
    _close(mean, (7 * np.arange(rows) + 3) / 10.0, 1e-6, 0, "worked example mean")
    _close(rstd, np.full(rows, 1 / np.sqrt(0.04 + eps)), 0, 1e-5, "worked example rstd")
    dX, dg, db, _, _ = oracle.layernorm_backward(X, np.ones(cols), np.ones_like(X), mean, rstd,
                                                 lib=lib)
    assert dX.shape == X.shape and dg.shape == db.shape == (cols,)
    _close(dX, np.zeros_like(X), 1e-12, 0, "worked example dX = 0")
    _close(dg, 3 * expect_row, 1e-5, 1e-6, "worked example dgamma = 3 Y_0j")
    _close(db, np.full(cols, 3.0), 0, 0, "worked example dbeta = 3")


def pin_shift_and_scale(lib):
    rng = np.random.default_rng(17)
    N, D = 4, 64
    # fp16 values in [-1, 1) with at most 5 fraction bits, so X + 50 is exact in fp16.
    Z = rng.integers(-32, 32, size=(N, D)) / 32.0
    gamma = 1 + 0.1 * rng.standard_normal(D)
    beta = 0.1 * rng.standard_normal(D)
    dY = rng.standard_normal((N, D))
    assert np.array_equal(oracle.round_fp16(Z + 50).astype(np.float64), Z + 50)
    Y0, m0, r0 = oracle.layernorm_forward(Z, gamma, beta, 1e-5, lib=lib)
    Y1, m1, r1 = oracle.layernorm_forward(Z + 50, gamma, beta, 1e-5, lib=lib)
    _close(Y1, Y0, 1e-12, 1e-10, "ln shift invariance Y")
    _close(m1, m0 + 50, 1e-12, 0, "ln shift mean")
    _close(r1, r0, 0, 1e-10, "ln shift rstd")
    dX0, dg0, db0, _, _ = oracle.layernorm_backward(Z, gamma, dY, m0, r0, lib=lib)
    dX1, dg1, db1, _, _ = oracle.layernorm_backward(Z + 50, gamma, dY, m1, r1, lib=lib)
    _close(dX1, dX0, 1e-11, 1e-9, "ln shift invariance dX")
    _close(dg1, dg0, 1e-11, 1e-9, "ln shift invariance dgamma")
    _close(db1, db0, 0, 0, "ln shift invariance dbeta")
    # RMS at eps = 0: y(a x) = y(x), dX(a x) = dX(x) / a.
    X = rng.standard_normal((N, D))
    for a in (0.25, 3.0, 1000.0):
        Ya, ra = oracle.rmsnorm_forward(a * X, gamma, 0.0, lib=lib)
        Y1, r1 = oracle.rmsnorm_forward(X, gamma, 0.0, lib=lib)
        _close(Ya, Y1, 1e-12, 1e-10, "rms scale invariance Y")
        _close(ra, r1 / a, 0, 1e-12, "rms scale rstd")
        dXa, dga, _ = oracle.rmsnorm_backward(a * X, gamma, dY, ra, lib=lib)
        dX1, dg1, _ = oracle.rmsnorm_backward(X, gamma, dY, r1, lib=lib)
        _close(dXa, dX1 / a, 1e-12, 1e-9, "rms scale dX")
        _close(dga, dg1, 1e-12, 1e-10, "rms scale dgamma")


def pin_special_cases(lib):
    rng = np.random.default_rng(18)
    # D = 1
    X = rng.standard_normal((5, 1))
    gamma = np.array([1.3])
    beta = np.array([-0.4])
    dY = rng.standard_normal((5, 1))
    Y, mean, rstd = oracle.layernorm_forward(X, gamma, beta, 1e-5, lib=lib)
    _close(Y, np.full((5, 1), -0.4), 0, 1e-15, "ln D=1: y = beta")
    dX, _, _, _, _ = oracle.layernorm_backward(X, gamma, dY, mean, rstd, lib=lib)
    _close(dX, np.zeros((5, 1)), 1e-15, 0, "ln D=1: dX = 0")
    eps = 1e-3
    Y, rstd = oracle.rmsnorm_forward(X, gamma, eps, lib=lib)
    _close(Y, X / np.sqrt(X * X + eps) * 1.3, 0, 1e-14, "rms D=1")
    # constant row, LayerNorm: y = beta, dX = r (g - mean g)
    D = 16
    Xc = np.full((2, D), 3.25)
    gamma = 1 + 0.1 * rng.standard_normal(D)
    beta = rng.standard_normal(D)
    dY = rng.standard_normal((2, D))
    Y, mean, rstd = oracle.layernorm_forward(Xc, gamma, beta, 1e-5, lib=lib)
    _close(Y, np.tile(beta, (2, 1)), 0, 1e-15, "ln constant row: y = beta")
    _close(rstd, np.full(2, 1e-5 ** -0.5), 0, 1e-12, "ln constant row rstd")
    dX, _, _, _, _ = oracle.layernorm_backward(Xc, gamma, dY, mean, rstd, lib=lib)
    g = dY * gamma
    _close(dX, rstd[:, None] * (g - g.mean(axis=1, keepdims=True)), 1e-12, 1e-12,
           "ln constant row dX")
    # zero row, RMSNorm: y = 0, rstd = eps^-1/2
    Y, rstd = oracle.rmsnorm_forward(np.zeros((3, D)), gamma, 1e-6, lib=lib)
    _close(Y, np.zeros((3, D)), 0, 0, "rms zero row y")
    _close(rstd, np.full(3, 1e3), 0, 1e-12, "rms zero row rstd")


# --------------------------------------------------------------------------- #
# Row softmax and per-row cross-entropy.
# --------------------------------------------------------------------------- #
def pin_fd_softmax(lib):
    """Finite differences of L = sum dY * Y for softmax and log-softmax (4 x 8)."""
    rng = np.random.default_rng(21)
    X = 3.0 * rng.standard_normal((4, 8))
    dY = rng.standard_normal((4, 8))
    for log in (False, True):
        def loss():
            return float(np.sum(dY * oracle.softmax_forward(X, log, lib=lib)))
        Y = oracle.softmax_forward(X, log, lib=lib)
        dX = oracle.softmax_backward(Y, dY, log, lib=lib)
        _close(dX, _fd(loss, X), 1e-7, 1e-6, f"softmax(log={log}) dX vs finite differences")


def pin_fd_cross_entropy(lib):
    """Finite differences of L = sum_i g_i loss_i w.r.t. the logits, with label smoothing,
    z-loss and an ignored row (5 x 8)."""
    rng = np.random.default_rng(22)
    X = 2.0 * rng.standard_normal((5, 8))
    T = np.array([3, 0, -100, 7, 5])
    g = rng.standard_normal(5)
    for eps, z in ((0.0, 0.0), (0.1, 0.0), (0.0, 1e-2), (0.2, 3e-2)):
        def loss():
            l, _ = oracle.cross_entropy_forward(X, T, -100, eps, z, lib=lib)
            return float(np.sum(g * l))
        _, lse = oracle.cross_entropy_forward(X, T, -100, eps, z, lib=lib)
        dX = oracle.cross_entropy_backward(X, T, lse, g, -100, eps, z, lib=lib)
        _close(dX, _fd(loss, X), 1e-7, 1e-6, f"ce(eps={eps}, z={z}) dX vs finite differences")


def pin_torch_softmax_ce(lib):
    """torch's fp64 CPU softmax / log_softmax / cross_entropy (label smoothing, ignore
    index, none/sum/mean) with autograd; the z-loss term z * logsumexp^2 added in torch."""
    import torch
    import torch.nn.functional as F

    rng = np.random.default_rng(23)
    N, D = 17, 257
    X = 4.0 * rng.standard_normal((N, D))
    dY = rng.standard_normal((N, D))
    tight = dict(atol=1e-12, rtol=1e-10)
    for log in (False, True):
        x = torch.tensor(X, requires_grad=True)
        y = F.log_softmax(x, dim=1) if log else F.softmax(x, dim=1)
        (y * torch.tensor(dY)).sum().backward()
        Y = oracle.softmax_forward(X, log, lib=lib)
        _close(Y, y.detach().numpy(), what=f"softmax(log={log}) vs torch", **tight)
        _close(oracle.softmax_backward(Y, dY, log, lib=lib), x.grad.numpy(),
               what=f"softmax(log={log}) dX vs torch autograd", **tight)
    T = rng.integers(0, D, N)
    T[[2, 9]] = -100
    for eps, z, red in ((0.0, 0.0, "none"), (0.1, 0.0, "sum"), (0.05, 1e-3, "mean"),
                        (0.0, 1e-2, "mean")):
        x = torch.tensor(X, requires_grad=True)
        t = torch.tensor(T)
        ce = F.cross_entropy(x, t, reduction="none", ignore_index=-100, label_smoothing=eps)
        lse_t = torch.logsumexp(x, dim=1)
        rows = ce + z * lse_t ** 2 * (t != -100)
        valid = float((t != -100).sum())
        tot = rows if red == "none" else (rows.sum() if red == "sum" else rows.sum() / valid)
        up = rng.standard_normal(N) if red == "none" else np.array([1.7])
        (tot * torch.tensor(up if red == "none" else up[0])).sum().backward()
        loss, lse = oracle.cross_entropy_forward(X, T, -100, eps, z, lib=lib)
        val, nv = oracle.cross_entropy_reduce(loss, T, -100, red)
        _close(lse, lse_t.detach().numpy(), what="ce lse vs torch logsumexp", **tight)
        _close(val, tot.detach().numpy(), what=f"ce {red} loss vs torch", **tight)
        g = oracle.cross_entropy_row_grad(up, N, nv, red)
        dX = oracle.cross_entropy_backward(X, T, lse, g, -100, eps, z, lib=lib)
        _close(dX, x.grad.numpy(), what=f"ce {red} dX vs torch autograd", **tight)


def pin_softmax_ce_closed_forms(lib):
    """Uniform logits: softmax = 1/D, log-softmax = -log D, loss = log D + z log^2 D (any
    smoothing), gradient = (1 + 2 z log D)/D - q. Rows sum to one; a shifted row gives the
    same softmax; the gradient rows sum to 2 z lse g; the report's peak/total/selected
    formula on a row; an out-of-range target gives NaN and an ignored row 0."""
    D = 10
    X = np.full((2, D), 0.37)
    Y = oracle.softmax_forward(X, False, lib=lib)
    _close(Y, np.full((2, D), 1.0 / D), 0, 1e-15, "softmax of a constant row")
    _close(oracle.softmax_forward(X, True, lib=lib), np.full((2, D), -np.log(D)), 1e-15, 1e-15,
           "log-softmax of a constant row")
    z, eps = 0.02, 0.3
    loss, lse = oracle.cross_entropy_forward(X, [4, 0], -100, eps, z, lib=lib)
    ld = np.log(D) + 0.37
    _close(loss, np.full(2, np.log(D) + z * ld * ld), 1e-14, 1e-14, "ce of a constant row")
    g = np.array([1.0, -2.0])
    dX = oracle.cross_entropy_backward(X, [4, 0], lse, g, -100, eps, z, lib=lib)
    q = np.full((2, D), eps / D)
    q[0, 4] += 1 - eps
    q[1, 0] += 1 - eps
    want = g[:, None] * ((1 + 2 * z * ld) / D - q)
    _close(dX, want, 1e-14, 1e-13, "ce gradient of a constant row")
    rng = np.random.default_rng(24)
    X = 5.0 * rng.standard_normal((6, 33))
    Y = oracle.softmax_forward(X, False, lib=lib)
    _close(Y.sum(axis=1), np.ones(6), 1e-14, 0, "softmax rows sum to one")
    _close(oracle.softmax_forward(X + 11.5, False, lib=lib), Y, 1e-15, 1e-12, "softmax shift")
    _close(oracle.softmax_backward(Y, rng.standard_normal((6, 33)), False, lib=lib).sum(axis=1),
           np.zeros(6), 1e-14, 0, "softmax dX rows sum to zero")
    T = rng.integers(0, 33, 6)
    loss, lse = oracle.cross_entropy_forward(X, T, -100, 0.0, 0.0, lib=lib)
    peak = X.max(axis=1)
    total = np.exp(X - peak[:, None]).sum(axis=1)
    _close(loss, np.log(total) + peak - X[np.arange(6), T], 1e-13, 1e-13,
           "report formula log(total) + peak - selected")
    g = rng.standard_normal(6)
    dX = oracle.cross_entropy_backward(X, T, lse, g, -100, 0.1, 0.05, lib=lib)
    _, lse2 = oracle.cross_entropy_forward(X, T, -100, 0.1, 0.05, lib=lib)
    _close(dX.sum(axis=1), 2 * 0.05 * lse2 * g, 1e-12, 1e-12, "ce gradient rows sum")
    loss, _ = oracle.cross_entropy_forward(X[:2], [-100, 40], -100, 0.0, 0.0, lib=lib)
    assert loss[0] == 0.0 and np.isnan(loss[1]), "ignored row 0, out-of-range target NaN"
    val, nv = oracle.cross_entropy_reduce(np.zeros(3), [-100, -100, -100], -100, "mean")
    assert val == 0.0 and nv == 0.0, "mean over no valid row is 0"


def pin_norm_gemv_torch(lib):
    """torch's fp64 CPU rms_norm / layer_norm followed by a matmul (tensorcore "Fused Norm
    + GEMV": Y = Norm(X, gamma[, beta]) @ W, W [K, N]), M = 3, K = 40, N = 24, and the
    absolute-term sums against |xn| @ |W|."""
    import torch
    import torch.nn.functional as F

    rng = np.random.default_rng(31)
    M, K, N = 3, 40, 24
    X = rng.standard_normal((M, K)) + 2.0
    gamma = 1 + 0.1 * rng.standard_normal(K)
    beta = 0.1 * rng.standard_normal(K)
    W = rng.standard_normal((K, N))
    t = lambda a: torch.tensor(a, dtype=torch.float64)
    for op in ("rmsnorm", "layernorm"):
        if op == "rmsnorm":
            xn = F.rms_norm(t(X), (K,), weight=t(gamma), eps=1e-6)
        else:
            xn = F.layer_norm(t(X), (K,), weight=t(gamma), bias=t(beta), eps=1e-6)
        Y, Ya = oracle.norm_gemv(op, X, gamma, beta, W, 1e-6, lib=lib)
        _close(Y, (xn @ t(W)).numpy(), 1e-12, 1e-12, f"{op} gemv vs torch")
        _close(Ya, (xn.abs() @ t(W).abs()).numpy(), 1e-12, 1e-12, f"{op} gemv |terms|")


def pin_norm_gemv_closed_forms(lib):
    """A hand-worked case and structural checks of Y = Norm(X) @ W:
    * RMSNorm of x = [3, 4] (eps 0, gamma = [1, 2]) times W = [[1, 2], [3, 4]]:
      ms = 12.5, xn = [3, 8] / sqrt(12.5), Y = [27, 38] / sqrt(12.5);
    * a permutation matrix W (W[k, p(k)] = 1, p not an involution) moves feature k of the
      normalized row to output column p(k): Y[:, p(k)] = Norm(X)[:, k] (an operand
      transposition would apply p's inverse);
    * LayerNorm of constant rows normalizes to beta, so Y = beta @ W for every row."""
    Y, _ = oracle.norm_gemv("rmsnorm", [[3.0, 4.0]], [1.0, 2.0], None, [[1.0, 2.0], [3.0, 4.0]],
                            0.0, lib=lib)
    _close(Y, [[27 / np.sqrt(12.5), 38 / np.sqrt(12.5)]], 0, 1e-15, "hand-worked rmsnorm gemv")
    rng = np.random.default_rng(32)
    K = 7
    perm = np.array([1, 2, 3, 4, 5, 6, 0])            # a 7-cycle
    W = np.zeros((K, K))
    W[np.arange(K), perm] = 1.0
    X = rng.standard_normal((2, K))
    gamma = 1 + 0.1 * rng.standard_normal(K)
    beta = 0.1 * rng.standard_normal(K)
    for op in ("rmsnorm", "layernorm"):
        if op == "rmsnorm":
            xn, _ = oracle.rmsnorm_forward(X, gamma, 1e-5, lib=lib)
        else:
            xn, _, _ = oracle.layernorm_forward(X, gamma, beta, 1e-5, lib=lib)
        Y, _ = oracle.norm_gemv(op, X, gamma, beta, W, 1e-5, lib=lib)
        _close(Y[:, perm], xn, 0, 1e-15, f"{op} gemv with a permutation")
    Xc = np.full((3, K), 2.5)
    Wr = rng.standard_normal((K, 5))
    Y, _ = oracle.norm_gemv("layernorm", Xc, gamma, beta, Wr, 1e-5, lib=lib)
    _close(Y, np.tile(beta @ Wr, (3, 1)), 1e-15, 1e-13, "layernorm gemv of constant rows")


ALL_PINS = [
    pin_norm_gemv_torch,
    pin_norm_gemv_closed_forms,
    pin_fd_rmsnorm,
    pin_fd_layernorm,
    pin_fd_add_rmsnorm,
    pin_torch_fp64,
    pin_closed_forms,
    pin_invariants,
    pin_worked_example,
    pin_shift_and_scale,
    pin_special_cases,
    pin_fd_softmax,
    pin_fd_cross_entropy,
    pin_torch_softmax_ce,
    pin_softmax_ce_closed_forms,
]
