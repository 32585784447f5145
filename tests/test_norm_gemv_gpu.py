"""Fused normalization + GEMV for decode (tensorcore "Training kernels", "Fused Norm +
GEMV"): Y = Norm(X, gamma[, beta]) @ W on the GPU against the fp64 oracle, which applies
the normalized rows unrounded, as the fused kernels do.

Inputs are seeded and synthetic: X ~ N(0, 1) (LayerNorm also 50 + N(0, 1)), gamma =
1 + 0.1 N(0, 1), beta = 0.1 N(0, 1), W ~ N(0, 1/K) (a projection at its usual scale), all
fp16. Shapes: the decode batches M = 1..8 (the page tunes for M <= 4), ragged and aligned
N, K from 64 to the 32768 bound, and the bench shape M = 4, K = 4096, N = 12288 (a Llama-7B
fused QKV projection).

Tolerance: |y - ref| <= 1e-3 |ref| + 4e-5 sum_k |xn_k W_kn|. The fp16 output rounding is
2^-11 |ref| (4.9e-4); the fp32 sums run over at most a few hundred terms per thread before
fixed-order trees, about (K / 512 + 16) 2^-24 of the sum of absolute terms, under 4e-6 for
every K here, so the bound leaves a margin of ten.
"""
import numpy as np
import pytest
import torch

import oracle
import row_wise_rmsnorm_gb300 as mt
from parity import f64

pytestmark = pytest.mark.gpu

F16 = torch.float16


def _inputs(M, K, N, seed, shifted=False):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    x = torch.randn((M, K), generator=g, device="cuda") + (50.0 if shifted else 0.0)
    gamma = 1 + 0.1 * torch.randn(K, generator=g, device="cuda")
    beta = 0.1 * torch.randn(K, generator=g, device="cuda")
    w = torch.randn((K, N), generator=g, device="cuda") / np.sqrt(K)
    return x.to(F16), gamma.to(F16), beta.to(F16), w.to(F16)


def _check(y, ref, ref_abs, what):
    err = np.abs(f64(y) - ref)
    bound = 1e-3 * np.abs(ref) + 4e-5 * ref_abs + 1e-7
    bad = ~(err <= bound)
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} out of tolerance; worst "
                           f"err {err.max():.3e}")


def _run(op, x, gamma, beta, w, eps):
    return mt.norm_gemv(x, gamma, w, beta if op == "layernorm" else None, eps)


SHAPES = [(64, 8), (257, 100), (1024, 4096), (4096, 1000), (2048, 12288), (32768, 256),
          (32768, 4096)]


@pytest.mark.parametrize("KN", SHAPES, ids=lambda s: f"K{s[0]}-N{s[1]}")
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 8])
@pytest.mark.parametrize("op", ["rmsnorm", "layernorm"])
def test_norm_gemv_parity(op, M, KN):
    K, N = KN
    x, gamma, beta, w = _inputs(M, K, N, seed=M * 7 + K)
    y = _run(op, x, gamma, beta, w, 1e-5)
    torch.cuda.synchronize()
    ref, ref_abs = oracle.norm_gemv(op, f64(x), f64(gamma), f64(beta), f64(w), 1e-5)
    _check(y, ref, ref_abs, f"{op} M{M} K{K} N{N}")


def test_layernorm_gemv_large_mean():
    x, gamma, beta, w = _inputs(4, 4096, 2048, seed=3, shifted=True)
    y = _run("layernorm", x, gamma, beta, w, 1e-5)
    ref, ref_abs = oracle.norm_gemv("layernorm", f64(x), f64(gamma), f64(beta), f64(w), 1e-5)
    _check(y, ref, ref_abs, "layernorm gemv, mean 50")


@pytest.mark.parametrize("op", ["rmsnorm", "layernorm"])
def test_misaligned_weights(op):
    """W one element off 16 bytes (the per-element load path), same results."""
    M, K, N = 3, 512, 1024
    x, gamma, beta, w = _inputs(M, K, N, seed=9)
    buf = torch.empty(K * N + 1, dtype=F16, device="cuda")
    ws = buf[1:].view(K, N)
    ws.copy_(w)
    y = _run(op, x, gamma, beta, ws, 1e-5)
    ref, ref_abs = oracle.norm_gemv(op, f64(x), f64(gamma), f64(beta), f64(w), 1e-5)
    _check(y, ref, ref_abs, f"{op} misaligned W")


@pytest.mark.parametrize("op", ["rmsnorm", "layernorm"])
def test_deterministic(op):
    x, gamma, beta, w = _inputs(4, 4096, 12288, seed=11)
    a = _run(op, x, gamma, beta, w, 1e-5)
    b = _run(op, x, gamma, beta, w, 1e-5)
    assert torch.equal(a, b)


@pytest.mark.parametrize("op", ["rmsnorm", "layernorm"])
def test_against_the_separate_path(op):
    """The page validates the fused kernels against the separate norm forward + GEMM by the
    relative RMS of the difference (<= 5e-3). Here: this library's norm forward (fp16
    x_norm) followed by a torch fp32 matmul."""
    M, K, N = 4, 4096, 4096
    x, gamma, beta, w = _inputs(M, K, N, seed=13)
    y = _run(op, x, gamma, beta, w, 1e-5).float()
    if op == "rmsnorm":
        xn, _ = mt.rmsnorm_forward(x, gamma, 1e-5)
    else:
        xn, _, _ = mt.layernorm_forward(x, gamma, beta, 1e-5)
    sep = xn.float() @ w.float()
    rel = ((y - sep).pow(2).mean().sqrt() / sep.pow(2).mean().sqrt()).item()
    assert rel <= 5e-3, rel


def test_full_size_sampled():
    """M = 4, K = 4096, N = 12288 (the bench shape): sampled columns against the oracle."""
    M, K, N = 4, 4096, 12288
    x, gamma, beta, w = _inputs(M, K, N, seed=17)
    cols = np.array([0, 1, 7, 8, 255, 256, 4095, 6000, 12280, N - 1])
    for op in ("rmsnorm", "layernorm"):
        y = _run(op, x, gamma, beta, w, 1e-5)
        ref, ref_abs = oracle.norm_gemv(op, f64(x), f64(gamma), f64(beta),
                                        f64(w[:, torch.as_tensor(cols, device="cuda")]), 1e-5)
        _check(y[:, torch.as_tensor(cols, device="cuda")], ref, ref_abs, f"{op} sampled")


def test_empty_and_bounds():
    x, gamma, beta, w = _inputs(2, 64, 16, seed=1)
    e = torch.empty((0, 16), dtype=F16, device="cuda")
    mt.mt_fused_rmsnorm_gemv(None, None, None, None, 0, 16, 64, 1e-5)   # M = 0: no-op
    mt.mt_fused_layernorm_gemv(None, None, None, None, None, 2, 0, 64, 1e-5)  # N = 0
    assert e.shape == (0, 16)
    y = torch.empty((9, 16), dtype=F16, device="cuda")
    with pytest.raises(mt.MtNormError) as err:
        mt.mt_fused_rmsnorm_gemv(x, gamma, w, y, 9, 16, 64, 1e-5)
    assert err.value.status == mt.MT_ERR_UNSUPPORTED
