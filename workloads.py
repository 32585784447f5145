"""Seeded synthetic workloads for row-wise normalization (inputs only).

This module draws the inputs that both the CUDA path and the fp64 oracle are fed.
It holds none of the normalization arithmetic: only shapes, distributions, the
seed and the draw order, plus the byte accounting used to express throughput.

Every tensor is drawn from ONE seeded torch generator in the fixed order
X, R, s_row, gamma, beta, dY, dS (absent entries are skipped), as fp32, then
rounded to its storage type (round-to-nearest-even; fp16 unless a call asks for
bf16 or fp32 per role) before either side sees it. ``N(m, s)`` means mean m and
standard deviation s.

The seven workloads (name: op, N x D, recipe):
  rmsnorm_17x257        RMSNorm, ragged width. X, dY ~ N(0,1); gamma = 1 + 0.1 N(0,1); eps 1e-6.
  layernorm_128x1024    LayerNorm. X, dY ~ N(0,1); gamma = 1 + 0.1 N(0,1);
                        beta = 0.1 N(0,1); eps 1e-5.
  rmsnorm_16384x4096    RMSNorm at the Llama-7B activation shape (batch 4 x seq 4096,
                        hidden 4096). X = N(0,1) * s_row, s_row ~ U(0.5, 4) per row;
                        dY ~ N(0, 0.01); gamma = 1 + 0.1 N(0,1); eps 1e-6.
  add_rmsnorm_32768x4096  fused residual-add + RMSNorm. X, R ~ N(0,1); dY, dS ~ N(0, 0.01);
                        gamma = 1 + 0.1 N(0,1); eps 1e-6.
  layernorm_2048x16384  wide-row LayerNorm with a large mean (cancellation stress).
                        X = 50 + N(0,1); gamma = 1 + 0.1 N(0,1); beta = N(0, 0.1);
                        dY ~ N(0, 0.01); eps 1e-5.
  rmsnorm_4096x32768    RMSNorm on rows wider than one CTA's slice (a cluster of 2 CTAs per
                        row); the rmsnorm_16384x4096 recipe.
  layernorm_1024x131072 LayerNorm at the widest supported row (a cluster of 8 CTAs per
                        row). X, dY ~ N(0,1) and N(0, 0.01); gamma = 1 + 0.1 N(0,1);
                        beta = N(0, 0.1); eps 1e-5.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

RMSNORM = "rmsnorm"
LAYERNORM = "layernorm"
ADD_RMSNORM = "add_rmsnorm"
OPS = (RMSNORM, LAYERNORM, ADD_RMSNORM)


@dataclass(frozen=True)
class Workload:
    name: str
    op: str
    N: int
    D: int
    eps: float
    x_kind: str          # "normal", "row_scaled", "shifted"
    dy_std: float
    beta_std: float = 0.0  # LayerNorm only

    @property
    def shape(self) -> tuple[int, int]:
        return (self.N, self.D)


WORKLOADS = {
    w.name: w
    for w in (
        Workload("rmsnorm_17x257", RMSNORM, 17, 257, 1e-6, "normal", 1.0),
        Workload("layernorm_128x1024", LAYERNORM, 128, 1024, 1e-5, "normal", 1.0, beta_std=0.1),
        Workload("rmsnorm_16384x4096", RMSNORM, 16384, 4096, 1e-6, "row_scaled", 0.01),
        Workload("add_rmsnorm_32768x4096", ADD_RMSNORM, 32768, 4096, 1e-6, "normal", 0.01),
        Workload("layernorm_2048x16384", LAYERNORM, 2048, 16384, 1e-5, "shifted", 0.01,
                 beta_std=0.1),
        Workload("rmsnorm_4096x32768", RMSNORM, 4096, 32768, 1e-6, "row_scaled", 0.01),
        Workload("layernorm_1024x131072", LAYERNORM, 1024, 131072, 1e-5, "normal", 0.01,
                 beta_std=0.1),
    )
}
WORKLOAD_ORDER = list(WORKLOADS)


def make_generator(device, seed: int = 0) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(seed)
    return g


def generate(op: str, N: int, D: int, *, device="cpu", seed: int = 0,
             x_kind: str = "normal", dy_std: float = 1.0, beta_std: float = 0.1,
             with_ds: bool = True, x_dtype=torch.float16, w_dtype=torch.float16,
             g_dtype=torch.float16) -> dict[str, torch.Tensor]:
    """Draw one op's inputs on ``device``: X and R stored as ``x_dtype``, gamma and beta as
    ``w_dtype``, dY and dS as ``g_dtype`` (fp16, bf16 or fp32; the draws do not depend on
    the types).

    Returns a dict with X, gamma, dY and, by op: R and dS (fused add), beta (LayerNorm).
    ``with_ds=False`` leaves out dS for the fused op (the absent-cotangent case).
    """
    if op not in OPS:
        raise ValueError(f"unknown op {op!r}")
    dev = torch.device(device)
    g = make_generator(dev, seed)

    def normal(shape, mean=0.0, std=1.0):
        t = torch.randn(shape, generator=g, device=dev, dtype=torch.float32)
        if std != 1.0:
            t.mul_(std)
        if mean != 0.0:
            t.add_(mean)
        return t

    out: dict[str, torch.Tensor] = {}
    X = normal((N, D), mean=50.0 if x_kind == "shifted" else 0.0)
    R = normal((N, D)) if op == ADD_RMSNORM else None
    if x_kind == "row_scaled":
        s_row = torch.rand((N, 1), generator=g, device=dev, dtype=torch.float32)
        s_row.mul_(3.5).add_(0.5)          # U(0.5, 4)
        X.mul_(s_row)
    gamma = normal((D,), mean=1.0, std=0.1)
    beta = normal((D,), std=beta_std) if op == LAYERNORM else None
    dY = normal((N, D), std=dy_std)
    dS = normal((N, D), std=dy_std) if (op == ADD_RMSNORM and with_ds) else None

    out["X"] = X.to(x_dtype)
    if R is not None:
        out["R"] = R.to(x_dtype)
    out["gamma"] = gamma.to(w_dtype)
    if beta is not None:
        out["beta"] = beta.to(w_dtype)
    out["dY"] = dY.to(g_dtype)
    if dS is not None:
        out["dS"] = dS.to(g_dtype)
    return out


def generate_workload(name: str, *, device="cpu", seed: int = 0, rows: int | None = None,
                      with_ds: bool = True) -> dict[str, torch.Tensor]:
    """Draw a named workload's inputs; ``rows`` overrides N (same recipe, fewer rows)."""
    w = WORKLOADS[name]
    return generate(w.op, rows if rows is not None else w.N, w.D, device=device, seed=seed,
                    x_kind=w.x_kind, dy_std=w.dy_std, beta_std=w.beta_std, with_ds=with_ds)


def compulsory_bytes(op: str, direction: str, N: int, D: int, with_ds: bool = True,
                     xb: int = 2, wb: int = 2, gb: int = 2) -> int:
    """Bytes that any implementation must move: activations of xb bytes per element,
    parameters of wb, cotangents of gb (2 for fp16/bf16, 4 for fp32), fp32 statistics and
    parameter gradients. With the defaults (fp16 everywhere):

    forward:  RMSNorm 4ND + 4N + 2D; LayerNorm 4ND + 8N + 4D; fused add 8ND + 4N + 2D.
    backward: RMSNorm 6ND + 4N + 6D; LayerNorm 6ND + 8N + 10D; fused add 8ND + 4N + 6D
              (6ND + 4N + 6D when the residual-output cotangent is absent).
    Workspace traffic (dgamma/dbeta partials) is not compulsory.
    """
    nd = N * D
    if direction == "forward":
        return {RMSNORM: 2 * xb * nd + 4 * N + wb * D,
                LAYERNORM: 2 * xb * nd + 8 * N + 2 * wb * D,
                ADD_RMSNORM: 4 * xb * nd + 4 * N + wb * D}[op]
    if direction == "backward":
        if op == ADD_RMSNORM:
            return (2 * xb + (2 if with_ds else 1) * gb) * nd + 4 * N + (wb + 4) * D
        return {RMSNORM: (2 * xb + gb) * nd + 4 * N + (wb + 4) * D,
                LAYERNORM: (2 * xb + gb) * nd + 8 * N + (wb + 8) * D}[op]
    raise ValueError(direction)
