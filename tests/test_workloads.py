"""The seeded input generator: shapes, dtypes, recipes, determinism and byte accounting."""
import numpy as np
import pytest
import torch

import workloads as W


def test_seven_workloads():
    assert W.WORKLOAD_ORDER == ["rmsnorm_17x257", "layernorm_128x1024", "rmsnorm_16384x4096",
                                "add_rmsnorm_32768x4096", "layernorm_2048x16384",
                                "rmsnorm_4096x32768", "layernorm_1024x131072"]


@pytest.mark.parametrize("name", W.WORKLOAD_ORDER)
def test_shapes_and_dtypes(name):
    w = W.WORKLOADS[name]
    rows = min(w.N, 64)
    t = W.generate_workload(name, rows=rows)
    assert t["X"].shape == (rows, w.D) and t["X"].dtype == torch.float16
    assert t["gamma"].shape == (w.D,) and t["dY"].shape == (rows, w.D)
    assert ("R" in t) == ("dS" in t) == (w.op == W.ADD_RMSNORM)
    assert ("beta" in t) == (w.op == W.LAYERNORM)


def test_deterministic_and_seeded():
    a = W.generate_workload("rmsnorm_17x257")
    b = W.generate_workload("rmsnorm_17x257")
    c = W.generate_workload("rmsnorm_17x257", seed=1)
    assert torch.equal(a["X"], b["X"]) and torch.equal(a["dY"], b["dY"])
    assert not torch.equal(a["X"], c["X"])


def test_recipes():
    t = W.generate_workload("layernorm_2048x16384", rows=64)
    x = t["X"].double()
    assert abs(x.mean().item() - 50) < 0.05 and abs(x.std().item() - 1) < 0.05
    assert abs(t["dY"].double().std().item() - 0.01) < 0.001
    assert abs(t["beta"].double().std().item() - 0.1) < 0.02
    t = W.generate_workload("rmsnorm_16384x4096", rows=256)
    rs = t["X"].double().pow(2).mean(dim=1).sqrt()
    assert rs.min().item() > 0.45 and rs.max().item() < 4.1 and rs.std().item() > 0.5
    g = t["gamma"].double()
    assert abs(g.mean().item() - 1) < 0.01 and abs(g.std().item() - 0.1) < 0.01


def test_compulsory_bytes_match_published_accounting():
    # values of the byte formulas at the large shapes
    assert W.compulsory_bytes("rmsnorm", "forward", 16384, 4096) == 268_509_184
    assert W.compulsory_bytes("rmsnorm", "backward", 16384, 4096) == 402_743_296
    assert W.compulsory_bytes("add_rmsnorm", "forward", 32768, 4096) == 1_073_881_088
    assert W.compulsory_bytes("add_rmsnorm", "backward", 32768, 4096) == 1_073_897_472
    assert W.compulsory_bytes("layernorm", "forward", 2048, 16384) == 134_299_648
    assert W.compulsory_bytes("layernorm", "backward", 2048, 16384) == 201_506_816
