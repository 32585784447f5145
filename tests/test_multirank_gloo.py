"""The N > 1 host logic on CPU with two gloo ranks (no GPU).

* bench.max_over_ranks: every rank gets the slowest rank's step time.
* Row sharding: each rank normalises a contiguous block of rows (the oracle stands in
  for the per-rank kernel on CPU); dgamma/dbeta are combined in rank order. The result
  equals the unsharded computation (fp64, to rounding) and is identical on every rank,
  which is what a data-parallel deployment of the kernels needs from its combine.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out_dir):
    import sys
    for p in (ROOT, os.path.join(ROOT, "tests")):
        if p not in sys.path:
            sys.path.insert(0, p)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import oracle
    import workloads as W

    # slowest replica's time
    mx = bench.max_over_ranks(1.5 + rank)
    # row-sharded LayerNorm forward + backward, fixed rank-order combine of dgamma/dbeta
    t = W.generate_workload("layernorm_128x1024")
    X, g, b, dY = (t[k].double().numpy() for k in ("X", "gamma", "beta", "dY"))
    N = X.shape[0]
    lo, hi = rank * N // world, (rank + 1) * N // world
    _, mean, rstd = oracle.layernorm_forward(X[lo:hi], g, b, 1e-5)
    _, dg, db, _, _ = oracle.layernorm_backward(X[lo:hi], g, dY[lo:hi], mean, rstd)
    parts = [torch.zeros(2, X.shape[1], dtype=torch.float64) for _ in range(world)]
    dist.all_gather(parts, torch.tensor(np.stack([dg, db])))
    combined = parts[0].clone()
    for p in parts[1:]:  # ascending rank order
        combined += p
    np.save(os.path.join(out_dir, f"rank{rank}.npy"), np.concatenate([[mx], combined.numpy().ravel()]))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks(tmp_path):
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    r0 = np.load(tmp_path / "rank0.npy")
    r1 = np.load(tmp_path / "rank1.npy")
    assert r0[0] == r1[0] == 2.5  # max over ranks of 1.5 and 2.5
    assert np.array_equal(r0, r1)  # identical combine on every rank

    import oracle
    import workloads as W
    t = W.generate_workload("layernorm_128x1024")
    X, g, b, dY = (t[k].double().numpy() for k in ("X", "gamma", "beta", "dY"))
    _, mean, rstd = oracle.layernorm_forward(X, g, b, 1e-5)
    _, dg, db, dga, dba = oracle.layernorm_backward(X, g, dY, mean, rstd)
    combined = r0[1:].reshape(2, -1)
    assert np.all(np.abs(combined[0] - dg) <= 1e-12 * dga + 1e-15)
    assert np.all(np.abs(combined[1] - db) <= 1e-12 * dba + 1e-15)
