"""The multi-rank layout of the estimator, on CPU with gloo (world size 2).

Sequences are independent and the noise is keyed by the global token index,
so ranks that each estimate their own slice of a batch (token offset
rank * T_rank, as bench.py gives them) reproduce the single-rank result: the
rows of g concatenate, and the per-rank weight gradients sum to the full one
through the same helper bench.py's multi-rank step calls after every
estimate (the step's one exchange).  The oracle stands in for the per-rank
compute; the point here is the layout and the reductions.
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


def _problem():
    rng = np.random.default_rng(5)
    T, V, d = 16, 24, 5
    x = rng.standard_normal((T, d)).astype(np.float32)
    z = rng.standard_normal((T, V)).astype(np.float32)
    y = rng.integers(0, V, T).astype(np.int32)
    return x, z, y


def _worker(rank, world, port, out_path):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    import oracle
    import activation_perturbation_es_noise_b300 as dust
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    x, z, y = _problem()
    T = z.shape[0] // world
    t0 = bench.rank_token0(rank, T)
    sl = slice(t0, t0 + T)
    res = oracle.head_estimate(z[sl], y[sl], x[sl], 0.05, 6, 1234, 0, 0, t0)
    g = torch.from_numpy(res["g"])
    gathered = [torch.empty_like(g) for _ in range(world)]
    dist.all_gather(gathered, g)
    G = torch.from_numpy(res["G"])
    dust.sum_over_ranks(G)
    slowest = bench.max_over_ranks(float(rank + 1), dist)
    if rank == 0:
        np.savez(out_path, g=torch.cat(gathered).numpy(), G=G.numpy(), slowest=slowest)
    dist.barrier()
    dist.destroy_process_group()


def test_two_ranks_reproduce_single_rank(tmp_path, orc):
    out = str(tmp_path / "r.npz")
    mp.start_processes(_worker, args=(2, _free_port(), out), nprocs=2, join=True,
                       start_method="spawn")
    r = np.load(out)
    x, z, y = _problem()
    full = orc.head_estimate(z, y, x, 0.05, 6, 1234, 0)
    np.testing.assert_allclose(r["g"], full["g"], rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(r["G"], full["G"], rtol=1e-12, atol=1e-12)
    assert float(r["slowest"]) == 2.0
