"""Multi-process (gloo, world size 2) checks of the block-sharded path on CPU:
the shards tile the stack exactly, the job timing takes the slowest rank, and
running the oracle step shard by shard gives the unsharded result (blocks are
independent, so no exchange is needed)."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from matrix_inverse_roots_gb300.shard import block_range, job_throughput, max_over_ranks


def free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, n, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle

        start, stop = block_range(n, rank, world)
        # Each rank runs the step on its own gradient blocks only.
        rng = np.random.default_rng(7)
        G = rng.standard_normal((n, 8, 8))
        Gs = G[start:stop]
        F = oracle.accumulate(np.zeros((2 * len(Gs), 8, 8)), Gs, 0.9)
        F += 1e-3 * np.eye(8)
        lam = oracle.power_lambda(F, np.ones((len(F), 8, 2)), 20)
        X, _, _ = oracle.cn_inv_root(F, lam, 12)
        U = oracle.apply_preconditioner(Gs, X)
        np.save(os.path.join(out_dir, "U%d.npy" % rank), U)
        # Timing: rank r pretends its step took 10 (r + 1) ms.
        thr, ms = job_throughput(2 * len(Gs), 10.0 * (rank + 1))
        mx = max_over_ranks(rank + 0.5)
        ranges = [None] * world
        dist.all_gather_object(ranges, (start, stop))
        with open(os.path.join(out_dir, "r%d.txt" % rank), "w") as f:
            f.write("%r %r %r %r\n" % (thr, ms, mx, ranges))
    finally:
        dist.destroy_process_group()


def test_block_range_partitions():
    for n in (0, 1, 5, 2496, 3815):
        for world in (1, 2, 3, 8):
            spans = [block_range(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            for a, b in zip(spans, spans[1:]):
                assert a[1] == b[0]
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        block_range(4, 2, 2)


def test_two_rank_gloo_sharded_step(tmp_path):
    n, world = 5, 2
    mp.spawn(_worker, args=(world, free_port(), n, str(tmp_path)), nprocs=world, join=True)
    import oracle

    rng = np.random.default_rng(7)
    G = rng.standard_normal((n, 8, 8))
    F = oracle.accumulate(np.zeros((2 * n, 8, 8)), G, 0.9) + 1e-3 * np.eye(8)
    lam = oracle.power_lambda(F, np.ones((2 * n, 8, 2)), 20)
    X, _, _ = oracle.cn_inv_root(F, lam, 12)
    U = oracle.apply_preconditioner(G, X)
    got = np.concatenate([np.load(tmp_path / ("U%d.npy" % r)) for r in range(world)])
    np.testing.assert_allclose(got, U, rtol=1e-12, atol=1e-12)
    for r in range(world):
        thr, ms, mx, ranges = open(tmp_path / ("r%d.txt" % r)).read().split(" ", 3)
        assert float(ms) == 20.0                       # slowest rank
        assert abs(float(thr) - 2 * n / 0.020) < 1e-6  # all blocks / slowest time
        assert float(mx) == 1.5
        assert eval(ranges) == [(0, 3), (3, 5)]
