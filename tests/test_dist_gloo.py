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


class _OracleRankStep:
    """The hot path on the owned blocks, in float64 by the oracle: this rank's L and
    R factors persist across steps (the EMA)."""

    def __init__(self, n_own, b):
        self.F = np.zeros((2 * n_own, b, b))

    def __call__(self, G_own):
        import oracle

        G64 = G_own.double().numpy()
        self.F = oracle.accumulate(self.F, G64, 0.9)
        A = self.F + 1e-3 * np.eye(G64.shape[1])
        lam = oracle.power_lambda(A, np.ones((len(A), A.shape[1], 2)), 20)
        X, _, _ = oracle.cn_inv_root(A, lam, 12)
        return torch.from_numpy(oracle.apply_preconditioner(G64, X))


def _dp_worker(rank, world, port, ng, steps, out_dir):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        from matrix_inverse_roots_gb300.shard import DataParallelStep

        st = DataParallelStep(ng, None, u_dtype=torch.float64)
        st.local_step = _OracleRankStep(st.stop - st.start, 8)
        rng = np.random.default_rng(100 + rank)  # this rank's own data
        for k in range(steps):
            G = torch.from_numpy(rng.standard_normal((ng, 8, 8)))
            U = st(G)
            np.save(os.path.join(out_dir, "U%d_%d.npy" % (rank, k)), U.numpy())
        with open(os.path.join(out_dir, "own%d.txt" % rank), "w") as f:
            f.write("%d %d %d" % (st.start, st.stop, st.chunk))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("ng", [5, 1])
def test_two_rank_data_parallel_step_matches_unsharded(tmp_path, ng):
    """The reduce-scatter / local step / all-gather orchestration at world size 2,
    with a ragged split (ng = 5: 3 + 2 blocks) and a rank that owns nothing
    (ng = 1), over two steps (the owning rank's factors carry the EMA), against the
    unsharded oracle step on the summed gradients."""
    world, steps = 2, 2
    mp.spawn(_dp_worker, args=(world, free_port(), ng, steps, str(tmp_path)), nprocs=world,
             join=True)
    rngs = [np.random.default_rng(100 + r) for r in range(world)]
    ref = _OracleRankStep(ng, 8)
    for k in range(steps):
        Gsum = sum(r.standard_normal((ng, 8, 8)) for r in rngs)
        want = ref(torch.from_numpy(Gsum)).numpy()
        for r in range(world):
            got = np.load(tmp_path / ("U%d_%d.npy" % (r, k)))
            np.testing.assert_allclose(got, want, rtol=1e-10, atol=1e-12)
    own = [tuple(int(x) for x in open(tmp_path / ("own%d.txt" % r)).read().split())
           for r in range(world)]
    assert own == ([(0, 3, 3), (3, 5, 3)] if ng == 5 else [(0, 1, 1), (1, 1, 1)])


def test_owned_range_partitions():
    from matrix_inverse_roots_gb300.shard import owned_range

    for n in (0, 1, 5, 1248, 2496):
        for world in (1, 2, 3, 8):
            spans = [owned_range(n, r, world) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == n
            for a, b in zip(spans, spans[1:]):
                assert a[1] == b[0]
            assert all(s[1] - s[0] <= s[2] for s in spans)
