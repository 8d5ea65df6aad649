"""Block sharding across GPUs for the batched preconditioner step.

Every block of the (N, B, B) stack is independent through accumulate, scale,
root and apply, so a multi-GPU run needs no data exchange on the hot path: each
rank owns a contiguous range of blocks (factor j and its gradient block live on
the same rank) and works on it alone.  The only cross-rank traffic is timing:
the step time of a run is the slowest rank's, and throughput counts the blocks
of all ranks.  These helpers take a torch.distributed process group (any
backend) or run single-process when world size is 1.
"""

import torch


def block_range(n, rank, world):
    """Contiguous [start, stop) of the n blocks owned by `rank` of `world`;
    sizes differ by at most one, lower ranks take the extra blocks."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError("bad shard arguments n=%r rank=%r world=%r" % (n, rank, world))
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def _dist():
    import torch.distributed as dist

    return dist if dist.is_available() and dist.is_initialized() else None


def max_over_ranks(value, device="cpu"):
    """The largest `value` over all ranks (the step time of a data-parallel run)."""
    dist = _dist()
    if dist is None:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value, device="cpu"):
    dist = _dist()
    if dist is None:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def job_throughput(local_blocks, local_ms, device="cpu"):
    """Whole-job blocks per second: blocks of all ranks over the slowest rank's time."""
    total = sum_over_ranks(local_blocks, device)
    ms = max_over_ranks(local_ms, device)
    return total / (ms * 1e-3), ms
