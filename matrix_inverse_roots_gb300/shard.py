"""Block sharding across GPUs for the batched preconditioner step.

Every block of the (N, B, B) stack is independent through accumulate, scale,
root and apply, so the blocks are partitioned over the ranks: each rank owns a
contiguous range of gradient blocks, and with them the L and R factors of those
blocks.  In data-parallel training every rank computes a gradient for every
block from its own data, so the step has two exchanges (Distributed Shampoo's
assignment of blocks to workers, [pt] Definicao do Problema):
  * before accumulate, a reduce-scatter sums the ranks' gradients and leaves each
    rank with the summed gradient of the blocks it owns;
  * after apply, an all-gather gives every rank the preconditioned update U of
    every block.
DataParallelStep runs that exchange around a per-rank step on the owned blocks
(on the GPU, the library's accumulate / scale / root / apply).  The other
helpers partition the blocks and reduce timings: the step time of a run is the
slowest rank's, and throughput counts the blocks of all ranks.  Everything takes
the default torch.distributed process group (any backend) or runs
single-process when world size is 1.
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


def owned_range(n, rank, world):
    """(start, stop, chunk): the blocks [start, stop) rank owns when n blocks are
    cut into `world` equal chunks of ceil(n / world) (the last ranks may own fewer,
    or none); equal chunks let the exchanges use one reduce-scatter and one
    all-gather of uniform pieces."""
    if world < 1 or not 0 <= rank < world or n < 0:
        raise ValueError("bad shard arguments n=%r rank=%r world=%r" % (n, rank, world))
    chunk = -(-n // world)
    start = min(n, rank * chunk)
    return start, min(n, start + chunk), chunk


class DataParallelStep:
    """One data-parallel preconditioner step over the default process group.

    local_step(G_owned) -> U_owned computes the hot path on this rank's owned
    gradient blocks G_owned (n_own, B, B) and returns their updates (n_own, B, B).
    Calling the object with this rank's gradients of all ng blocks returns U of all
    ng blocks:
      1. reduce-scatter (sum) of the ranks' (ng, B, B) gradient stacks: this rank
         receives the summed gradients of its owned blocks -- the gradient of a
         loss summed over the global batch (scale the local gradients by 1/world
         beforehand for the mean);
      2. local_step on them;
      3. all-gather of the owned updates into (ng, B, B).
    u_dtype is the dtype of the updates every rank gathers.
    Stacks whose block count is not a multiple of world are padded with zero
    blocks for the exchanges (padding is never passed to local_step).  The returned
    stack is a view of a buffer the next call overwrites."""

    def __init__(self, ng, local_step, u_dtype=torch.float32):
        dist = _dist()
        self.world = dist.get_world_size() if dist is not None else 1
        self.rank = dist.get_rank() if dist is not None else 0
        self.ng = int(ng)
        self.start, self.stop, self.chunk = owned_range(self.ng, self.rank, self.world)
        self.local_step = local_step
        # Every rank must all-gather pieces of one dtype, also a rank owning none.
        self.u_dtype = u_dtype
        self._gpad = None
        self._gown = None
        self._upad = None
        self._uall = None

    def __call__(self, G):
        dist = _dist()
        ng, world, chunk = self.ng, self.world, self.chunk
        if G.shape[0] != ng:
            raise ValueError("expected %d gradient blocks, got %d" % (ng, G.shape[0]))
        n_own = self.stop - self.start
        if dist is None or world == 1:
            return self.local_step(G)
        shape = (chunk,) + tuple(G.shape[1:])
        if world * chunk != ng:
            if self._gpad is None or self._gpad.dtype != G.dtype or self._gpad.device != G.device:
                self._gpad = torch.zeros((world * chunk,) + shape[1:], dtype=G.dtype,
                                         device=G.device)
            self._gpad[:ng].copy_(G)
            src = self._gpad
        else:
            src = G
        if (self._gown is None or self._gown.dtype != G.dtype or self._gown.device != G.device
                or tuple(self._gown.shape) != shape):
            self._gown = torch.empty(shape, dtype=G.dtype, device=G.device)
        G_own = self._gown
        dist.reduce_scatter_tensor(G_own, src, op=dist.ReduceOp.SUM)
        U_own = self.local_step(G_own[:n_own]) if n_own > 0 else None
        if U_own is not None and n_own == chunk and U_own.dtype == self.u_dtype:
            upiece = U_own.contiguous()
        else:
            dt = self.u_dtype
            if self._upad is None or self._upad.device != G.device:
                self._upad = torch.zeros(shape, dtype=dt, device=G.device)
            if n_own > 0:
                self._upad[:n_own].copy_(U_own)
            upiece = self._upad
        if (self._uall is None or self._uall.dtype != upiece.dtype
                or self._uall.device != upiece.device):
            self._uall = torch.empty((world * chunk,) + shape[1:], dtype=upiece.dtype,
                                     device=upiece.device)
        dist.all_gather_into_tensor(self._uall, upiece)
        return self._uall[:ng]
