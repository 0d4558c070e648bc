"""Data parallelism over the minibatch for BlocksparseMatMul, one process per GPU.

The three passes shard naturally along the minibatch: with the weight W replicated on every
rank, rank r runs fprop and bprop on its own rows of x and dy (columns, for feature_axis 0) and
gets its rows of y and dx with no exchange; the weight gradient of the whole minibatch is the sum
over ranks of the gradients of their shards (updat sums over minibatch rows), so one all-reduce of
the float32 dW, nnz * bs * bs values, is the only collective.  (The kiteco/blocksparse page, "Kite
usage, read first", lists the library's own NCCL all-reduce op, allreduce_nccl, among its tests.)

Every compute step runs in the CUDA library (through the binding); this module only splits the
minibatch and calls torch.distributed for the sum.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_bounds(N: int, rank: int, world: int, align: int = 1):
    """[lo, hi): rank's contiguous share of N minibatch entries.  Shares differ by at most `align`
    entries and start on multiples of `align` (8 keeps a (C, N) row pitch of 16-bit values a
    multiple of 16 bytes); together the ranks cover 0..N exactly once."""
    if world < 1 or not 0 <= rank < world or N < 0 or align < 1:
        raise ValueError("bad shard arguments")
    units = -(-N // align)
    lo_u = rank * units // world
    hi_u = (rank + 1) * units // world
    return min(N, lo_u * align), min(N, hi_u * align)


def shard(act: torch.Tensor, lo: int, hi: int, feature_axis: int) -> torch.Tensor:
    """The minibatch entries [lo, hi) of an activation in feature_axis layout, contiguous:
    rows of (N, F) (a view) or columns of (F, N) (a copy)."""
    if feature_axis == 1:
        return act[lo:hi]
    return act[:, lo:hi].contiguous()


def allreduce_dw(dw: torch.Tensor, group=None) -> torch.Tensor:
    """Sums dw over the ranks of `group` in place (the one exchange of a data-parallel step)."""
    if dist.is_available() and dist.is_initialized() and dist.get_world_size(group) > 1:
        dist.all_reduce(dw, op=dist.ReduceOp.SUM, group=group)
    return dw


def data_parallel_updat(x_shard, dy_shard, updat, dw=None, group=None):
    """Weight gradient of the whole minibatch: updat(x_shard, dy_shard[, dw]) on this rank's shard
    (the library's BlocksparseMatMul.updat on the GPU), then summed over the ranks."""
    g = updat(x_shard, dy_shard) if dw is None else updat(x_shard, dy_shard, dw)
    return allreduce_dw(g, group)


def data_parallel_step(m, x, w, dy, rank: int, world: int, group=None):
    """One training step of a block-sparse layer on this rank: fprop and bprop of its shard of the
    minibatch (no exchange) and the weight gradient summed over ranks.  x, dy hold the whole
    minibatch; returns (y_shard, dx_shard, dw, (lo, hi))."""
    N = m._N(x, m.C)
    align = 8 if (m.feature_axis == 0 and x.element_size() == 2) else (4 if m.feature_axis == 0 else 1)
    lo, hi = shard_bounds(N, rank, world, align)
    xs, dys = shard(x, lo, hi, m.feature_axis), shard(dy, lo, hi, m.feature_axis)
    y = m.fprop(xs, w)
    dx = m.bprop(dys, w)
    dw = data_parallel_updat(xs, dys, m.updat, group=group)
    return y, dx, dw, (lo, hi)
