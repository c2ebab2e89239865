"""Data-parallel split of one attention call over ranks, one GPU per rank.

The (batch, head) problems of a call are independent: each needs only its own
q rows, the full K/V of its head and the shared tables.  So a call over BH
problems is partitioned into contiguous ranges, rank r taking
``[r*BH//world, (r+1)*BH//world)``; every rank runs the fused entry on its
range and nothing is exchanged while computing.  Only a consumer that needs the
whole output gathers it afterwards (``gather=True``), with one all-gather of
the output slices over the process group.

The backward splits the same way, with one exchange step: the tables are
shared by every (batch, head), so their gradients are the sum over ranks of
each rank's partial gradients (``fused_backward_shard``).

This module holds no arithmetic of the method: it slices, calls the library
entry point on the slice, gathers, and adds the ranks' table-gradient partials.
"""
from __future__ import annotations

from typing import Callable

import torch
import torch.distributed as dist

from . import api


def bh_range(BH: int, rank: int, world: int) -> tuple[int, int]:
    """Contiguous range ``[lo, hi)`` of the BH problems that `rank` of `world` computes.

    The ranges of ranks 0 .. world-1 tile ``[0, BH)`` in order; their sizes differ by at most one
    (BH need not be a multiple of world; ranks may get an empty range when BH < world)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} outside a world of {world}")
    if BH < 0:
        raise ValueError("BH must be >= 0")
    return rank * BH // world, (rank + 1) * BH // world


def fused_shard(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, rel_pos_h: torch.Tensor,
                rel_pos_w: torch.Tensor, H: int, W: int, scale: float | None = None, *, rank: int | None = None,
                world: int | None = None, gather: bool = False, group=None,
                compute: Callable[..., torch.Tensor] | None = None, **kwargs) -> torch.Tensor:
    """This rank's share of one fused call.

    q, k, v are the whole call's ``[BH, N, d]`` tensors (or any tensors whose first dimension is
    BH; only the rank's rows are read).  Returns the rank's output slice ``[hi - lo, N, d]``, or,
    with ``gather=True``, the whole ``[BH, N, d]`` output assembled by one all-gather of the
    slices.  `compute` defaults to the library's fused entry point; extra keyword arguments go to
    it."""
    if rank is None or world is None:
        if dist.is_available() and dist.is_initialized():
            rank, world = dist.get_rank(group), dist.get_world_size(group)
        else:
            rank, world = 0, 1
    BH = q.shape[0]
    lo, hi = bh_range(BH, rank, world)
    fn = compute or api.fused
    # an empty range (BH < world) is still one call: the entry point returns an empty slice
    # without touching the device, so every rank's slice has the same dtype
    part = fn(q[lo:hi], k[lo:hi], v[lo:hi], rel_pos_h, rel_pos_w, H, W, scale, **kwargs)
    if not gather or world == 1:
        return part
    # all_gather wants equal-sized buffers: pad every slice to the largest range
    width = -(-BH // world)
    buf = torch.zeros((width,) + tuple(part.shape[1:]), dtype=part.dtype, device=part.device)
    buf[:hi - lo] = part
    bufs = [torch.empty_like(buf) for _ in range(world)]
    dist.all_gather(bufs, buf, group=group)
    out = torch.empty((BH,) + tuple(part.shape[1:]), dtype=part.dtype, device=part.device)
    for r in range(world):
        a, b = bh_range(BH, r, world)
        out[a:b] = bufs[r][:b - a]
    return out


def fused_backward_shard(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, rel_pos_h: torch.Tensor,
                         rel_pos_w: torch.Tensor, out: torch.Tensor, lse: torch.Tensor, dout: torch.Tensor, H: int,
                         W: int, scale: float | None = None, *, rank: int | None = None, world: int | None = None,
                         group=None, reduce_tables: bool = True, compute: Callable[..., tuple] | None = None,
                         **kwargs):
    """This rank's share of one backward call: ``(dq, dk, dv, drel_pos_h, drel_pos_w)``.

    Every tensor with a leading BH dimension (q, k, v, out, lse, dout) is the whole call's; only
    the rank's range is read, and dq, dk, dv come back for that range.  The tables are shared by
    every (batch, head), so their gradients are the sum of all ranks' partial gradients: the one
    exchange step of the backward.  The partials are all-gathered and added in rank order, so
    every rank holds the same table gradients, bit for bit, whatever the backend.  With
    ``reduce_tables=False`` the rank's partial table gradients come back instead (no process
    group needed).  `compute` defaults to the library's backward entry point; extra keyword
    arguments go to it."""
    if rank is None or world is None:
        if dist.is_available() and dist.is_initialized():
            rank, world = dist.get_rank(group), dist.get_world_size(group)
        else:
            rank, world = 0, 1
    BH = q.shape[0]
    lo, hi = bh_range(BH, rank, world)
    fn = compute or api.fused_backward
    dq, dk, dv, dth, dtw = fn(q[lo:hi], k[lo:hi], v[lo:hi], rel_pos_h, rel_pos_w, out[lo:hi], lse[lo:hi],
                              dout[lo:hi], H, W, scale, **kwargs)
    if world == 1 or not reduce_tables:
        return dq, dk, dv, dth, dtw
    summed = []
    for part in (dth, dtw):
        bufs = [torch.empty_like(part) for _ in range(world)]
        dist.all_gather(bufs, part.contiguous(), group=group)
        total = bufs[0].clone()
        for r in range(1, world):
            total += bufs[r]
        summed.append(total)
    return dq, dk, dv, summed[0], summed[1]
