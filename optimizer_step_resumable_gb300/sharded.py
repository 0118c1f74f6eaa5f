"""Sharded (ZeRO-1 style) optimizer step: host-side partition and exchange.

Each rank owns one contiguous range of the flat state (its shard of w, m, v
and the gradient of that range).  The global clip needs the norm of the
whole gradient, so the ranks exchange their shards' sums of squares -- one
double each.  The library adds them in rank order (adamw_clip_step_ranks on
the host, adamw_clip_step_gathered on the device), which makes the result
the same on every rank and from run to run, and runs the fused update on
the rank's own shard with that global sum.  This module only partitions and
exchanges (torch.distributed, gloo or NCCL); the arithmetic runs in the
library.
"""
from __future__ import annotations

import time

from . import (adamw_clip_step_gathered, adamw_clip_step_ranks, ckpt_consolidate,
               ckpt_manifest_commit, ckpt_pack, ckpt_probe, ckpt_read_range, ckpt_shard_read,
               ckpt_shard_write, grad_sumsq, grad_sumsq_to)


def shard_range(n: int, rank: int, world: int, align: int = 4):
    """(offset, numel) of rank's contiguous shard of [0, n): equal shards of
    a multiple of `align` elements (16-byte boundaries for float32), the
    remainder on the last rank."""
    if world < 1 or not 0 <= rank < world or n < world:
        raise ValueError("need 0 <= rank < world <= n")
    base = (n // world) // align * align
    if base == 0:
        base = n // world
    off = rank * base
    numel = n - off if rank == world - 1 else base
    return off, numel


def gather_sumsq(local: float, group=None) -> list:
    """Every rank's local sum of squares, in rank order (an all-gather; the
    library adds them up).  Without an initialised process group: [local]."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return [float(local)]
    world = dist.get_world_size(group)
    backend = dist.get_backend(group)
    device = (torch.device("cuda", torch.cuda.current_device())
              if backend == "nccl" else torch.device("cpu"))
    mine = torch.tensor([float(local)], dtype=torch.float64, device=device)
    parts = [torch.empty_like(mine) for _ in range(world)]
    dist.all_gather(parts, mine, group=group)
    return [p.item() for p in parts]


def sharded_clip_step(ctx, w, g, m, v, t, lr, wd, clip, grad_scale=1.0, zero_grad=False,
                      group=None, stream=None):
    """One clipped-AdamW step on this rank's shard; returns the gathered
    per-rank sums of squares of the raw gradient (rank order)."""
    parts = gather_sumsq(grad_sumsq(ctx, g, stream=stream), group)
    adamw_clip_step_ranks(ctx, w, g, m, v, t, lr, wd, clip, parts, grad_scale=grad_scale,
                          zero_grad=zero_grad, stream=stream)
    return parts


class DeviceExchange:
    """Buffers of the on-device exchange: one float64 to send, one per rank
    to receive (CUDA tensors, reused every step)."""

    def __init__(self, world: int, device):
        import torch
        self.send = torch.zeros(1, dtype=torch.float64, device=device)
        self.recv = torch.zeros(world, dtype=torch.float64, device=device)


def sharded_clip_step_device(ctx, w, g, m, v, t, lr, wd, clip, exchange, grad_scale=1.0,
                             zero_grad=False, group=None):
    """One clipped-AdamW step on this rank's shard with no host round trip:
    the shard's sum of squares goes to exchange.send on the current stream,
    an all-gather (NCCL: on the device) fills exchange.recv in rank order,
    and the library adds it up in rank order on the device and updates the
    shard -- the same bits as sharded_clip_step."""
    import torch.distributed as dist
    grad_sumsq_to(ctx, g, exchange.send)
    if dist.is_available() and dist.is_initialized():
        dist.all_gather_into_tensor(exchange.recv, exchange.send, group=group)
    else:
        exchange.recv.copy_(exchange.send)
    adamw_clip_step_gathered(ctx, w, g, m, v, t, lr, wd, clip, exchange.recv,
                             grad_scale=grad_scale, zero_grad=zero_grad)


def _gather_objects(obj, group=None):
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized():
        return [obj]
    out = [None] * dist.get_world_size(group)
    dist.all_gather_object(out, obj, group=group)
    return out


def save_sharded(ctx, directory, step, w, m, v, rank, world, offsets, numels, group=None,
                 main_stream=None, side_stream=None, wall_clock_seconds=None):
    """Sharded checkpoint of this rank's shard: pack, write rank<R>.bin and
    take its sha256; exchange the digests; rank 0 commits the manifest and
    renames the step directory; all ranks return its path."""
    import torch.distributed as dist
    ckpt_pack(ctx, step, w, m, v, main_stream=main_stream, side_stream=side_stream)
    digest = ckpt_shard_write(ctx, directory, rank)
    digests = _gather_objects(digest, group)
    path = None
    if rank == 0:
        wall = time.time() if wall_clock_seconds is None else wall_clock_seconds
        path = ckpt_manifest_commit(directory, step, offsets, numels, digests, wall)
    paths = _gather_objects(path, group)
    if dist.is_available() and dist.is_initialized():
        dist.barrier(group)
    return paths[0]


def load_sharded(ctx, step_dir, rank, world, w, m, v, stream=None):
    """Reads this rank's shard after validating the manifest against the
    world size and the shard's sha256; returns the stored step."""
    return ckpt_shard_read(ctx, step_dir, rank, w, m, v, expected_world=world, stream=stream)


def consolidate(step_dir, out_dir, expected_world=-1):
    """The flat step_NNNNNN.bin of a sharded checkpoint (host only; every
    shard's sha256 checked); returns its path."""
    return ckpt_consolidate(step_dir, out_dir, expected_world)


def load_range(ctx, flat_path, rank, world, w, m, v, stream=None):
    """This rank's shard_range of a flat checkpoint -- for example one
    consolidated from a run with another world size -- into w, m, v (the
    context holds exactly that range); returns the stored step."""
    _, n_total = ckpt_probe(flat_path)
    off, numel = shard_range(n_total, rank, world)
    if numel != ctx.n:
        raise ValueError(f"rank {rank} of {world} owns {numel} parameters, the context {ctx.n}")
    return ckpt_read_range(ctx, flat_path, off, w, m, v, stream=stream)
