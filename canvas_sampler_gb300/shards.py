"""Exchange of vocabulary-shard records between ranks: each rank runs the step over its token
range (Sampler.step_shard), the records are gathered in rank order (= token order) and every
rank merges them (Sampler.merge_shards). Only tensors move here; the arithmetic of the step
and of the merge is in the library's kernels."""
from __future__ import annotations

import torch

from .sampler import ShardPartial


def shard_range(vocab_total: int, world: int, rank: int, align: int = 256) -> tuple[int, int]:
    """Token range [begin, end) of a rank: contiguous, in rank order, multiples of `align`
    (the last rank takes the remainder)."""
    if vocab_total % align or world < 1 or not 0 <= rank < world:
        raise ValueError("vocabulary must be a multiple of the alignment, rank in [0, world)")
    units = vocab_total // align
    per = units // world
    if per == 0:
        raise ValueError("fewer alignment units than ranks")
    begin = rank * per * align
    end = vocab_total if rank == world - 1 else (rank + 1) * per * align
    return begin, end


def gather_partials(part: ShardPartial, group=None) -> ShardPartial:
    """All-gather one record per rank (each of shard count 1) into records stacked in rank
    order. Works for any backend whose tensors live where the record does (CPU tensors for
    gloo, CUDA tensors for NCCL)."""
    import torch.distributed as dist
    world = dist.get_world_size(group)
    out = []
    for t in part.tensors():
        bufs = [torch.empty_like(t) for _ in range(world)]
        dist.all_gather(bufs, t.contiguous(), group=group)
        out.append(torch.cat(bufs))
    return ShardPartial(*out) if len(out) == 4 else ShardPartial(out[0], out[1], out[2], None)
