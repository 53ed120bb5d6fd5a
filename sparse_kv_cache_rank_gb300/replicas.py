"""Replica bookkeeping for runs on several GPUs of one node.

The refresh shards over independent sequences and has no exchange step, so N GPUs
run N independent replicas: each rank owns a contiguous slice of the sequences and
nothing crosses ranks on the data path.  The only cross-rank operations are host-side
timing reductions (a barrier around the timed region and the maximum elapsed time),
done with torch.distributed on whatever backend the process group uses.
"""
from __future__ import annotations

import os


def env_rank():
    """(rank, world_size, local_rank) from the torchrun environment (1 process if unset)."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_sequences(B: int, world: int, rank: int):
    """Contiguous [start, stop) slice of B sequences owned by `rank` (sizes differ by at most 1)."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad rank/world")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    return start, start + base + (1 if rank < extra else 0)


def max_over_ranks(values, device=None):
    """Element-wise maximum of a list of floats over all ranks (identity without a group)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def sum_over_ranks(values, device=None):
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return [float(v) for v in values]
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return [float(x) for x in t.tolist()]
