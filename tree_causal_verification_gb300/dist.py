"""Multi-GPU plumbing for the step: the path shards by sequence.

Every unit of work in one step (a sequence's depth rows, its tree, its KV
heads, its acceptance walk) is independent of every other sequence, so N
GPUs run N independent shards with no data-path collective. The helpers here
are the only cross-rank logic: which sequences a rank owns, the slowest
rank's time, and whole-job throughput.
"""
from __future__ import annotations

import os


def rank_world():
    """(rank, world_size, local_rank) from the torchrun environment."""
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_sequences(batch: int, rank: int, world: int) -> range:
    """Contiguous, balanced slice of a batch of sequences owned by `rank`.

    Sizes differ by at most one; the slices of all ranks cover 0..batch-1
    exactly once, in order.
    """
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"bad rank {rank} of {world}")
    base, extra = divmod(batch, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks (identity without torch.distributed)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(value: float, device=None) -> float:
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def job_throughput(units_this_rank: float, seconds_this_rank: float, device=None) -> float:
    """Whole-job units per second: the units of all ranks over the slowest rank's time."""
    units = sum_over_ranks(units_this_rank, device)
    seconds = max_over_ranks(seconds_this_rank, device)
    return units / seconds
