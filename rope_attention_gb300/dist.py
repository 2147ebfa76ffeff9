"""Multi-process plumbing for the data-parallel path: one process per GPU.

When every head of a call sits on one GPU (tp = 1), a token's projection row,
its norm and RoPE, and its KV-cache row depend on no other token (qkv_cte page,
Design 1b: the only cross-device step is the all-reduce of the per-token sums of
squares when heads are split).  A batch therefore shards by contiguous blocks of
rows, with W and the small per-channel tensors replicated, and no collective on
the data path: each process scatters its own tokens into its own cache replica
(slots are unique per token).  The collectives here are the ones a benchmark
needs around the timed region: a barrier and the maximum of the ranks' times.
"""
from __future__ import annotations

import os
from dataclasses import dataclass


@dataclass(frozen=True)
class DistEnv:
    world: int
    rank: int
    local_rank: int


def env() -> DistEnv:
    """World size and ranks from the launcher's environment (torchrun sets them)."""
    return DistEnv(int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
                   int(os.environ.get("LOCAL_RANK", "0")))


def shard_rows(total: int, world: int, rank: int) -> tuple[int, int]:
    """[begin, end) of rank `rank`'s contiguous block of `total` rows; block sizes
    differ by at most one and the blocks cover every row exactly once."""
    if world < 1 or not 0 <= rank < world or total < 0:
        raise ValueError(f"bad shard request: total={total} world={world} rank={rank}")
    base, extra = divmod(total, world)
    begin = rank * base + min(rank, extra)
    return begin, begin + base + (1 if rank < extra else 0)


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks (the slowest rank's time); the identity
    when no process group is running."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank: float, world: int, slowest_seconds: float) -> float:
    """Whole-job throughput: the units all ranks processed over the slowest rank's time."""
    if slowest_seconds <= 0:
        raise ValueError("elapsed time must be positive")
    return units_per_rank * world / slowest_seconds
