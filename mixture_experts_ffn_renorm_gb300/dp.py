"""Data-parallel replicas of the MoE block: the host-side logic.

Tokens are independent, so N GPUs process N disjoint token batches with the
same (replicated) expert weights and no collective on the data path.  This
module holds the pieces that decide who does what and how the per-rank timings
combine; the only collectives are a barrier and a max (gloo or NCCL).
"""
from __future__ import annotations

import os


def world() -> tuple[int, int, int]:
    """(world_size, rank, local_rank) from the torchrun environment (1, 0, 0 without)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def shard_range(n_total: int, rank: int, world_size: int) -> tuple[int, int]:
    """Contiguous, balanced [lo, hi) share of n_total items for `rank`."""
    base, extra = divmod(n_total, world_size)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def barrier(world_size: int) -> None:
    if world_size > 1:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v: float, world_size: int, device=None) -> float:
    """The largest v over all ranks (the step time of the slowest replica)."""
    if world_size == 1:
        return float(v)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(v)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_tokens_per_s(tokens_per_rank: int, world_size: int, max_ms: float) -> float:
    """Whole-job throughput: all ranks' tokens over the slowest rank's time."""
    return world_size * tokens_per_rank / (max_ms / 1000.0)
