"""Host-side helpers for running one decode replica per GPU (one process per
rank, torch.distributed): batches are independent, so ranks share nothing on
the data path and only the timing is combined -- the slowest rank's time, and
the work of all ranks, give the whole-job rate."""
from __future__ import annotations

import os
from typing import Tuple


def world() -> Tuple[int, int, int]:
    """(world_size, rank, local_rank) from the torchrun environment (1, 0, 0 when absent)."""
    return (int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")),
            int(os.environ.get("LOCAL_RANK", "0")))


def max_over_ranks(x: float, world_size: int, device="cpu") -> float:
    """The maximum of x over all ranks (x itself for one rank)."""
    if world_size == 1:
        return float(x)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world_size: int, max_seconds: float) -> float:
    """Units processed by all ranks per second of the slowest rank."""
    return world_size * units_per_rank / max_seconds


def barrier(world_size: int) -> None:
    if world_size > 1:
        import torch.distributed as dist

        dist.barrier()
