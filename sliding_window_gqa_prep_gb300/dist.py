"""Multi-GPU plumbing of the token path: sequences are independent (each has
its own ring, meta and sinks), so N GPUs split the sequences of a batch and
no collective touches the data path. Only timings cross ranks.
"""
from __future__ import annotations

import torch


def shard_sequences(B: int, rank: int, world: int) -> list:
    """Sequences rank `rank` of `world` takes from a batch of B: a contiguous
    block, sizes differing by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError(f"rank {rank} of world {world}")
    base, extra = divmod(B, world)
    start = rank * base + min(rank, extra)
    return list(range(start, start + base + (1 if rank < extra else 0)))


def max_over_ranks(value: float, device=None) -> float:
    """Largest `value` over all ranks (a plain float when not distributed)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())
