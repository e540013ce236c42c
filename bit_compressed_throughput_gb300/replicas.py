"""Host logic for running the block schedule on several GPUs as independent replicas.

Sequences never interact in a decoder stack, so the path partitions by blocks: rank r owns
the block of B sequences with global ids [r*B, (r+1)*B) and runs it start to finish with
no data-path collective (weak scaling: per-GPU work is fixed).  The only cross-rank
operation is the timing reduction (the slowest rank's time) and, for checking, a gather.
"""
from __future__ import annotations

import numpy as np


def block_sequences(rank: int, B: int) -> np.ndarray:
    """Global sequence ids of rank ``rank``'s block."""
    return np.arange(rank * B, (rank + 1) * B)


def max_over_ranks(value: float, dist=None, device=None) -> float:
    """The slowest rank's elapsed time (no-op without a process group)."""
    if dist is None or not dist.is_initialized() or dist.get_world_size() == 1:
        return float(value)
    import torch
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def total_tokens(world: int, B: int, n: int, steps: int) -> int:
    """Generated tokens of a timed run over all ranks."""
    return world * B * n * steps
