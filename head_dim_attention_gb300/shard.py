"""Host-side work split for several GPUs (one process per GPU).

Attention over (batch, kv-head group) units is embarrassingly parallel: a
unit's forward and backward read only its own Q/K/V/O/dO rows, and the dK/dV
sums over the query heads of a GQA group stay inside the unit.  So ranks split
units and never exchange data; the only collective is the MAX of the elapsed
time that the benchmark reports.
"""
from __future__ import annotations

from typing import List, Tuple


def units(batch: int, hkv: int) -> List[Tuple[int, int]]:
    """All (batch index, kv head) units of a problem."""
    if batch < 0 or hkv < 0:
        raise ValueError("batch and hkv must be non-negative")
    return [(b, h) for b in range(batch) for h in range(hkv)]


def shard(all_units: List[Tuple[int, int]], rank: int, world: int) -> List[Tuple[int, int]]:
    """Contiguous block of units for `rank` of `world`; sizes differ by at most one."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("need 0 <= rank < world")
    n = len(all_units)
    base, extra = divmod(n, world)
    start = rank * base + min(rank, extra)
    stop = start + base + (1 if rank < extra else 0)
    return all_units[start:stop]


def max_over_ranks(value: float, device=None) -> float:
    """MAX of a float over all ranks of the default process group (identity without one)."""
    import torch
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
