"""Multi-GPU layout of the hot path: independent sequences, no exchange.

Sequences (and their block pools) are independent units of the paged-attention
hot path, so N GPUs run N shards of a global batch with no collective on the
data path: rank r owns its own pool, block tables and sequences (drawn with
seed + r).  The only cross-rank operations are host-side bookkeeping used by
the benchmark: a barrier and the max over ranks of the measured step time.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def shard_seed(base_seed: int, rank: int) -> int:
    """Seed of rank ``rank``'s shard: every rank draws a different batch of the same shape."""
    return int(base_seed) + int(rank)


def max_over_ranks(values, device=None) -> list:
    """Element-wise max of a list of floats over all ranks (identity when not distributed)."""
    vals = [float(v) for v in values]
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return vals
    t = torch.tensor(vals, dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return t.tolist()


def total_units(units_per_rank: int) -> int:
    """Units (decode tokens) processed by the whole job in one step."""
    world = dist.get_world_size() if (dist.is_available() and dist.is_initialized()) else 1
    return int(units_per_rank) * world
