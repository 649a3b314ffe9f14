"""Query sharding across GPUs (host logic only).

Decode queries are independent, so a batch splits across ranks by query with
no exchange on the data path; the only collective is the harness's
max-over-ranks of the measured time.
"""
from __future__ import annotations


def shard_queries(n_queries: int, world: int, rank: int) -> range:
    """Contiguous, balanced share of queries 0..n_queries-1 for `rank`."""
    if world <= 0 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(n_queries, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def max_over_ranks(value: float, device=None) -> float:
    """The largest `value` over all ranks of the default process group (the
    value itself when no group is initialised)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return float(value)
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())
