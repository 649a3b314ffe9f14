"""Sharding across GPUs (host logic only): a batch by query, or one long
history by group ranges.

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


# ---- one long sequence across ranks ------------------------------------------
#
# "Top-k chooses the set; time chooses the order" (AFN-017) and "A sparse mask
# is not sparse attention" (AFN-016) define the path for one query over its
# whole history.  When one history is split across ranks by contiguous ranges
# of complete groups (rank r holds groups [g_lo, g_hi) and, on the last rank,
# the raw tail), the path needs exactly one exchange:
#   1. each rank scores its groups and keeps its local top min(budget, n_r)
#      by (score descending, position ascending) -- every group of the global
#      set is in its own rank's local set, because the local order is the
#      global order restricted to the rank's groups;
#   2. the candidates are exchanged (all-gather of at most budget per rank)
#      and every rank merges them with the same rule: the chosen set, ties
#      decided during membership exactly as on one device;
#   3. the emitted row (chosen groups ascending, x4, then the tail) is the same
#      on every rank; the rows of rank r form one contiguous slice of it, and
#      rank order is time order;
#   4. each rank runs the online softmax over its slice, in order
#      (qsa_attend_state), and the per-rank states (m, l, acc) are merged in
#      ascending rank order (qsa_merge_states).


def shard_groups(n_groups: int, world: int, rank: int) -> range:
    """Contiguous, balanced share of groups 0..n_groups-1 for `rank`."""
    return shard_queries(n_groups, world, rank)


def order_keys(scores) -> "np.ndarray":
    """Order-preserving uint32 images of scores in [+0, +inf] (-0 read as +0)."""
    import numpy as np
    s = np.asarray(scores, dtype=np.float32)
    if s.size and (np.isnan(s).any() or (s < 0).any()):
        raise ValueError("scores must lie in [+0, +inf]")
    s = np.where(s == 0, np.float32(0.0), s).astype(np.float32)
    return s.view(np.uint32)


def _rank_order(keys, groups):
    """Indices ordering (key, group) by key descending, then group ascending."""
    import numpy as np
    return np.lexsort((np.asarray(groups, np.int64), -np.asarray(keys, np.int64)))


def local_candidates(scores, g_lo: int, budget: int):
    """This rank's top min(budget, n) groups of scores[0..n) (groups g_lo +
    i) as (keys uint32, groups int64), best first."""
    import numpy as np
    keys = order_keys(scores)
    groups = np.arange(g_lo, g_lo + keys.size, dtype=np.int64)
    take = _rank_order(keys, groups)[:min(budget, keys.size)]
    return keys[take], groups[take]


def merge_candidates(parts, budget: int, n_groups: int):
    """The chosen set of the whole history, ascending, from every rank's
    local candidates (any rank order)."""
    import numpy as np
    keys = np.concatenate([np.asarray(p[0], np.uint32) for p in parts]) if parts else np.zeros(0, np.uint32)
    groups = np.concatenate([np.asarray(p[1], np.int64) for p in parts]) if parts else np.zeros(0, np.int64)
    k = min(budget, n_groups)
    if groups.size < k:
        raise ValueError("fewer candidates than the budget: a rank sent too few")
    return np.sort(groups[_rank_order(keys, groups)[:k]])


def emitted_row(chosen, T: int):
    """Chosen groups (ascending) expanded to 4 token IDs each, then the raw
    tail [4 * floor(T/4), T): the row every rank holds."""
    import numpy as np
    chosen = np.asarray(chosen, np.int64)
    body = (4 * chosen[:, None] + np.arange(4, dtype=np.int64)[None, :]).reshape(-1)
    tail = np.arange(4 * (T // 4), T, dtype=np.int64)
    return np.concatenate([body, tail]).astype(np.int32)


def rank_rows(ids, g_lo: int, g_hi: int, last: bool) -> slice:
    """The contiguous slice of the emitted row owned by the rank holding
    groups [g_lo, g_hi) (and the tail, when it is the last rank)."""
    import numpy as np
    ids = np.asarray(ids, np.int64)
    start = int(np.searchsorted(ids, 4 * g_lo, side="left"))
    stop = ids.size if last else int(np.searchsorted(ids, 4 * g_hi, side="left"))
    return slice(start, stop)


def merge_states(dims, states, stream=None):
    """The attention output [B, n_q, d] of rows whose consecutive slices were
    attended apart (one slice per rank), from the slices' online-softmax
    states in row (rank) order: states = [(m [B, n_q], l [B, n_q],
    acc [B, n_q, d]), ...], device tensors as qsa_attend_state returns them.
    The merge itself runs in the library (qsa_merge_states); here the states
    are only stacked into the layout it takes."""
    import torch
    from . import qsa
    m = torch.stack([st[0] for st in states]).contiguous()
    l = torch.stack([st[1] for st in states]).contiguous()
    acc = torch.stack([st[2] for st in states]).contiguous()
    out = torch.empty_like(states[0][2])
    qsa.qsa_merge_states(dims, len(states), m, l, acc, out, stream)
    return out
