"""Seeded synthetic inputs for physically sparse QSA decode.

This module holds no step of the method: no pooling, scoring, selection or
attention arithmetic.  It only draws the arrays a decode step consumes, with
the shapes, value distributions and slot-map structures of the five
workloads the library is checked and measured on.  The CUDA path's tests and
benchmark and the CPU oracle read the very same host arrays.

Recipe (all draws on the CPU from ``torch.Generator().manual_seed(seed)``,
in this order: indexer queries, raw index keys, attention queries, K cache,
V cache, slot-map permutation):

* values ``normal``: N(0, 1) float32;  ``grid8``: integers uniform in
  [-4, 4] divided by 8, so that pooled keys, products and dot sums are all
  exactly representable in float32;
* history ``independent``: query b owns its own history of T_b tokens,
  laid out back to back in logical order; ``shared``: every query reads a
  prefix of one history (chunked prefill, the dense-parity sweep);
* slot maps (logical token -> physical KV slot, per history):
  ``identity``; ``permutation`` (a seeded random permutation of all slots);
  ``paged16`` (16-token pages drawn from one seeded random permutation of a
  page pool; slot = page * 16 + t % 16); ``ring`` (each history owns a ring
  of R slots that has wrapped: slot = base + (t + shift) mod R).

No public dataset is involved: the notes measure on model-free synthetic
inputs, which these stand in for.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

GROUP = 4
DEFAULT_BUDGET = 512


@dataclasses.dataclass
class QsaWorkload:
    name: str
    idx_heads: int
    idx_dim: int
    q_heads: int
    kv_heads: int
    head_dim: int
    budget: int
    scale: float
    max_visible: int
    q_idx: np.ndarray        # float32 [B, idx_heads, idx_dim]
    idx_keys: np.ndarray     # float32 [total_tokens, idx_dim], logical order
    key_offset: np.ndarray   # int64 [B]: first row of query b's history
    visible: np.ndarray      # int32 [B]: T_b
    q: np.ndarray            # float32 [B, q_heads, head_dim]
    k_cache: np.ndarray      # float32 [num_slots, kv_heads, head_dim]
    v_cache: np.ndarray      # float32 [num_slots, kv_heads, head_dim]
    slot_map: np.ndarray     # int32 [total_tokens]: logical -> physical slot
    slot_offset: np.ndarray  # int64 [B]: first slot-map entry of query b
    seed: int = 0
    values: str = "normal"
    slots: str = "identity"

    @property
    def batch(self) -> int:
        return int(self.visible.shape[0])

    @property
    def num_slots(self) -> int:
        return int(self.k_cache.shape[0])

    @property
    def total_tokens(self) -> int:
        return int(self.idx_keys.shape[0])

    @property
    def row_cap(self) -> int:
        """Capacity of one emitted ID row: budget groups of 4 plus a 3-token tail."""
        return GROUP * self.budget + GROUP - 1

    def subset(self, queries) -> "QsaWorkload":
        """The same histories and caches with a subset of the queries."""
        sel = np.asarray(queries, dtype=np.int64)
        return dataclasses.replace(
            self, q_idx=self.q_idx[sel], key_offset=self.key_offset[sel],
            visible=self.visible[sel], q=self.q[sel], slot_offset=self.slot_offset[sel],
            max_visible=int(max(self.visible[sel].max(initial=0), 0)))


def _draw(gen: torch.Generator, shape, values: str) -> np.ndarray:
    shape = tuple(int(s) for s in shape)
    if values == "normal":
        t = torch.randn(shape, generator=gen, dtype=torch.float32)
    elif values == "grid8":
        t = torch.randint(-4, 5, shape, generator=gen, dtype=torch.int32).to(torch.float32) / 8.0
    else:
        raise ValueError(values)
    return t.numpy()


def make_workload(name: str, visible, *, idx_heads: int, idx_dim: int, q_heads: int,
                  kv_heads: int, head_dim: int, seed: int, history: str = "independent",
                  slots: str = "identity", index_values: str = "normal",
                  budget: int = DEFAULT_BUDGET, ring_size: int | None = None,
                  ring_shift: int | None = None, page: int = 16,
                  extra_pages: int = 0, scale: float | None = None) -> QsaWorkload:
    """Build one seeded workload.

    visible: the T_b of each query.  history 'independent' gives each query
    its own history of T_b tokens; 'shared' gives all queries one history of
    max(T_b) tokens.  index_values applies to indexer queries and index
    keys; attention queries and K/V are always N(0, 1).
    """
    vis = np.asarray(list(visible), dtype=np.int32)
    B = int(vis.shape[0])
    gen = torch.Generator().manual_seed(int(seed))
    if history == "independent":
        lengths = [int(t) for t in vis]
        key_offset = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64) if B else np.zeros(0, np.int64)
    elif history == "shared":
        lengths = [int(vis.max(initial=0))]
        key_offset = np.zeros(B, np.int64)
    else:
        raise ValueError(history)
    total = int(sum(lengths))
    region_start = np.concatenate([[0], np.cumsum(lengths)[:-1]]).astype(np.int64) if lengths else np.zeros(0, np.int64)

    q_idx = _draw(gen, (B, idx_heads, idx_dim), index_values)
    idx_keys = _draw(gen, (max(total, 0), idx_dim), index_values)
    q = _draw(gen, (B, q_heads, head_dim), "normal")

    # Slot-map structure decides how many physical slots the caches hold.
    if slots in ("identity", "permutation"):
        num_slots = max(total, 1)
    elif slots == "paged16":
        pages_per = [-(-L // page) + extra_pages for L in lengths]
        num_slots = max(sum(pages_per) * page, 1)
    elif slots == "ring":
        R = int(ring_size if ring_size is not None else max(lengths, default=1))
        num_slots = max(R * len(lengths), 1)
    else:
        raise ValueError(slots)

    k_cache = _draw(gen, (num_slots, kv_heads, head_dim), "normal")
    v_cache = _draw(gen, (num_slots, kv_heads, head_dim), "normal")

    slot_map = np.empty(max(total, 0), np.int32)
    if slots == "identity":
        slot_map[:] = np.arange(total, dtype=np.int32)
    elif slots == "permutation":
        slot_map[:] = torch.randperm(total, generator=gen).numpy().astype(np.int32)
    elif slots == "paged16":
        perm = torch.randperm(num_slots // page, generator=gen).numpy().astype(np.int64)
        first_page = 0
        for r, L in enumerate(lengths):
            t = np.arange(L, dtype=np.int64)
            pages = perm[first_page:first_page + pages_per[r]]
            slot_map[region_start[r]:region_start[r] + L] = (pages[t // page] * page + t % page).astype(np.int32)
            first_page += pages_per[r]
    elif slots == "ring":
        shift = int(ring_shift if ring_shift is not None else R // 2)
        for r, L in enumerate(lengths):
            t = np.arange(L, dtype=np.int64)
            slot_map[region_start[r]:region_start[r] + L] = (r * R + (t + shift) % R).astype(np.int32)

    slot_offset = key_offset.copy()
    return QsaWorkload(
        name=name, idx_heads=idx_heads, idx_dim=idx_dim, q_heads=q_heads,
        kv_heads=kv_heads, head_dim=head_dim, budget=int(budget),
        scale=float(np.float32(1.0 / math.sqrt(head_dim))) if scale is None else float(scale),
        max_visible=int(vis.max(initial=0)), q_idx=q_idx, idx_keys=idx_keys,
        key_offset=key_offset, visible=vis, q=q, k_cache=k_cache, v_cache=v_cache,
        slot_map=slot_map, slot_offset=slot_offset, seed=int(seed),
        values=index_values, slots=slots)


# ---- the five named workloads ---------------------------------------------

def single_t37(seed: int = 1) -> QsaWorkload:
    """One decode query over 37 visible tokens (9 groups + 1-token tail, below
    budget): indexer 4 heads x 32, attention 1 KV head x 64, identity slots."""
    return make_workload("single_t37", [37], idx_heads=4, idx_dim=32, q_heads=1,
                         kv_heads=1, head_dim=64, seed=seed, slots="identity")


DENSE_SWEEP_T = (0, 1, 2, 3, 4, 5, 2047, 2048, 2049, 2050, 2051, 2052)


def dense_parity_sweep(seed: int = 2) -> QsaWorkload:
    """One query per T in {0..5, 2047..2052} over one shared history of 2,052
    tokens; indexer values on the k/8 grid (exact dots, many ties); 2 KV
    heads x 64; slot map a seeded random permutation."""
    return make_workload("dense_parity_sweep", DENSE_SWEEP_T, idx_heads=4, idx_dim=32,
                         q_heads=2, kv_heads=2, head_dim=64, seed=seed, history="shared",
                         slots="permutation", index_values="grid8")


def batched_65537(seed: int = 3, batch: int = 32, T: int = 65537) -> QsaWorkload:
    """32 independent decode queries at T = 65,537 (16,384 groups + 1 tail);
    indexer 8 x 64; GQA 16 q / 2 KV heads x 128; 16-token pages."""
    return make_workload("batched_65537", [T] * batch, idx_heads=8, idx_dim=64,
                         q_heads=16, kv_heads=2, head_dim=128, seed=seed, slots="paged16")


def long_262144(seed: int = 4, batch: int = 8, T: int = 262144) -> QsaWorkload:
    """8 independent decode queries at T = 262,144 (65,536 groups, no tail);
    indexer 8 x 64; GQA 16 q / 2 KV heads x 128; each history a ring buffer
    of 262,144 slots that has wrapped once (slot = (t + 131,072) mod 262,144)."""
    return make_workload("long_262144", [T] * batch, idx_heads=8, idx_dim=64,
                         q_heads=16, kv_heads=2, head_dim=128, seed=seed, slots="ring",
                         ring_size=T, ring_shift=T // 2)


def chunked_prefill_100000(seed: int = 5, n: int = 256, first: int = 100000) -> QsaWorkload:
    """256 consecutive queries at positions 100,000..100,255 of one history,
    query at position p seeing tokens 0..p (T = p + 1); indexer 8 x 64;
    GQA 16 q / 2 KV heads x 128; 16-token pages."""
    return make_workload("chunked_prefill_100000", [first + i + 1 for i in range(n)],
                         idx_heads=8, idx_dim=64, q_heads=16, kv_heads=2, head_dim=128,
                         seed=seed, history="shared", slots="paged16")


WORKLOADS = {
    "single_t37": single_t37,
    "dense_parity_sweep": dense_parity_sweep,
    "batched_65537": batched_65537,
    "long_262144": long_262144,
    "chunked_prefill_100000": chunked_prefill_100000,
}
