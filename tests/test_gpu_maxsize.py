"""The largest history the library accepts, through the whole-path call.

Query 0 sees T = QSA_MAX_VISIBLE = 2^26 tokens (16,777,216 groups: the
selection's plain path over every key, a scores row of 64 MiB); query 1's
history starts right after it, at index-key element 2^26 * 32 = 2^31, so
every address of its keys lies past the reach of 32-bit element arithmetic.
Both queries' scores and ID rows must equal the oracle's bit for bit, and
their outputs must be within 1e-5 * max|V|.  The K/V cache is a ring of
65,536 slots per history (the slot map folds the tokens onto it), so the
device holds ~9 GB, nearly all of it index keys."""
import gc

import numpy as np
import pytest

from gpu_helpers import (assert_attention_close, assert_ids_equal, assert_scores_equal,
                         need_gpu, oracle_run, run_decode)
from top_group_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

QSA_MAX_VISIBLE = 1 << 26


def test_max_visible_history_and_keys_past_2_31_elements():
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.make_workload("maxsize", [QSA_MAX_VISIBLE, 5003], idx_heads=4, idx_dim=32, q_heads=2,
                         kv_heads=1, head_dim=64, seed=123, slots="ring", ring_size=65536)
    assert int(w.key_offset[1]) * w.idx_dim == 1 << 31
    db = qsa.DeviceBatch(w)
    gpu = run_decode(w, db=db)
    gpu.pop("batch")
    assert gpu["status"] == 0, f"device error flags {gpu['flags']:#x}"
    db.score()
    torch.cuda.synchronize()
    gpu["scores"] = db.scores.cpu().numpy()
    assert db.check_errors() == (0, 0)
    del db
    gc.collect()
    torch.cuda.empty_cache()
    ref = oracle_run(w)
    assert_scores_equal(w, gpu, ref)
    assert_ids_equal(w, gpu, ref)
    assert_attention_close(w, gpu, ref)
    assert gpu["n_ids"].tolist() == [2048, 2051]
    del w, gpu, ref
    gc.collect()


def test_max_batch_of_65535_queries():
    """The largest accepted batch (65,535 queries: the attention grid's query
    dimension and its merge launch at their limit, a selection grid of
    65,535 CTAs): T_b = b mod 41 (no groups, dense rows below the budget),
    every 1,000th query T = 5,000 + b mod 4 (top-k with a tail).  ID rows
    bit-exact and outputs within 1e-5 * max|V| for every query."""
    need_gpu()
    from top_group_sparse_gb300 import qsa
    B = 65535
    vis = [5000 + b % 4 if b % 1000 == 999 else b % 41 for b in range(B)]
    w = wl.make_workload("maxbatch", vis, idx_heads=4, idx_dim=32, q_heads=2, kv_heads=1, head_dim=64,
                         seed=124, slots="paged16")
    db = qsa.DeviceBatch(w)
    gpu = run_decode(w, db=db)
    gpu.pop("batch")
    assert gpu["status"] == 0, f"device error flags {gpu['flags']:#x}"
    del db
    gc.collect()
    ref = oracle_run(w)
    assert_ids_equal(w, gpu, ref)
    assert_attention_close(w, gpu, ref)
    assert gpu["n_ids"].tolist() == [4 * min(t // 4, 512) + t % 4 for t in vis]
    del w, gpu, ref
    gc.collect()
