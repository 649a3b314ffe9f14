"""The shared-history scorer (queries of one chunked prefill), through the C
ABI: qsa_score_groups_shared and qsa_decode_shared.

"Top-k chooses the set; time chooses the order" (AFN-017) requires chunk =
decode: a query of a chunked prefill must see exactly what a single-query
decode at its position sees.  The shared scorer pools each tile of the
history once for many queries (one lane per query, two heads per lane, the
head sums in a second pass), so its scores, rows and outputs are checked bit
for bit against the per-query path (itself checked against the oracle
elsewhere)."""
import numpy as np
import pytest

from gpu_helpers import need_gpu, oracle_run, assert_ids_equal, assert_attention_close
from top_group_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _scores_equal(db, w):
    import torch
    db.score()
    torch.cuda.synchronize()
    ref = db.scores.cpu().numpy().copy()
    db.scores.fill_(float("nan"))
    db.score_shared()
    assert db.check_errors() == (0, 0)
    got = db.scores.cpu().numpy()
    for b in range(w.batch):
        G = int(w.visible[b]) // 4
        assert got[b, :G].tobytes() == ref[b, :G].tobytes(), b


def _decode_equal(db, w):
    import torch
    db.decode()
    torch.cuda.synchronize()
    ids, n, out = db.ids.cpu().numpy().copy(), db.n_ids.cpu().numpy().copy(), db.out.cpu().numpy().copy()
    db.ids.fill_(-1)
    db.out.fill_(float("nan"))
    db.decode_shared()
    assert db.check_errors() == (0, 0)
    assert np.array_equal(db.n_ids.cpu().numpy(), n)
    got = db.ids.cpu().numpy()
    for b in range(w.batch):
        assert got[b, :n[b]].tobytes() == ids[b, :n[b]].tobytes(), b
    assert db.out.cpu().numpy().tobytes() == out.tobytes()


@pytest.mark.parametrize("shape", [(8, 64, 16, 2, 128), (4, 32, 4, 4, 64), (8, 32, 8, 2, 64), (4, 64, 2, 2, 64)])
def test_shared_scores_and_decode_equal_per_query(shape):
    """Every compiled indexer shape; ragged T over one history (one query
    below the budget, one with a tail, one past a tile boundary); 37 queries
    so the last query block is partly empty."""
    need_gpu()
    from top_group_sparse_gb300 import qsa
    H, dI, nq, nkv, hd = shape
    vis = [9001 + 7 * i for i in range(34)] + [37, 2052, 4 * 777 + 3]
    w = wl.make_workload("shared", vis, idx_heads=H, idx_dim=dI, q_heads=nq, kv_heads=nkv, head_dim=hd,
                         seed=81 + H * dI, history="shared", slots="paged16")
    db = qsa.DeviceBatch(w)
    _scores_equal(db, w)
    _decode_equal(db, w)


@pytest.mark.parametrize("nq", [150, 65])
def test_shared_partial_last_query_block(nq):
    """Batches of several 64-query blocks whose last block is partial (150 =
    64 + 64 + 22; 65 = 64 + 1): the blocks get CTAs in proportion to their
    queries, and every query's scores and rows equal the per-query path."""
    need_gpu()
    from top_group_sparse_gb300 import qsa
    vis = [4000 + 13 * i for i in range(nq - 2)] + [2051, 4 * 1001]
    w = wl.make_workload("shared_blocks", vis, idx_heads=8, idx_dim=64, q_heads=16, kv_heads=2, head_dim=128,
                         seed=91 + nq, history="shared", slots="paged16")
    db = qsa.DeviceBatch(w)
    _scores_equal(db, w)
    _decode_equal(db, w)


def test_shared_decode_matches_oracle_small():
    need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.chunked_prefill_100000(n=24, first=9000)
    db = qsa.DeviceBatch(w)
    db.decode_shared()
    st, flags = db.check_errors()
    assert st == 0, hex(flags)
    import torch
    torch.cuda.synchronize()
    gpu = {"ids": db.ids.cpu().numpy(), "n_ids": db.n_ids.cpu().numpy(), "out": db.out.cpu().numpy()}
    ref = oracle_run(w)
    assert_ids_equal(w, gpu, ref)
    assert_attention_close(w, gpu, ref)


def test_shared_full_size_chunked_prefill_100000():
    """The chunked-prefill workload at full size: 256 queries at positions
    100,000..100,255 of one history."""
    need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.chunked_prefill_100000()
    db = qsa.DeviceBatch(w)
    _scores_equal(db, w)
    _decode_equal(db, w)


def test_shared_flags_queries_of_another_history():
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.make_workload("two", [5000, 6000, 7000], idx_heads=8, idx_dim=64, q_heads=16, kv_heads=2,
                         head_dim=128, seed=83, history="independent", slots="identity")
    db = qsa.DeviceBatch(w)
    db.score_shared()
    st, flags = db.check_errors()
    assert st == qsa.QSA_ERR_DEVICE_FAULT and flags & qsa.QSA_DEVERR_NOT_SHARED
    # query 0 (the history at key_offset[0]) is still scored exactly
    torch.cuda.synchronize()
    got = db.scores.cpu().numpy()[0, :1250].copy()
    db.score()
    torch.cuda.synchronize()
    assert got.tobytes() == db.scores.cpu().numpy()[0, :1250].tobytes()
