"""The incremental form of the scorer, through the C ABI: a pooled-key cache
appended as groups complete (qsa_pool_groups), scored from (qsa_score_pooled,
qsa_decode_pooled).

"Top-k chooses the set; time chooses the order" (AFN-017) names the
full-raw / incremental identity among its checks: pooling the raw keys at
every step and scoring from a cache of pooled keys must give the same scores,
hence the same rows and outputs, bit for bit.  Checked here against the
oracle's cache (built token by token) and against the full-raw GPU path, at
small sizes, across a run of decode steps that complete new groups, and at
the benchmark's full size."""
import numpy as np
import pytest

from gpu_helpers import need_gpu
from top_group_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _logical(rows):
    """The cache's rows [G, d] with their 16-byte chunks put back in order:
    chunk c of group g is stored at position c ^ (g & 7)."""
    G, D = rows.shape
    idx = np.arange(D // 4)[None, :] ^ (np.arange(G)[:, None] & 7)
    return np.take_along_axis(rows.reshape(G, D // 4, 4), idx[:, :, None], axis=1).reshape(G, D)


def _paged():
    return wl.make_workload("inc", [9001, 2052, 40003, 5, 0], idx_heads=8, idx_dim=64, q_heads=16,
                            kv_heads=2, head_dim=128, seed=71, slots="paged16")


def _batch(w):
    from top_group_sparse_gb300 import qsa
    db = qsa.DeviceBatch(w)
    db.make_pooled_cache()
    return db


def test_pooled_cache_matches_oracle_bitwise():
    torch = need_gpu()
    import oracle
    w = _paged()
    db = _batch(w)
    db.pool_all()
    assert db.check_errors() == (0, 0)
    pooled = db.pooled.cpu().numpy()
    po = db.pool_offset.cpu().numpy()
    for b in range(w.batch):
        T = int(w.visible[b])
        G = T // 4
        ko = int(w.key_offset[b])
        ref = oracle.pool_cache(w.idx_keys[ko:ko + T], T)
        got = _logical(pooled[po[b]:po[b] + G])
        assert got.tobytes() == ref.tobytes(), b


@pytest.mark.parametrize("kind", ["paged", "shared_history", "idx4x32", "idx8x32", "idx4x64"])
def test_score_pooled_equals_full_raw_bitwise(kind):
    """The pooled-key scorer (a thread holds two heads and runs H chains over
    H/2 groups) against the raw-key scorer, bit for bit, on every compiled
    indexer shape, and against the oracle's incremental scores."""
    torch = need_gpu()
    import oracle
    if kind == "paged":
        w = _paged()
    elif kind == "shared_history":
        w = wl.chunked_prefill_100000(n=12, first=9000)
    elif kind == "idx4x32":
        w = wl.make_workload("inc4", [7777, 4100, 12], idx_heads=4, idx_dim=32, q_heads=4,
                             kv_heads=4, head_dim=64, seed=72, slots="permutation")
    elif kind == "idx8x32":
        w = wl.make_workload("inc8x32", [6001, 4099, 513, 3], idx_heads=8, idx_dim=32, q_heads=8,
                             kv_heads=2, head_dim=64, seed=73, slots="paged16")
    else:
        w = wl.make_workload("inc4x64", [8191, 1030, 77], idx_heads=4, idx_dim=64, q_heads=2,
                             kv_heads=2, head_dim=64, seed=74, slots="identity")
    db = _batch(w)
    db.score()
    torch.cuda.synchronize()
    raw = db.scores.cpu().numpy().copy()
    db.scores.fill_(float("nan"))
    db.pool_all()
    db.score_pooled()
    assert db.check_errors() == (0, 0)
    pooled = db.scores.cpu().numpy()
    for b in range(w.batch):
        G = int(w.visible[b]) // 4
        assert pooled[b, :G].tobytes() == raw[b, :G].tobytes(), b
    # and the oracle's incremental scores, for one query
    b = 0
    ko, T = int(w.key_offset[b]), int(w.visible[b])
    ref = oracle.score_groups_incremental(w.q_idx[b], w.idx_keys[ko:ko + T], T)
    assert pooled[b, :T // 4].tobytes() == ref.tobytes()


def test_decode_steps_append_groups_and_match_full_raw():
    """A decode loop: T grows one token per step; whenever a group completes,
    only that group is pooled (max_groups = 1); every step's rows and outputs
    equal the full-raw path's bit for bit."""
    torch = need_gpu()
    T0 = [8190, 2047, 30001]
    steps = 9
    w = wl.make_workload("steps", [t + steps for t in T0], idx_heads=8, idx_dim=64, q_heads=16,
                         kv_heads=2, head_dim=128, seed=73, slots="ring", ring_size=40000,
                         ring_shift=12345)
    db = _batch(w)
    T = np.array(T0, np.int32)
    db.visible.copy_(torch.from_numpy(T))
    G = T // 4
    db.pool(np.zeros_like(G), G)
    for step in range(steps + 1):
        db.decode()
        torch.cuda.synchronize()
        ids, n, out = db.ids.cpu().numpy().copy(), db.n_ids.cpu().numpy().copy(), db.out.cpu().numpy().copy()
        db.out.fill_(float("nan"))
        db.decode_pooled()
        assert db.check_errors() == (0, 0)
        assert np.array_equal(db.n_ids.cpu().numpy(), n)
        for b in range(w.batch):
            assert db.ids.cpu().numpy()[b, :n[b]].tobytes() == ids[b, :n[b]].tobytes(), (step, b)
        assert db.out.cpu().numpy().tobytes() == out.tobytes(), step
        if step == steps:
            break
        T = T + 1
        db.visible.copy_(torch.from_numpy(T))
        G_new = T // 4
        if np.any(G_new > G):
            db.pool(G, G_new)  # only the groups completed by this token
            G = G_new


def test_pooling_in_pieces_equals_at_once():
    torch = need_gpu()
    w = _paged()
    db = _batch(w)
    db.pool_all()
    torch.cuda.synchronize()
    once = db.pooled.cpu().numpy().copy()
    db.pooled.zero_()
    G = (w.visible // 4).astype(np.int32)
    owner = db._pool_owner
    cut = (G // 3).astype(np.int32)
    db.pool(np.zeros_like(G), np.where(owner, cut, 0))
    db.pool(np.where(owner, cut, 0), np.where(owner, G, 0))
    assert db.check_errors() == (0, 0)
    assert db.pooled.cpu().numpy().tobytes() == once.tobytes()


def test_pool_groups_flags_bad_ranges():
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = _paged()
    db = _batch(w)
    dev = db.q.device
    g_max = int(db.dims.max_visible) // 4
    B = w.batch

    def call(begin, end, max_groups):
        gb = torch.tensor(begin, dtype=torch.int32, device=dev)
        ge = torch.tensor(end, dtype=torch.int32, device=dev)
        qsa.qsa_pool_groups(db.dims, db.inputs, gb, ge, max_groups, db.pooled, db.pool_offset, db.ws)
        return db.check_errors()

    # a range ending past max_visible / 4: skipped and flagged on the device
    st, flags = call([g_max - 1] + [0] * (B - 1), [g_max + 1] + [0] * (B - 1), 2)
    assert st == qsa.QSA_ERR_DEVICE_FAULT and flags & qsa.QSA_DEVERR_VISIBLE_RANGE
    # a range longer than the max_groups the call was sized for: the same
    st, flags = call([0] * B, [2] + [0] * (B - 1), 1)
    assert st == qsa.QSA_ERR_DEVICE_FAULT and flags & qsa.QSA_DEVERR_VISIBLE_RANGE
    # a host-side max_groups above max_visible / 4 is rejected before any launch
    with pytest.raises(qsa.QsaError):
        call([0] * B, [0] * B, g_max + 1)
    # nothing was written by the rejected ranges
    assert db.check_errors() == (0, 0)
    assert float(db.pooled.abs().sum()) == 0.0


def test_decode_pooled_full_size_long_262144():
    """The benchmark workload: 8 queries x 262,144 tokens, cache of 65,536
    pooled keys per query; rows and outputs equal the full-raw decode's."""
    torch = need_gpu()
    w = wl.long_262144()
    db = _batch(w)
    db.decode()
    torch.cuda.synchronize()
    ids, out = db.ids.cpu().numpy().copy(), db.out.cpu().numpy().copy()
    db.pool_all()
    db.out.fill_(float("nan"))
    db.decode_pooled()
    assert db.check_errors() == (0, 0)
    assert db.ids.cpu().numpy().tobytes() == ids.tobytes()
    assert db.out.cpu().numpy().tobytes() == out.tobytes()
