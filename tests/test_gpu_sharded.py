"""The attention state of a slice of the emitted row (qsa_attend_state), and
one history split across ranks with every device step on the GPU.

"Top-k chooses the set; time chooses the order" (AFN-017) fixes the chosen
set and its chronological order; "Floating point makes order observable"
asks for one canonical order of the softmax.  When one history is split
across ranks by contiguous group ranges, each rank scores and chooses among
its own groups, the candidates are merged on the host with the same tie rule,
every rank attends to its contiguous slice of the emitted row, and the
slices' states are merged in row order.  Here the ranks run one after
another on one GPU (independent launches, nothing waits on another); the
host logic is the one the gloo tests run across processes.
"""
import dataclasses

import numpy as np
import pytest

from gpu_helpers import ATTN_TOL, need_gpu
from top_group_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _shapes():
    return [dict(idx_heads=8, idx_dim=64, q_heads=16, kv_heads=2, head_dim=128),
            dict(idx_heads=4, idx_dim=32, q_heads=4, kv_heads=4, head_dim=64)]


def _states(db, rows, counts, device=False):
    """qsa_attend_state over rows [B, <= row_cap] with counts [B]: (acc, m, l)
    as host arrays, or as the device tensors when device=True."""
    import torch
    from top_group_sparse_gb300 import qsa
    B = db.dims.batch
    ids = torch.full((B, db.row_cap), -1, dtype=torch.int32, device="cuda")
    for b in range(B):
        n = int(counts[b])
        if n:
            ids[b, :n] = torch.from_numpy(np.ascontiguousarray(rows[b][:n], np.int32)).cuda()
    n_ids = torch.from_numpy(np.asarray(counts, np.int32)).cuda()
    acc = torch.full((B, db.w.q_heads, db.w.head_dim), float("nan"), dtype=torch.float32, device="cuda")
    m = torch.full((B, db.w.q_heads), float("nan"), dtype=torch.float32, device="cuda")
    l = torch.full_like(m, float("nan"))
    qsa.qsa_attend_state(db.dims, db.inputs, ids, n_ids, acc, m, l, db.ws)
    assert db.check_errors() == (0, 0)
    if device:
        return acc, m, l
    return acc.cpu().numpy(), m.cpu().numpy(), l.cpu().numpy()


def _vmax(w, b, ids):
    slots = w.slot_map[w.slot_offset[b] + np.asarray(ids, np.int64)]
    return float(np.abs(w.v_cache[slots]).max()) if len(slots) else 1.0


@pytest.mark.parametrize("shape", range(2))
def test_state_of_the_whole_row_is_the_decode_output(shape):
    """acc / l of the whole emitted row is qsa_decode's output bit for bit
    (the same runs, the same merge, the same division), and so is that one
    state passed through qsa_merge_states; an empty row gives the empty state
    (m = -inf, l = 0, acc = 0) and a zero output."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.make_workload("state", [9001, 37, 2052, 0, 40003], seed=81, slots="paged16", **_shapes()[shape])
    db = qsa.DeviceBatch(w)
    db.decode()
    torch.cuda.synchronize()
    ids, n, out = db.ids.cpu().numpy(), db.n_ids.cpu().numpy(), db.out.cpu().numpy()
    acc_d, m_d, l_d = _states(db, ids, n, device=True)
    acc, m, l = acc_d.cpu().numpy(), m_d.cpu().numpy(), l_d.cpu().numpy()
    from top_group_sparse_gb300 import sharding as sh
    one = sh.merge_states(db.dims, [(m_d, l_d, acc_d)])
    torch.cuda.synchronize()
    assert one.cpu().numpy().tobytes() == out.tobytes()
    for b in range(w.batch):
        if n[b] == 0:
            assert np.all(m[b] == -np.inf) and np.all(l[b] == 0) and not acc[b].any()
            continue
        assert np.all(l[b] > 0) and np.all(np.isfinite(m[b]))
        got = (acc[b] / l[b][:, None]).astype(np.float32)
        assert got.tobytes() == out[b].tobytes(), b


def test_row_slices_merge_to_the_row_attention():
    """Consecutive slices of each query's row (empty ones included), each
    attended on its own: every slice's state matches the oracle's state of
    that slice, and the states merged in row order by qsa_merge_states give
    the row's attention within 1e-5 * max|V| of the oracle."""
    need_gpu()
    import oracle
    from top_group_sparse_gb300 import qsa
    from top_group_sparse_gb300 import sharding as sh
    w = wl.make_workload("slices", [40003, 2051, 9001], seed=82, slots="paged16", **_shapes()[0])
    ref = oracle.decode(w)
    db = qsa.DeviceBatch(w)
    rows = [ref["ids"][b, :ref["n_ids"][b]] for b in range(w.batch)]
    cuts = [[0, len(r) // 3, len(r) // 3, min(len(r), (2 * len(r)) // 3 + 5), len(r)] for r in rows]
    n_sl = len(cuts[0]) - 1
    states = []
    for s in range(n_sl):
        sl = [rows[b][cuts[b][s]:cuts[b][s + 1]] for b in range(w.batch)]
        states.append((sl, _states(db, sl, [len(x) for x in sl], device=True)))
    merged_all = sh.merge_states(db.dims, [(m, l, acc) for _, (acc, m, l) in states]).cpu().numpy()
    states = [(sl, tuple(t.cpu().numpy() for t in st)) for sl, st in states]
    for b in range(w.batch):
        vmax = _vmax(w, b, rows[b])
        slots_all = w.slot_map[w.slot_offset[b] + rows[b].astype(np.int64)]
        for s, (sl, (acc, m, l)) in enumerate(states):
            n = len(sl[b])
            pm, pl, pacc = oracle.attend_partial(w.q[b], w.k_cache, w.v_cache,
                                                 slots_all[cuts[b][s]:cuts[b][s + 1]], w.scale)
            if n == 0:
                assert np.all(m[b] == -np.inf) and np.all(l[b] == 0) and not acc[b].any()
                continue
            assert np.abs(m[b] - pm).max() <= 1e-5 * max(1.0, float(np.abs(pm).max())), (b, s)
            assert np.abs(l[b] / pl - 1.0).max() <= 1e-5, (b, s)
            err = np.abs(acc[b] / l[b][:, None] - pacc / pl[:, None]).max() / vmax
            assert err <= ATTN_TOL, (b, s, err)
        err = float(np.abs(merged_all[b].astype(np.float64) - ref["out"][b]).max()) / vmax
        assert err <= ATTN_TOL, (b, err)


@pytest.mark.parametrize("world", [2, 3])
def test_one_history_across_ranks_on_the_gpu(world):
    """Each rank scores its contiguous group range (qsa_score_groups on its
    shard of the keys; the last rank holds the raw tail) and chooses its local
    set (qsa_select on the shard); the host merges the candidates with the
    tie rule; each rank attends to its slice of the emitted row
    (qsa_attend_state) and the states are merged in rank order.  The row
    equals the oracle's single-history row bit for bit, the local sets equal
    the host rule's, and the output is within 1e-5 * max|V| of the oracle."""
    torch = need_gpu()
    import oracle
    from top_group_sparse_gb300 import qsa
    from top_group_sparse_gb300 import sharding as sh
    T = 4 * 3001 + 2
    w = wl.make_workload("one", [T], seed=83, slots="paged16", **_shapes()[0])
    ref = oracle.decode(w)
    G = T // 4
    parts, ranges = [], []
    for r in range(world):
        rg = sh.shard_groups(G, world, r)
        last = r == world - 1
        k_hi = T if last else 4 * rg.stop
        shard = dataclasses.replace(w, key_offset=w.key_offset + 4 * rg.start,
                                    visible=np.array([k_hi - 4 * rg.start], np.int32))
        db = qsa.DeviceBatch(shard)
        db.score()
        db.select()
        torch.cuda.synchronize()
        assert db.check_errors() == (0, 0)
        G_r = rg.stop - rg.start
        scores = db.scores[0, :G_r].cpu().numpy()
        k = min(w.budget, G_r)
        local = db.ids[0, :4 * k:4].cpu().numpy().astype(np.int64) // 4  # chosen groups, ascending
        keys, groups = sh.local_candidates(scores, rg.start, w.budget)
        assert np.array_equal(np.sort(groups), local + rg.start), r
        parts.append((sh.order_keys(scores[local]), local + rg.start))
        ranges.append((rg, last))
        del db
    chosen = sh.merge_candidates(parts, w.budget, G)
    row = sh.emitted_row(chosen, T)
    assert row.tobytes() == ref["ids"][0, :ref["n_ids"][0]].tobytes()
    db = qsa.DeviceBatch(w)
    states = []
    for rg, last in ranges:
        sl = row[sh.rank_rows(row, rg.start, rg.stop, last)]
        acc, m, l = _states(db, [sl], [len(sl)], device=True)
        states.append((m, l, acc))
    out = sh.merge_states(db.dims, states).cpu().numpy()[0]
    err = float(np.abs(out.astype(np.float64) - ref["out"][0]).max()) / _vmax(w, 0, row)
    assert err <= ATTN_TOL, err
