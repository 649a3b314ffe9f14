"""The multi-rank path on CPU: two gloo ranks each decode their shard of a
batch with the CPU oracle; gathered, the shards equal the whole batch bit for
bit (queries are independent, no exchange on the data path), and the
max-over-ranks timing reduction picks the slowest rank."""
import os
import socket

import numpy as np
import pytest
import torch.multiprocessing as mp

from top_group_sparse_gb300.sharding import shard_queries


def test_shard_queries_partition():
    for n in (0, 1, 7, 8, 256):
        for world in (1, 2, 3, 8):
            parts = [shard_queries(n, world, r) for r in range(world)]
            flat = [q for p in parts for q in p]
            assert flat == list(range(n))
            sizes = [len(p) for p in parts]
            assert max(sizes) - min(sizes) <= 1
    with pytest.raises(ValueError):
        shard_queries(4, 2, 2)


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out_dir):
    import torch
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from top_group_sparse_gb300 import workloads as wl
    from top_group_sparse_gb300.sharding import max_over_ranks, shard_queries
    w = wl.make_workload("shard", [4 * 700 + 1, 37, 2052, 3001, 0, 9000], idx_heads=4,
                         idx_dim=32, q_heads=4, kv_heads=2, head_dim=64, seed=17,
                         slots="paged16")
    mine = list(shard_queries(w.batch, world, rank))
    res = oracle.decode(w, queries=mine)
    parts = [None] * world
    dist.all_gather_object(parts, {"q": mine, "ids": res["ids"], "n": res["n_ids"],
                                   "out": res["out"]})
    slowest = max_over_ranks(1.0 + rank)
    if rank == 0:
        full = oracle.decode(w)
        qs = [q for p in parts for q in p["q"]]
        assert qs == list(range(w.batch))
        ids = np.concatenate([p["ids"] for p in parts])
        out = np.concatenate([p["out"] for p in parts])
        n = np.concatenate([p["n"] for p in parts])
        ok = (ids.tobytes() == full["ids"].tobytes() and out.tobytes() == full["out"].tobytes()
              and n.tobytes() == full["n_ids"].tobytes() and slowest == float(world))
        open(os.path.join(out_dir, "ok"), "w").write("1" if ok else "0")
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_shard_the_batch(tmp_path):
    import oracle
    oracle.lib()  # build once before the ranks start
    world = 2
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    assert (tmp_path / "ok").read_text() == "1"


# ---- one long history split across ranks by group ranges ---------------------

def test_shard_groups_partition():
    from top_group_sparse_gb300.sharding import shard_groups
    for n in (0, 3, 513, 65536):
        for world in (1, 2, 5):
            parts = [shard_groups(n, world, r) for r in range(world)]
            assert [g for p in parts for g in p] == list(range(n))


def _sharded_choice(scores, T, budget, world):
    from top_group_sparse_gb300 import sharding as sh
    G = T // 4
    parts = []
    for r in range(world):
        rg = sh.shard_groups(G, world, r)
        parts.append(sh.local_candidates(scores[rg.start:rg.stop], rg.start, budget))
    chosen = sh.merge_candidates(parts[::-1], budget, G)  # arrival order does not matter
    return chosen, sh.emitted_row(chosen, T)


@pytest.mark.parametrize("T", [0, 5, 2051, 2052, 2055, 9001, 40003])
def test_sharded_selection_equals_one_device(T):
    """The merged set and row equal the oracle's single-history selection
    bit for bit, for any number of ranks (including ranks with fewer groups
    than the budget, or none), with heavy ties across range boundaries."""
    import oracle
    rng = np.random.default_rng(T + 7)
    G = T // 4
    for values in ("normal", "ties"):
        x = np.abs(rng.standard_normal(G)).astype(np.float32)
        if values == "ties":
            x = (np.round(x * 2.0) / 2.0).astype(np.float32)  # a few distinct values, many equal
        for budget in (1, 7, 512):
            ref_ids, ref_chosen = oracle.select(x, T, budget, return_chosen=True)
            for world in (1, 2, 3, 5):
                chosen, row = _sharded_choice(x, T, budget, world)
                assert chosen.astype(np.int32).tobytes() == ref_chosen.tobytes(), (values, budget, world)
                assert row.tobytes() == ref_ids.tobytes(), (values, budget, world)


def test_sharded_selection_rejects_short_candidate_lists():
    from top_group_sparse_gb300 import sharding as sh
    keys, groups = sh.local_candidates(np.ones(10, np.float32), 0, 4)
    with pytest.raises(ValueError):
        sh.merge_candidates([(keys, groups)], 8, 20)
    with pytest.raises(ValueError):
        sh.order_keys(np.array([1.0, -1.0], np.float32))


def test_partial_states_merge_to_the_sequential_softmax():
    """Per-rank online-softmax states over consecutive slices of the row,
    merged in rank order: within 1e-5 * max|V| of the one-pass oracle (the
    merge re-associates the rescaling), bit-identical for one slice, and
    empty slices contribute nothing."""
    import oracle
    from top_group_sparse_gb300 import sharding as sh
    rng = np.random.default_rng(3)
    n_q, n_kv, d, S = 4, 2, 64, 600
    q = rng.standard_normal((n_q, d)).astype(np.float32)
    kc = rng.standard_normal((S, n_kv, d)).astype(np.float32)
    vc = rng.standard_normal((S, n_kv, d)).astype(np.float32)
    slots = rng.permutation(S)[:513].astype(np.int32)
    scale = 1.0 / np.sqrt(d)
    ref = oracle.attend(q, kc, vc, slots, scale)
    one = oracle.merge_states([oracle.attend_partial(q, kc, vc, slots, scale)])
    assert one.tobytes() == ref.tobytes()
    tol = 1e-5 * float(np.abs(vc).max())
    for cuts in ([0, 513], [0, 200, 513], [0, 0, 100, 100, 400, 513], [0, 513, 513]):
        parts = [oracle.attend_partial(q, kc, vc, slots[a:b], scale) for a, b in zip(cuts, cuts[1:])]
        got = oracle.merge_states(parts)
        assert float(np.abs(got - ref).max()) <= tol, cuts
    empty = oracle.merge_states([oracle.attend_partial(q, kc, vc, slots[:0], scale)])
    assert not empty.any()


def _one_history_worker(rank, world, port, out_dir):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import oracle
    from top_group_sparse_gb300 import sharding as sh
    from top_group_sparse_gb300 import workloads as wl
    ok = True
    for T, values in ((4 * 3001 + 2, "normal"), (4 * 1500, "grid8")):
        w = wl.make_workload("one", [T], idx_heads=4, idx_dim=32, q_heads=4, kv_heads=2,
                             head_dim=64, seed=19, slots="paged16", index_values=values)
        G = T // 4
        rg = sh.shard_groups(G, world, rank)
        last = rank == world - 1
        # this rank's keys: its groups (and, on the last rank, the tail)
        k_hi = T if last else 4 * rg.stop
        keys = w.idx_keys[4 * rg.start:k_hi]
        sc = oracle.score_groups(w.q_idx[0], keys, k_hi - 4 * rg.start)[:len(rg)]
        cand = sh.local_candidates(sc, rg.start, w.budget)
        allc = [None] * world
        dist.all_gather_object(allc, cand)  # the one exchange of the selection
        ids = sh.emitted_row(sh.merge_candidates(allc, w.budget, G), T)
        mine = ids[sh.rank_rows(ids, rg.start, rg.stop, last)]
        st, slots = oracle.resolve(mine, w.slot_map[int(w.slot_offset[0]):], w.num_slots)
        assert st == 0
        part = oracle.attend_partial(w.q[0], w.k_cache, w.v_cache, slots, w.scale)
        parts = [None] * world
        dist.all_gather_object(parts, (rank, part))
        out = oracle.merge_states([p for _, p in sorted(parts, key=lambda x: x[0])])
        if rank == 0:
            ref = oracle.decode(w)
            n = int(ref["n_ids"][0])
            tol = 1e-5 * float(np.abs(w.v_cache).max())
            ok &= ids.tobytes() == ref["ids"][0, :n].tobytes()
            ok &= float(np.abs(out - ref["out"][0]).max()) <= tol
    if rank == 0:
        open(os.path.join(out_dir, "ok"), "w").write("1" if ok else "0")
    dist.barrier()
    dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_gloo_ranks_shard_one_history(tmp_path, world):
    """One query's history split across gloo ranks by group ranges: scores,
    local candidates, one all-gather, merged set, per-rank attention states
    merged in rank order -- the row equals the single-device oracle's bit for
    bit, the output within 1e-5 * max|V|."""
    import oracle
    oracle.lib()
    mp.spawn(_one_history_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    assert (tmp_path / "ok").read_text() == "1"
