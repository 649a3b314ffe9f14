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
