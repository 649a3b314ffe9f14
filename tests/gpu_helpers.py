"""Shared plumbing of the GPU parity tests: run the library through its C ABI
on a workload and compare every stage with the CPU oracle.

The bar (from the method's contract): group scores and selected ID rows
bit-exact; the gathered K/V scratch bit-exact (a pure copy); attention
within max|delta| <= 1e-5 * max|V| of the oracle, V taken over the query's
selected rows; every run bit-identical to the previous one.
"""
import numpy as np
import pytest

ATTN_TOL = 1e-5


def need_gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from top_group_sparse_gb300 import build
    build.build()
    return torch


def run_stages(w, budget=None, stream=None):
    """Score -> select -> gather -> attend through the four split entry points."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    db = qsa.DeviceBatch(w, budget=budget)
    db.score(stream)
    db.select(stream)
    db.gather(stream)
    db.attend(stream)
    st, flags = db.check_errors(stream)
    res = _fetch(db)
    res.update(status=st, flags=flags, batch=db)
    return res


def run_decode(w, budget=None, stream=None, db=None):
    need_gpu()
    from top_group_sparse_gb300 import qsa
    db = db or qsa.DeviceBatch(w, budget=budget)
    db.decode(stream)
    st, flags = db.check_errors(stream)
    res = _fetch(db, with_scratch=False)
    res.update(status=st, flags=flags, batch=db)
    return res


def _fetch(db, with_scratch=True):
    import torch
    torch.cuda.synchronize()
    r = {"ids": db.ids.cpu().numpy(), "n_ids": db.n_ids.cpu().numpy(), "out": db.out.cpu().numpy()}
    if with_scratch:
        r["scores"] = db.scores.cpu().numpy()
        r["k_scr"] = db.k_scr.cpu().numpy()
        r["v_scr"] = db.v_scr.cpu().numpy()
    return r


def oracle_run(w, budget=None, queries=None):
    import dataclasses
    import oracle
    if budget is not None:
        w = dataclasses.replace(w, budget=budget)
    return oracle.decode(w, with_scores=True, queries=queries)


def assert_ids_equal(w, gpu, ref, queries=None):
    qs = range(w.batch) if queries is None else queries
    for j, b in enumerate(qs):
        n = int(ref["n_ids"][j])
        assert int(gpu["n_ids"][b]) == n, f"query {b}: n {gpu['n_ids'][b]} != {n}"
        g = gpu["ids"][b, :n]
        o = ref["ids"][j, :n]
        if g.tobytes() != o.tobytes():
            bad = np.flatnonzero(g != o)
            raise AssertionError(f"query {b}: {len(bad)} ID mismatches, first at {bad[0]}: "
                                 f"gpu {g[bad[0]]} oracle {o[bad[0]]}")


def assert_scores_equal(w, gpu, ref, queries=None):
    qs = range(w.batch) if queries is None else queries
    for j, b in enumerate(qs):
        G = int(w.visible[b]) // 4
        g = gpu["scores"][b, :G]
        o = ref["scores"][j, :G]
        if g.tobytes() != o.tobytes():
            bad = np.flatnonzero(g.view(np.uint32) != o.view(np.uint32))
            raise AssertionError(f"query {b}: {len(bad)} score mismatches, first group {bad[0]}: "
                                 f"gpu {g[bad[0]]!r} oracle {o[bad[0]]!r}")


def assert_gather_exact(w, gpu, queries=None):
    qs = range(w.batch) if queries is None else queries
    for b in qs:
        n = int(gpu["n_ids"][b])
        ids = gpu["ids"][b, :n]
        slots = w.slot_map[w.slot_offset[b] + ids]
        assert gpu["k_scr"][b, :n].tobytes() == w.k_cache[slots].tobytes(), f"K rows, query {b}"
        assert gpu["v_scr"][b, :n].tobytes() == w.v_cache[slots].tobytes(), f"V rows, query {b}"


def assert_attention_close(w, gpu, ref, queries=None, tol=ATTN_TOL):
    qs = range(w.batch) if queries is None else queries
    worst = 0.0
    for j, b in enumerate(qs):
        n = int(ref["n_ids"][j])
        o = ref["out"][j]
        g = gpu["out"][b]
        assert np.all(np.isfinite(g)), f"query {b}: non-finite output"
        if n == 0:
            assert np.all(g == 0), f"query {b}: empty row must give zeros"
            continue
        slots = w.slot_map[w.slot_offset[b] + ref["ids"][j, :n]]
        vmax = float(np.abs(w.v_cache[slots]).max())
        err = float(np.abs(g.astype(np.float64) - o).max()) / vmax
        worst = max(worst, err)
        assert err <= tol, f"query {b}: max|delta|/max|V| = {err:.3e} > {tol:.0e}"
    return worst


def full_parity(w, gpu, ref, queries=None, scores=True, gather=True):
    if scores:
        assert_scores_equal(w, gpu, ref, queries)
    assert_ids_equal(w, gpu, ref, queries)
    if gather:
        assert_gather_exact(w, gpu, queries)
    return assert_attention_close(w, gpu, ref, queries)
