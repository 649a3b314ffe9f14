"""Property tests of the host logic that splits one history across ranks
("Top-k chooses the set; time chooses the order", Decision and Tie handling
belongs to membership; "Floating point makes order observable"): for random
histories, tie patterns, budgets, rank counts and row cuts, the merged choice
equals the oracle's single-history selection bit for bit, every rank's slice
is contiguous and in rank order, and the merged attention states equal the
one-pass oracle within 1e-5 * max|V|."""
import numpy as np
import pytest

hypothesis = pytest.importorskip("hypothesis")
st = hypothesis.strategies
given, settings = hypothesis.given, hypothesis.settings


def _scores(seed, G, levels):
    rng = np.random.default_rng(seed)
    if levels == 0:
        return np.abs(rng.standard_normal(G)).astype(np.float32)
    # few distinct values: heavy ties, including +0 (ReLU's floor)
    return (rng.integers(0, levels, G) / 4.0).astype(np.float32)


@settings(max_examples=300, deadline=None, derandomize=True)
@given(T=st.integers(0, 3000), budget=st.integers(1, 600), world=st.integers(1, 7),
       levels=st.sampled_from([0, 1, 2, 5]), seed=st.integers(0, 2**31 - 1))
def test_sharded_choice_equals_the_oracle(T, budget, world, levels, seed):
    import oracle
    from top_group_sparse_gb300 import sharding as sh
    G = T // 4
    x = _scores(seed, G, levels)
    ref_ids, ref_chosen = oracle.select(x, T, budget, return_chosen=True)
    parts, spans = [], []
    for r in range(world):
        rg = sh.shard_groups(G, world, r)
        parts.append(sh.local_candidates(x[rg.start:rg.stop], rg.start, budget))
        spans.append((rg, r == world - 1))
    rng = np.random.default_rng(seed + 1)
    chosen = sh.merge_candidates([parts[i] for i in rng.permutation(world)], budget, G)
    assert chosen.astype(np.int32).tobytes() == ref_chosen.tobytes()
    row = sh.emitted_row(chosen, T)
    assert row.tobytes() == ref_ids.tobytes()
    # the ranks' slices tile the row in rank order, each holding only its own tokens
    pos = 0
    for rg, last in spans:
        sl = sh.rank_rows(row, rg.start, rg.stop, last)
        assert sl.start == pos
        pos = sl.stop
        own = row[sl]
        hi = T if last else 4 * rg.stop
        assert np.all((own >= 4 * rg.start) & (own < hi))
    assert pos == row.size


@settings(max_examples=120, deadline=None, derandomize=True)
@given(n=st.integers(0, 700), cuts=st.lists(st.integers(0, 700), max_size=5),
       gq=st.sampled_from([1, 2, 8]), seed=st.integers(0, 2**31 - 1))
def test_states_of_row_cuts_merge_to_the_one_pass_softmax(n, cuts, gq, seed):
    import oracle
    from top_group_sparse_gb300 import sharding as sh
    rng = np.random.default_rng(seed)
    n_kv, d, S = 2, 32, 800
    q = rng.standard_normal((n_kv * gq, d)).astype(np.float32)
    kc = rng.standard_normal((S, n_kv, d)).astype(np.float32)
    vc = rng.standard_normal((S, n_kv, d)).astype(np.float32)
    slots = rng.permutation(S)[:n].astype(np.int32)
    scale = 1.0 / np.sqrt(d)
    ref = oracle.attend(q, kc, vc, slots, scale)
    bounds = [0] + sorted(min(c, n) for c in cuts) + [n]
    parts = [oracle.attend_partial(q, kc, vc, slots[a:b], scale) for a, b in zip(bounds, bounds[1:])]
    got = oracle.merge_states(parts)
    if n == 0:
        assert not got.any()
        return
    tol = 1e-5 * float(np.abs(vc[slots]).max())
    assert float(np.abs(got.astype(np.float64) - ref).max()) <= tol
