"""Pins of the CPU oracle against what the notes and the mathematics fix.

Each test checks the oracle against something other than itself: values the
notes state (fixtures under tests/golden/), closed forms on an exact integer
grid, brute-force enumeration, float64 definitions written independently in
numpy, and invariants the notes name.  The notes are
"Top-k chooses the set; time chooses the order" (AFN-017) and
"A sparse mask is not sparse attention" (AFN-016).
"""
import itertools
import os

import numpy as np
import pytest

from top_group_sparse_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
U32 = 2.0 ** -24  # unit roundoff of binary32


def gamma(n):
    return n * U32 / (1 - n * U32)


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line)
    return rows


# ---------------------------------------------------------------- row shape

def test_golden_row_structure(oracle):
    """AFN-016 Decision: <= 512 groups + <= 3 tail = 2,051 keys; AFN-017
    Decision: expand each group to 4 consecutive IDs, append the tail."""
    rows = _golden_rows("row_structure.txt")
    assert len(rows) >= 15
    for r in rows:
        T, G, tail, W = map(int, r.split())
        assert oracle.num_groups(T) == G
        assert oracle.tail_len(T) == tail
        assert oracle.row_width(T, 512) == W
        assert W <= 2051


@pytest.mark.parametrize("T", [0, 1, 3, 4, 7, 37, 2051, 2052, 2053, 2055, 4099, 9000])
def test_emitted_row_invariants(oracle, T):
    """AFN-017 Tie handling...: chronological emission, group-contiguous
    expansion, raw-tail placement -- on N(0,1) scores."""
    rng = np.random.default_rng(T)
    G = T // 4
    scores = rng.standard_normal(G).astype(np.float32)
    ids, chosen = oracle.select(scores, T, 512, return_chosen=True)
    k = min(G, 512)
    assert len(ids) == 4 * k + T % 4
    assert np.all(np.diff(ids) > 0)                       # strictly increasing
    body = ids[:4 * k].reshape(k, 4)
    assert np.all(body[:, 0] % 4 == 0)                    # groups aligned at 4g
    assert np.all(body - body[:, :1] == np.arange(4))     # 4 consecutive IDs
    assert np.array_equal(body[:, 0] // 4, chosen)        # the chosen groups
    assert np.array_equal(ids[4 * k:], np.arange(4 * G, T))  # tail last, in order
    assert np.all(ids < T) and np.all(ids >= 0)


# ------------------------------------------------------------ selection rule

def test_golden_tie_cases(oracle):
    """Hand-worked cases of (score desc, position asc) membership."""
    for r in _golden_rows("tie_cases.txt"):
        b, s, c = [x.strip() for x in r.split("|")]
        budget = int(b)
        scores = np.array([float(x) for x in s.split()], np.float32)
        want = [int(x) for x in c.split()]
        T = 4 * len(scores)
        ids, chosen = oracle.select(scores, T, budget, return_chosen=True)
        assert chosen.tolist() == want, r
        assert ids.tolist() == [4 * g + u for g in want for u in range(4)], r


def _brute_force_set(scores, k):
    """The unique k-subset whose every member beats every non-member under
    the rule 'higher score wins, equal scores: smaller position wins'."""
    G = len(scores)
    beats = lambda a, b: scores[a] > scores[b] or (scores[a] == scores[b] and a < b)
    found = []
    for S in itertools.combinations(range(G), k):
        rest = [g for g in range(G) if g not in S]
        if all(beats(a, b) for a in S for b in rest):
            found.append(S)
    assert len(found) == 1
    return list(found[0])


def test_brute_force_topk_tiny(oracle):
    """Every budget 1..G on tiny inputs with heavy ties, every tail length,
    against explicit subset enumeration (AFN-017 Decision)."""
    rng = np.random.default_rng(7)
    cases = 0
    for G in range(1, 11):
        for trial in range(6):
            levels = 1 + trial % 4           # 1 level = everything ties
            scores = rng.integers(0, levels, G).astype(np.float32) / 4
            for k in range(1, G + 1):
                want = _brute_force_set(scores.tolist(), k)
                for tail in range(4):
                    T = 4 * G + tail
                    ids, chosen = oracle.select(scores, T, k, return_chosen=True)
                    assert chosen.tolist() == want
                    assert ids.tolist() == [4 * g + u for g in want for u in range(4)] + \
                        list(range(4 * G, T))
                    cases += 1
    assert cases > 1000


def test_tie_rule_is_applied_in_membership(oracle):
    """All scores equal and over budget: membership is the first 512 groups
    (smaller positions), never a later tie (AFN-017 Tie handling...)."""
    G = 600
    for value in (0.0, 1.5):
        ids, chosen = oracle.select(np.full(G, value, np.float32), 4 * G + 2, 512,
                                    return_chosen=True)
        assert chosen.tolist() == list(range(512))
        assert ids[-2:].tolist() == [4 * G, 4 * G + 1]


def test_select_negative_zero_ties_positive_zero(oracle):
    """-0 and +0 compare equal, so they tie and position decides."""
    scores = np.array([-0.0, 0.0, -0.0, 1.0], np.float32)
    _, chosen = oracle.select(scores, 16, 2, return_chosen=True)
    assert chosen.tolist() == [0, 3]


# ------------------------------------------------------------------- scores

def _grid_ints(w):
    """Integer numerators of the k/8 grid values (exact)."""
    qi = np.rint(w.q_idx * 8).astype(np.int64)
    ki = np.rint(w.idx_keys * 8).astype(np.int64)
    assert np.array_equal(qi / 8, w.q_idx) and np.array_equal(ki / 8, w.idx_keys)
    return qi, ki


def _closed_form_scores_x256(qi_b, ki, T):
    """256 * sum_h ReLU(q_h . mean(k_4g..k_4g+3)) in exact integer arithmetic:
    q = a/8, k = c/8, pooled = (sum of 4 c)/32, dot = sum a*(sum c) / 256."""
    G = T // 4
    csum = ki[:4 * G].reshape(G, 4, -1).sum(axis=1)          # [G, d] = 32 * pooled
    dots = csum @ qi_b.T                                     # [G, H] = 256 * dot
    return np.maximum(dots, 0).sum(axis=1)                   # [G]


def test_scores_exact_on_integer_grid(oracle):
    """AFN-016 Why a sparse mask can still be dense: sum(ReLU(dot_h)) over a
    pooled group key.  On the k/8 grid every FP32 step is exact, so 256*score
    must equal the integer closed form exactly -- a dropped term, wrong sign,
    wrong index, a ReLU after the head sum or a missing 1/4 all fail here."""
    w = wl.dense_parity_sweep()
    qi, ki = _grid_ints(w)
    T = int(w.visible.max())
    checked = 0
    for b in range(w.batch):
        s = oracle.score_groups(w.q_idx[b], w.idx_keys, T)
        want = _closed_form_scores_x256(qi[b], ki, T)
        assert np.array_equal((s.astype(np.float64) * 256).astype(np.int64), want)
        assert np.array_equal(s.astype(np.float64) * 256, want.astype(np.float64))
        checked += len(s)
    # the grid produces many exact ties, which is what makes the sweep useful
    assert checked == 12 * 513
    s0 = oracle.score_groups(w.q_idx[0], w.idx_keys, T)
    assert len(np.unique(s0)) < len(s0)


def test_non_finite_keys_follow_the_relu_reading(oracle):
    """Non-finite index keys.  The pages are silent on them; the reading is
    ReLU(x) = x > 0 ? x : +0, so scores lie in [+0, +inf].  With positive
    query weights: a +inf pooled element gives +inf dots and a +inf score, a
    -inf one -inf dots and ReLU +0, NaN (a NaN key, or +inf and -inf pooled
    together) ReLU +0.  The selection ranks +inf above every finite score and
    breaks ties among +inf by position."""
    d = 4
    q = np.array([[1.0, 1.0, 1.0, 1.0], [0.5, 0.5, 0.5, 0.5]], np.float32)
    keys = np.zeros((7 * 4, d), np.float32)
    keys[0:4] = 1.0                         # group 0: pooled 1 -> dots 4, 2 -> 6
    keys[4, 0] = np.inf                     # group 1: +inf
    keys[8, 1] = -np.inf                    # group 2: -inf dots -> +0
    keys[12, 2] = np.nan                    # group 3: NaN dots -> +0
    keys[16, 0], keys[17, 0] = np.inf, -np.inf  # group 4: inf - inf = NaN -> +0
    keys[20, 3] = np.inf                    # group 5: +inf
    keys[24:28] = 2.0                       # group 6: pooled 2 -> dots 8, 4 -> 12
    scores = oracle.score_groups(q, keys)
    want = np.array([6.0, np.inf, 0.0, 0.0, 0.0, np.inf, 12.0], np.float32)
    assert scores.tobytes() == want.tobytes()
    _, chosen = oracle.select(scores, keys.shape[0], 3, return_chosen=True)
    assert chosen.tolist() == [1, 5, 6]
    _, chosen = oracle.select(scores, keys.shape[0], 1, return_chosen=True)
    assert chosen.tolist() == [1]       # the +inf tie goes to the earlier group


def test_relu_before_head_sum_matters(oracle):
    """Order check on a hand case: heads with dots +1 and -1 give 1, not 0."""
    q = np.array([[1.0, 0.0], [-1.0, 0.0]], np.float32)
    keys = np.array([[1.0, 0.0]] * 4, np.float32)
    s = oracle.score_groups(q, keys, 4)
    assert s.tolist() == [1.0]


def test_scores_within_float64_error_bound(oracle):
    """N(0,1) inputs: the FP32 canonical-order score lies within the
    standard rounding bound of the float64 definition written in numpy."""
    rng = np.random.default_rng(11)
    H, d, T = 8, 64, 4 * 700 + 3
    q = rng.standard_normal((H, d)).astype(np.float32)
    keys = rng.standard_normal((T, d)).astype(np.float32)
    s32 = oracle.score_groups(q, keys, T).astype(np.float64)
    G = T // 4
    k64 = keys[:4 * G].astype(np.float64).reshape(G, 4, d)
    pooled = k64.mean(axis=1)
    dots = pooled @ q.astype(np.float64).T
    s64 = np.maximum(dots, 0).sum(axis=1)
    mag = np.abs(k64).mean(axis=1) @ np.abs(q.astype(np.float64)).T  # [G, H]
    bound = gamma(d + H + 3) * (1 + gamma(3)) * mag.sum(axis=1) + 1e-30
    err = np.abs(s32 - s64)
    assert np.all(err <= bound)
    assert err.max() > 0  # it really is FP32


def test_mean_and_sum_pooling_select_the_same_set(oracle):
    """The notes say 'pools' without naming the operator; mean (x0.25) and
    sum (x1) differ by a power of two, which commutes with round-to-nearest,
    so every score scales by exactly 4 and the selection is identical."""
    rng = np.random.default_rng(5)
    q = rng.standard_normal((8, 64)).astype(np.float32)
    keys = rng.standard_normal((4 * 3000 + 1, 64)).astype(np.float32)
    T = keys.shape[0]
    s_mean = oracle.score_groups(q, keys, T, pool_scale=0.25)
    s_sum = oracle.score_groups(q, keys, T, pool_scale=1.0)
    assert np.array_equal(s_sum, s_mean * np.float32(4))
    assert np.array_equal(oracle.select(s_mean, T), oracle.select(s_sum, T))


@pytest.mark.parametrize("T", [0, 3, 4, 5, 37, 2052, 4 * 1100 + 2])
def test_full_raw_equals_incremental(oracle, T):
    """AFN-017 Retrieval capsule (Evidence): full-raw/incremental identity --
    scoring from the raw keys equals scoring from a pooled-key cache appended
    one token at a time, bit for bit, and so does the selected row."""
    rng = np.random.default_rng(100 + T)
    q = rng.standard_normal((4, 32)).astype(np.float32)
    keys = rng.standard_normal((max(T, 1), 32)).astype(np.float32)
    a = oracle.score_groups(q, keys, T)
    b = oracle.score_groups_incremental(q, keys, T)
    assert a.tobytes() == b.tobytes()
    assert np.array_equal(oracle.select(a, T), oracle.select(b, T))


# ------------------------------------------------------- dense parity sweep

def test_dense_parity_sweep(oracle):
    """AFN-017 The dense-parity property: below the 512-group budget the
    sparse row is byte-for-byte the dense causal row plus tail (T = 0..5,
    2,047..2,051); at 2,052 exactly one group is dropped -- the one with the
    lowest score, and among equal lowest scores the largest position."""
    w = wl.dense_parity_sweep()
    qi, ki = _grid_ints(w)
    res = oracle.decode(w, with_scores=True)
    assert res["status"] == 0
    for b, T in enumerate(w.visible.tolist()):
        n = int(res["n_ids"][b])
        ids = res["ids"][b, :n]
        if T <= 2051:
            assert ids.tobytes() == np.arange(T, dtype=np.int32).tobytes()
            assert ids.tobytes() == oracle.dense_ids(T).tobytes()
        else:
            assert T == 2052 and n == 2048
            s256 = _closed_form_scores_x256(qi[b], ki, T)
            low = np.flatnonzero(s256 == s256.min())
            dropped = int(low.max())
            want = np.array([t for t in range(T) if t // 4 != dropped], np.int32)
            assert ids.tobytes() == want.tobytes()
    # the T = 2052 query really has a tie at the cut for this seed
    b = w.visible.tolist().index(2052)
    s256 = _closed_form_scores_x256(qi[b], ki, 2052)
    assert (s256 == s256.min()).sum() >= 2


def test_dense_parity_outputs_bitwise(oracle):
    """Below budget the sparse attention output equals the bounded dense
    oracle's output (AFN-016 Failure boundary: AFN-011 dense through 2,051
    keys), bit for bit, because the rows are identical."""
    w = wl.dense_parity_sweep()
    res = oracle.decode(w)
    for b, T in enumerate(w.visible.tolist()):
        if T > 2051:
            continue
        st, slots = oracle.resolve(oracle.dense_ids(T), w.slot_map, w.num_slots)
        assert st == 0
        dense = oracle.attend(w.q[b], w.k_cache, w.v_cache, slots, w.scale)
        assert dense.tobytes() == res["out"][b].tobytes()


# --------------------------------------------------------------- resolution

def test_resolve_ring_and_paged_closed_forms(oracle):
    """AFN-016 Decision: IDs resolve through the slot map at one boundary.
    Checked against the closed forms of a wrapped ring and of 16-token pages."""
    w = wl.make_workload("ring", [1000, 1000], idx_heads=1, idx_dim=4, q_heads=1,
                         kv_heads=1, head_dim=4, seed=1, slots="ring", ring_size=1000,
                         ring_shift=500)
    ids = np.arange(0, 1000, 7, dtype=np.int32)
    for b in range(2):
        st, slots = oracle.resolve(ids, w.slot_map[w.slot_offset[b]:], w.num_slots)
        assert st == 0
        assert np.array_equal(slots, b * 1000 + (ids + 500) % 1000)
    w = wl.make_workload("paged", [100, 37], idx_heads=1, idx_dim=4, q_heads=1,
                         kv_heads=1, head_dim=4, seed=2, slots="paged16")
    for b, T in enumerate((100, 37)):
        row = w.slot_map[w.slot_offset[b]:w.slot_offset[b] + T]
        pages = row[::16] // 16
        assert np.all(row[::16] % 16 == 0)
        assert np.array_equal(row, (pages[np.arange(T) // 16] * 16 + np.arange(T) % 16))
        st, slots = oracle.resolve(np.arange(T, dtype=np.int32), w.slot_map[w.slot_offset[b]:],
                                   w.num_slots)
        assert st == 0 and np.array_equal(slots, row)
    # all pages distinct across both histories
    allp = w.slot_map // 16
    assert len(np.unique(allp)) == 7 + 3


def test_resolve_rejects_out_of_range_slot(oracle):
    sm = np.array([0, 1, 5, 2], np.int32)
    st, _ = oracle.resolve(np.array([0, 1, 2, 3], np.int32), sm, 5)
    assert st == -3
    st, _ = oracle.resolve(np.array([0, 1, 3], np.int32), sm, 5)
    assert st == 0


# ---------------------------------------------------------------- attention

def _attend64(q, K, V, slots, scale, group):
    """float64 two-pass softmax attention, written independently."""
    n_q, d = q.shape
    out = np.zeros((n_q, d))
    for h in range(n_q):
        k = K[slots, h // group].astype(np.float64)
        v = V[slots, h // group].astype(np.float64)
        x = float(scale) * (k @ q[h].astype(np.float64))
        p = np.exp(x - x.max())
        out[h] = (p / p.sum()) @ v
    return out


def test_attention_single_row_is_v(oracle):
    """T = 1: one row, exp(0) = 1, l = 1, so out = V[slot(0)] bit for bit."""
    rng = np.random.default_rng(3)
    K = rng.standard_normal((10, 2, 64)).astype(np.float32)
    V = rng.standard_normal((10, 2, 64)).astype(np.float32)
    q = rng.standard_normal((4, 64)).astype(np.float32)
    out = oracle.attend(q, K, V, np.array([7], np.int32), 0.125)
    for h in range(4):
        assert out[h].tobytes() == V[7, h // 2].tobytes()


def test_attention_empty_row_is_zero(oracle):
    rng = np.random.default_rng(3)
    K = rng.standard_normal((4, 1, 64)).astype(np.float32)
    out = oracle.attend(rng.standard_normal((2, 64)).astype(np.float32), K, K,
                        np.zeros(0, np.int32), 0.125)
    assert np.all(out == 0)


def test_attention_equal_keys_average_values(oracle):
    """Identical keys give equal weights, so the output is the mean of V."""
    rng = np.random.default_rng(4)
    n = 300
    K = np.repeat(rng.standard_normal((1, 1, 64)).astype(np.float32), n, axis=0)
    V = rng.standard_normal((n, 1, 64)).astype(np.float32)
    q = rng.standard_normal((2, 64)).astype(np.float32)
    out = oracle.attend(q, K, V, np.arange(n, dtype=np.int32), 0.125)
    want = V[:, 0].astype(np.float64).mean(axis=0)
    assert np.abs(out - want).max() <= 4 * (n + 64) * U32 * np.abs(V).max()


@pytest.mark.parametrize("n,d,group", [(37, 64, 1), (2051, 64, 1), (2049, 128, 8), (513, 128, 4)])
def test_attention_within_float64_bound(oracle, n, d, group):
    """The FP32 online softmax in emitted order agrees with the float64
    two-pass softmax within a rounding bound of (n + d) unit roundoffs
    (relative to max|V|); a wrong scale, a missing rescale, a wrong KV head
    or a transposed operand is off by orders of magnitude more."""
    rng = np.random.default_rng(n + d)
    n_kv = 2
    n_q = n_kv * group
    K = rng.standard_normal((n + 17, n_kv, d)).astype(np.float32)
    V = rng.standard_normal((n + 17, n_kv, d)).astype(np.float32)
    q = rng.standard_normal((n_q, d)).astype(np.float32)
    slots = rng.permutation(n + 17)[:n].astype(np.int32)
    scale = np.float32(1 / np.sqrt(d))
    out = oracle.attend(q, K, V, slots, scale)
    want = _attend64(q, K, V, slots, scale, group)
    err = np.abs(out - want).max() / np.abs(V).max()
    assert err <= 4 * (n + d) * U32
    # and a typical error is far smaller than that bound
    assert err <= 2e-6


def test_attention_order_is_observable_but_bounded(oracle):
    """AFN-017 Floating point makes order observable: visiting the same rows
    in another order may change bits, but not beyond rounding."""
    rng = np.random.default_rng(9)
    K = rng.standard_normal((2051, 1, 64)).astype(np.float32) * 3
    V = rng.standard_normal((2051, 1, 64)).astype(np.float32)
    q = rng.standard_normal((1, 64)).astype(np.float32)
    slots = np.arange(2051, dtype=np.int32)
    a = oracle.attend(q, K, V, slots, 0.125)
    b = oracle.attend(q, K, V, slots[::-1].copy(), 0.125)
    assert np.abs(a - b).max() <= 4 * 2115 * U32 * np.abs(V).max()


def test_slot_map_invariance(oracle):
    """AFN-016 Decision: selection never sees the physical layout.  Moving
    the K/V rows to new slots together with the slot map leaves the IDs and
    the outputs bit-identical."""
    w = wl.make_workload("inv", [4 * 700 + 2, 1999], idx_heads=4, idx_dim=32, q_heads=4,
                         kv_heads=2, head_dim=64, seed=21, slots="paged16", budget=512)
    a = oracle.decode(w)
    rng = np.random.default_rng(0)
    perm = rng.permutation(w.num_slots)       # new slot of old slot s: perm[s]
    K2 = np.empty_like(w.k_cache)
    V2 = np.empty_like(w.v_cache)
    K2[perm] = w.k_cache
    V2[perm] = w.v_cache
    import dataclasses
    w2 = dataclasses.replace(w, k_cache=K2, v_cache=V2,
                             slot_map=perm[w.slot_map].astype(np.int32))
    b = oracle.decode(w2)
    assert a["ids"].tobytes() == b["ids"].tobytes()
    assert a["out"].tobytes() == b["out"].tobytes()


# ------------------------------------------------------- whole decode checks

def test_single_t37_is_dense_row(oracle):
    """37 visible tokens: 9 groups, below budget, so the row is 0..36 and the
    output equals the float64 dense attention within rounding."""
    w = wl.single_t37()
    res = oracle.decode(w)
    assert res["status"] == 0 and res["n_ids"][0] == 37
    assert np.array_equal(res["ids"][0, :37], np.arange(37))
    want = _attend64(w.q[0], w.k_cache, w.v_cache, w.slot_map[:37], w.scale, 1)
    assert np.abs(res["out"][0] - want).max() <= 4 * (37 + 64) * U32 * np.abs(w.v_cache).max()


def test_decode_composes_the_stages(oracle):
    """The batch decode equals score -> select -> resolve -> attend per query."""
    w = wl.make_workload("mix", [0, 5, 2052, 4 * 900 + 3], idx_heads=4, idx_dim=32,
                         q_heads=4, kv_heads=2, head_dim=64, seed=8, slots="permutation")
    res = oracle.decode(w, with_scores=True)
    for b, T in enumerate(w.visible.tolist()):
        ko = int(w.key_offset[b])
        s = oracle.score_groups(w.q_idx[b], w.idx_keys[ko:ko + T], T)
        assert s.tobytes() == res["scores"][b, :T // 4].tobytes()
        ids = oracle.select(s, T)
        assert ids.tobytes() == res["ids"][b, :res["n_ids"][b]].tobytes()
        st, slots = oracle.resolve(ids, w.slot_map[w.slot_offset[b]:], w.num_slots)
        out = oracle.attend(w.q[b], w.k_cache, w.v_cache, slots, w.scale)
        assert out.tobytes() == res["out"][b].tobytes()


def test_chunk_equals_decode(oracle):
    """AFN-017 Retrieval capsule (Evidence): chunk/decode equality -- a chunk
    of consecutive queries over one history equals independent single-query
    decodes, bit for bit."""
    w = wl.make_workload("chunk", [4 * 600 + i + 1 for i in range(6)], idx_heads=4,
                         idx_dim=32, q_heads=4, kv_heads=2, head_dim=64, seed=9,
                         history="shared", slots="paged16")
    chunk = oracle.decode(w)
    for b in range(w.batch):
        one = oracle.decode(w.subset([b]))
        n = int(one["n_ids"][0])
        assert n == chunk["n_ids"][b]
        assert one["ids"][0, :n].tobytes() == chunk["ids"][b, :n].tobytes()
        assert one["out"][0].tobytes() == chunk["out"][b].tobytes()


def test_decode_reports_bad_slot(oracle):
    w = wl.make_workload("bad", [40, 40], idx_heads=1, idx_dim=4, q_heads=1, kv_heads=1,
                         head_dim=4, seed=1)
    w.slot_map[w.slot_offset[1] + 3] = w.num_slots + 5
    res = oracle.decode(w)
    assert res["status"] == 2
    assert np.all(res["out"][1] == 0)


def test_budget_one_and_small_budgets(oracle):
    """Budgets below 512 follow the same rule (single best group, etc.)."""
    rng = np.random.default_rng(1)
    s = rng.standard_normal(50).astype(np.float32)
    for k in (1, 2, 7, 49, 50, 64):
        _, chosen = oracle.select(s, 4 * 50 + 1, k, return_chosen=True)
        order = sorted(range(50), key=lambda g: (-float(s[g]), g))[:min(k, 50)]
        assert chosen.tolist() == sorted(order)


def test_oracle_threads_do_not_change_results():
    """The oracle's OpenMP loops (queries, groups, heads) share out
    independent work only: any thread count gives the one-thread bytes."""
    import oracle
    from top_group_sparse_gb300 import workloads as wl
    w = wl.make_workload("thr", [9001, 37, 2052, 4 * 700 + 3, 0], idx_heads=4, idx_dim=32, q_heads=4,
                         kv_heads=2, head_dim=64, seed=23, slots="paged16")
    before = oracle.threads()
    try:
        oracle.threads(1)
        one = oracle.decode(w, with_scores=True)
        for n in (2, 3, 8):
            oracle.threads(n)
            many = oracle.decode(w, with_scores=True)
            for k in ("ids", "n_ids", "out", "scores"):
                assert many[k].tobytes() == one[k].tobytes(), (n, k)
    finally:
        oracle.threads(before)
