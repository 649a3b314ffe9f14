"""GPU parity of every stage against the CPU oracle, through the C ABI.

Sizes here finish in the oracle within seconds yet span many scorer tiles,
several select-cluster slices, several attention chunks and ragged tails."""
import dataclasses

import numpy as np
import pytest

from gpu_helpers import (full_parity, need_gpu, oracle_run, run_decode, run_stages,
                         assert_ids_equal, assert_attention_close)
from top_group_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_single_t37_dense_row():
    """37 visible tokens: 9 groups + 1 tail, below budget, row = 0..36."""
    w = wl.single_t37()
    gpu = run_stages(w)
    ref = oracle_run(w)
    assert gpu["status"] == 0
    full_parity(w, gpu, ref)
    assert gpu["ids"][0, :37].tolist() == list(range(37))


def test_dense_parity_sweep_with_ties():
    """T in {0..5, 2047..2052} on the exact k/8 grid: byte-identical dense rows
    below the cut; at 2052 the tie rule picks the dropped group."""
    w = wl.dense_parity_sweep()
    gpu = run_stages(w)
    ref = oracle_run(w)
    assert gpu["status"] == 0
    full_parity(w, gpu, ref)
    for b, T in enumerate(w.visible.tolist()):
        if T <= 2051:
            assert gpu["ids"][b, :T].tobytes() == np.arange(T, dtype=np.int32).tobytes()
    dec = run_decode(w)
    assert dec["ids"].tobytes() == gpu["ids"].tobytes()
    assert dec["out"].tobytes() == gpu["out"].tobytes()


@pytest.mark.parametrize("T", [2052, 2053, 2055, 4 * 513 + 3, 9001, 20003])
def test_paged_gqa_multi_tile(T):
    """GQA 16/2 x 128 with 16-token pages, several T around and above the cut."""
    w = wl.make_workload("paged", [T, T - 1, max(T - 5, 0)], idx_heads=8, idx_dim=64, q_heads=16,
                         kv_heads=2, head_dim=128, seed=T, slots="paged16")
    gpu = run_stages(w)
    ref = oracle_run(w)
    assert gpu["status"] == 0
    full_parity(w, gpu, ref)


def test_ragged_batch_all_edges():
    """One batch mixing empty, tail-only, exactly-budget, budget+1 and long rows."""
    vis = [0, 1, 2, 3, 4, 7, 2047, 2048, 2051, 2052, 2053, 4 * 600 + 1, 33333, 65537]
    w = wl.make_workload("ragged", vis, idx_heads=8, idx_dim=64, q_heads=16, kv_heads=2,
                         head_dim=128, seed=77, slots="permutation")
    gpu = run_stages(w)
    ref = oracle_run(w)
    assert gpu["status"] == 0
    full_parity(w, gpu, ref)
    assert np.all(gpu["out"][0] == 0)


@pytest.mark.parametrize("shape", [(4, 32, 2, 2, 64), (8, 32, 4, 1, 64), (4, 64, 8, 8, 128),
                                   (8, 64, 16, 1, 128)])
def test_every_built_shape(shape):
    """Each compiled (H_I, d_I) scorer and head_dim / GQA attention variant."""
    H, dI, nq, nkv, hd = shape
    w = wl.make_workload("shape", [5003, 12000, 2052], idx_heads=H, idx_dim=dI, q_heads=nq,
                         kv_heads=nkv, head_dim=hd, seed=H * dI + nq, slots="permutation")
    gpu = run_stages(w)
    ref = oracle_run(w)
    assert gpu["status"] == 0
    full_parity(w, gpu, ref)


@pytest.mark.parametrize("budget", [1, 2, 7, 100, 511, 512])
def test_budgets(budget):
    w = wl.make_workload("budget", [4 * 700 + 2, 3001, 4 * budget, 4 * budget + 4], idx_heads=4,
                         idx_dim=32, q_heads=2, kv_heads=2, head_dim=64, seed=budget,
                         slots="identity", budget=budget)
    gpu = run_stages(w)
    ref = oracle_run(w)
    assert gpu["status"] == 0
    full_parity(w, gpu, ref)


def test_all_scores_tie():
    """Identical index keys: every group scores the same, membership is the
    first `budget` groups (smaller positions win)."""
    w = wl.make_workload("ties", [9000, 4 * 513, 20001], idx_heads=4, idx_dim=32, q_heads=2,
                         kv_heads=2, head_dim=64, seed=3)
    w = dataclasses.replace(w, idx_keys=np.repeat(w.idx_keys[:1], w.total_tokens, axis=0))
    gpu = run_stages(w)
    ref = oracle_run(w)
    full_parity(w, gpu, ref)
    for b, T in enumerate(w.visible.tolist()):
        assert gpu["ids"][b, :2048].tolist() == list(range(2048))


def test_zero_scores_everywhere():
    """An all-zero indexer query: every dot is 0, every ReLU +0, all tie."""
    w = wl.make_workload("zeros", [6000, 2053], idx_heads=8, idx_dim=64, q_heads=16,
                         kv_heads=2, head_dim=128, seed=4)
    w = dataclasses.replace(w, q_idx=np.zeros_like(w.q_idx))
    gpu = run_stages(w)
    ref = oracle_run(w)
    full_parity(w, gpu, ref)
    assert np.all(gpu["scores"][0, :1500] == 0)


def test_heavy_ties_on_integer_grid_long():
    """k/8 grid values over a long history: many exact ties at the threshold."""
    w = wl.make_workload("grid", [40000, 40001, 40003], idx_heads=4, idx_dim=32, q_heads=2,
                         kv_heads=2, head_dim=64, seed=12, index_values="grid8",
                         history="shared", slots="permutation")
    gpu = run_stages(w)
    ref = oracle_run(w)
    full_parity(w, gpu, ref)
    s = ref["scores"][0, :10000]
    assert len(np.unique(s)) < 2000  # the ties are really there


def test_select_uncached_long_history():
    """A history long enough that a cluster slice of scores no longer fits in
    shared memory (G > 8 * 24576), so select streams scores from global."""
    T = 8 * 49152 * 4 + 4 * 1000 + 2
    w = wl.make_workload("long", [T], idx_heads=4, idx_dim=32, q_heads=2, kv_heads=2,
                         head_dim=64, seed=13, slots="ring", ring_size=T, ring_shift=777)
    gpu = run_stages(w)
    ref = oracle_run(w)
    full_parity(w, gpu, ref)


def test_decode_matches_stages_and_is_repeatable():
    w = wl.make_workload("rep", [30001, 4 * 512 + 1, 17], idx_heads=8, idx_dim=64, q_heads=16,
                         kv_heads=2, head_dim=128, seed=31, slots="paged16")
    st = run_stages(w)
    d1 = run_decode(w)
    d2 = run_decode(w, db=d1["batch"])
    for k in ("ids", "n_ids", "out"):
        assert d1[k].tobytes() == st[k].tobytes(), k
        assert d2[k].tobytes() == d1[k].tobytes(), k


def test_chunk_equals_decode_small():
    """Consecutive queries over one history equal single-query decodes, bit
    for bit (the attention split depends on the row length only)."""
    w = wl.chunked_prefill_100000(n=24, first=9000)
    chunk = run_decode(w)
    ref = oracle_run(w)
    assert_ids_equal(w, chunk, ref)
    assert_attention_close(w, chunk, ref)
    for b in range(w.batch):
        one = run_decode(w.subset([b]))
        n = int(one["n_ids"][0])
        assert n == int(chunk["n_ids"][b])
        assert one["ids"][0, :n].tobytes() == chunk["ids"][b, :n].tobytes()
        assert one["out"][0].tobytes() == chunk["out"][b].tobytes()


def test_non_default_stream():
    torch = need_gpu()
    w = wl.make_workload("stream", [9000, 2051], idx_heads=8, idx_dim=64, q_heads=16,
                         kv_heads=2, head_dim=128, seed=41)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        gpu = run_stages(w, stream=s)
    ref = oracle_run(w)
    full_parity(w, gpu, ref)


def test_stats_report_zero_dense_mask():
    need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.single_t37()
    db = qsa.DeviceBatch(w)
    st = qsa.qsa_get_stats(db.dims, w.visible)
    assert st["dense_mask_bytes"] == 0
    assert st["selected_tokens"] == 37 and st["candidate_groups"] == 9


@pytest.mark.parametrize("shape", [(16, 2, 128), (4, 4, 64), (12, 1, 64), (3, 3, 128)])
def test_gather_attend_equals_gather_then_attend(shape):
    """The fused stage writes the same scratch bytes as qsa_gather and the same
    output bits as qsa_attend on that scratch, for GQA ratios 8, 1, 12, 1."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    nq, nkv, hd = shape
    w = wl.make_workload("ga", [9001, 2052, 0, 3, 40000, 2051, 65], idx_heads=8, idx_dim=64,
                         q_heads=nq, kv_heads=nkv, head_dim=hd, seed=55 + nq, slots="paged16")
    db = qsa.DeviceBatch(w)
    db.score(); db.select(); db.gather(); db.attend()
    torch.cuda.synchronize()
    k1, v1, o1 = db.k_scr.clone(), db.v_scr.clone(), db.out.clone()
    db.k_scr.zero_(); db.v_scr.zero_(); db.out.fill_(float("nan"))
    db.gather_attend()
    st, flags = db.check_errors()
    assert st == 0, f"device error word {flags:#x}"
    n = db.n_ids.cpu().numpy()
    for b in range(w.batch):
        assert torch.equal(db.k_scr[b, :n[b]], k1[b, :n[b]])
        assert torch.equal(db.v_scr[b, :n[b]], v1[b, :n[b]])
    assert torch.equal(db.out, o1)
    ref = oracle_run(w)
    gpu = {"ids": db.ids.cpu().numpy(), "n_ids": n, "out": db.out.cpu().numpy()}
    assert_ids_equal(w, gpu, ref)
    assert_attention_close(w, gpu, ref)


def test_decode_profiled_matches_decode():
    """The instrumented decode issues the same launches: same bits, and its four
    events bracket the three stages in order."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.make_workload("prof", [30001, 65537, 2052, 5], idx_heads=8, idx_dim=64, q_heads=16,
                         kv_heads=2, head_dim=128, seed=61, slots="ring", ring_size=70000,
                         ring_shift=999)
    db = qsa.DeviceBatch(w)
    db.decode()
    torch.cuda.synchronize()
    ids, out = db.ids.clone(), db.out.clone()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    db.out.fill_(float("nan"))
    db.decode_profiled(ev)
    torch.cuda.synchronize()
    assert torch.equal(db.ids, ids) and torch.equal(db.out, out)
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(3)]
    assert all(t > 0 for t in times)
    assert db.check_errors() == (0, 0)
    ref = oracle_run(w)
    gpu = {"ids": db.ids.cpu().numpy(), "n_ids": db.n_ids.cpu().numpy(), "out": db.out.cpu().numpy()}
    assert_ids_equal(w, gpu, ref)
    assert_attention_close(w, gpu, ref)


def test_per_sm_balance_engages_and_leaves_results_unchanged():
    """The raw scorer's per-SM shares (weights learned from its own timings,
    kept in the workspace) move tiles between SMs and nothing else: the
    first decode on a fresh workspace (equal shares) and later ones
    (weighted shares) give the same rows and outputs bit for bit, and the
    weights are in place after the first decode."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.long_262144(batch=2)
    db = qsa.DeviceBatch(w)
    db.decode()
    torch.cuda.synchronize()
    ids, out = db.ids.cpu().numpy().copy(), db.out.cpu().numpy().copy()
    # the table sits after the error word and the attention tickets (qsa.h, workspace size)
    off = 256 + ((w.batch * w.kv_heads * 4 + 255) // 256) * 256
    tab = db.ws[off:off + 16].cpu().numpy().view(np.uint32)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert tab[0] == 0x51534231 and tab[1] == sms and tab[2] > 0, tab
    for _ in range(4):
        db.ids.fill_(-1)
        db.out.fill_(float("nan"))
        db.decode()
        assert db.check_errors() == (0, 0)
        assert db.ids.cpu().numpy().tobytes() == ids.tobytes()
        assert db.out.cpu().numpy().tobytes() == out.tobytes()
    w_sm = db.ws[off + 16 + 4 * 256:off + 16 + 8 * 256].cpu().numpy().view(np.uint32)
    assert (w_sm > 0).sum() == sms and w_sm.min(initial=1 << 30) >= 0
    assert w_sm[w_sm > 0].min() >= 1024 and w_sm.max() <= 16384


def test_per_sm_shares_cover_every_tile():
    """Under learned per-SM shares the raw scorer still writes every group's
    score exactly once: the scores of a call on a workspace whose weights are
    in place, written into a NaN-filled buffer (no score of an earlier call
    can stand in for a missed tile), equal the oracle's bit for bit."""
    torch = need_gpu()
    import oracle
    from top_group_sparse_gb300 import qsa
    w = wl.long_262144(batch=2, seed=12)
    db = qsa.DeviceBatch(w)
    for _ in range(3):
        db.decode()
    off = 256 + ((w.batch * w.kv_heads * 4 + 255) // 256) * 256
    assert db.ws[off:off + 4].cpu().numpy().view(np.uint32)[0] == 0x51534231
    db.scores.fill_(float("nan"))
    db.score()
    assert db.check_errors() == (0, 0)
    got = db.scores.cpu().numpy()
    for b in range(w.batch):
        ko, T = int(w.key_offset[b]), int(w.visible[b])
        ref = oracle.score_groups(w.q_idx[b], w.idx_keys[ko:ko + T], T)
        assert got[b, :T // 4].tobytes() == ref.tobytes(), b


def test_decode_from_host_buffers():
    """One copy in, qsa_decode, one copy out: the host buffers carry exactly
    the step's inputs and the device-side results."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.make_workload("host", [9001, 37, 2052, 0], idx_heads=8, idx_dim=64, q_heads=16,
                         kv_heads=2, head_dim=128, seed=91, slots="paged16")
    db = qsa.DeviceBatch(w)
    db.decode()
    torch.cuda.synchronize()
    ids, n, out = db.ids.cpu().numpy().copy(), db.n_ids.cpu().numpy().copy(), db.out.cpu().numpy().copy()
    h_in, h_out = db.step_host_buffers()
    db.ids.fill_(-1)
    db.out.fill_(float("nan"))
    db.q_idx.zero_()  # overwritten by the step's copy in
    db.decode_from_host(h_in, h_out)
    torch.cuda.synchronize()
    hi, hn, ho = db.host_outputs(h_out)
    assert hn.numpy().tobytes() == n.tobytes()
    assert hi.numpy().tobytes() == ids.tobytes()
    assert ho.numpy().tobytes() == out.tobytes()


def test_decode_from_host_as_a_cuda_graph():
    """The host-driven step captured once and replayed, with the outputs
    copied back and with the kernels storing them straight into the pinned
    host buffer: same counts, rows (up to each count: entries past it are
    untouched) and outputs as eager, and a replay after new inputs sees them."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.long_262144(batch=2)
    db = qsa.DeviceBatch(w)
    h_in, h_out = db.step_host_buffers()
    db.decode_from_host(h_in, h_out)
    torch.cuda.synchronize()
    ref = [t.numpy().copy() for t in db.host_outputs(h_out)]

    def same_as_ref():
        ids, n, out = (t.numpy() for t in db.host_outputs(h_out))
        if n.tobytes() != ref[1].tobytes() or out.tobytes() != ref[2].tobytes():
            return False
        return all(ids[b, :n[b]].tobytes() == ref[0][b, :n[b]].tobytes() for b in range(len(n)))

    h_out.zero_()
    db.decode_into_host(h_in, h_out)
    torch.cuda.synchronize()
    assert same_as_ref()
    for direct in (False, True):
        g = db.capture_decode_from_host(h_in, h_out, direct=direct)
        for _ in range(3):
            h_out.zero_()
            g.replay()
            torch.cuda.synchronize()
            assert same_as_ref(), direct
    # new step inputs in the host buffer reach the replayed graph
    qv = h_in[db.q.data_ptr() - db.step_in.data_ptr():][: db.q.numel() * 4].view(torch.float32)
    qv.mul_(2.0)
    g.replay()
    torch.cuda.synchronize()
    assert db.host_outputs(h_out)[2].numpy().tobytes() != ref[2].tobytes()
    assert db.check_errors() == (0, 0)


@pytest.mark.parametrize("q_heads,kv_heads,head_dim,nq", [(16, 2, 128, 12), (16, 1, 64, 40), (4, 4, 128, 30)])
def test_merge_path_does_not_change_bits(q_heads, kv_heads, head_dim, nq):
    """An attention grid of more than one wave merges its runs in a second
    launch, a one-wave grid in its last CTA: the merge arithmetic is the
    same, so a query's output in a batch of several waves equals its
    single-query decode bit for bit -- for one and two CTAs per SM (GQ 16,
    8 and 1; head dims 64 and 128), with rows of every length (runs without
    rows among them) and grids of up to seven waves."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    vis = [9001 + 1013 * (i % 11) for i in range(nq - 3)] + [2052, 40, 700]
    w = wl.make_workload("merge", vis, idx_heads=8, idx_dim=64, q_heads=q_heads, kv_heads=kv_heads,
                         head_dim=head_dim, seed=97 + nq, slots="paged16")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    per_sm = 2 if q_heads // kv_heads <= 8 else 1
    assert 17 * w.kv_heads * w.batch > per_sm * sms  # the batch takes the persistent grid
    db = qsa.DeviceBatch(w)
    db.decode()
    assert db.check_errors() == (0, 0)
    out = db.out.cpu().numpy()
    ids, n_ids = db.ids.cpu().numpy(), db.n_ids.cpu().numpy()
    for b in sorted({0, 5, nq - 3, nq - 2, nq - 1}):
        one = qsa.DeviceBatch(w, queries=[b])
        one.decode()
        assert one.check_errors() == (0, 0)
        assert one.out.cpu().numpy()[0].tobytes() == out[b].tobytes(), b
        assert int(one.n_ids[0]) == n_ids[b]
        assert np.array_equal(one.ids.cpu().numpy()[0, : n_ids[b]], ids[b, : n_ids[b]])


def test_multi_wave_grid_flags_a_bad_row_and_keeps_the_rest():
    """A query whose visible length exceeds the bound, inside a batch of
    several attention waves: its row is empty, its output zero and the
    error word flagged; every other query equals its single-query decode."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    vis = [6000 + 517 * i for i in range(12)]
    w = wl.make_workload("pbad", vis, idx_heads=8, idx_dim=64, q_heads=16, kv_heads=2, head_dim=128,
                         seed=131, slots="paged16")
    db = qsa.DeviceBatch(w)
    db.visible[4] = w.max_visible + 1
    db.decode()
    st, flags = db.check_errors()
    assert st == qsa.QSA_ERR_DEVICE_FAULT and flags & qsa.QSA_DEVERR_VISIBLE_RANGE
    assert int(db.n_ids[4]) == 0 and bool(torch.all(db.out[4] == 0))
    out = db.out.cpu().numpy()
    for b in (0, 3, 5, 11):
        one = qsa.DeviceBatch(w, queries=[b])
        one.decode()
        assert one.out.cpu().numpy()[0].tobytes() == out[b].tobytes(), b


def test_non_finite_index_keys_match_the_oracle():
    """Index keys with +inf, -inf and NaN planted (the reading ReLU(x) = x > 0
    ? x : +0 keeps every score in [+0, +inf]): 600 groups per history get a
    +inf element -- more than the budget, so the selection must take the 512
    earliest of the tied +inf scores -- others -inf, NaN, or +inf and -inf in
    one group.  Scores and ID rows bit-exact, outputs within 1e-5 * max|V|."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    from gpu_helpers import assert_scores_equal
    w = wl.make_workload("nonfinite", [20000, 9001, 3002], idx_heads=8, idx_dim=64, q_heads=16, kv_heads=2,
                         head_dim=128, seed=131, slots="paged16")
    rng = np.random.default_rng(7)
    for b in range(w.batch):
        base, G = int(w.key_offset[b]), int(w.visible[b]) // 4
        g = rng.permutation(G)
        rows = lambda gs: base + 4 * gs + rng.integers(0, 4, gs.shape[0])  # noqa: E731
        cols = lambda gs: rng.integers(0, w.idx_dim, gs.shape[0])  # noqa: E731
        gi, gm, gn, gp = g[:600], g[600:650], g[650:700], g[700:750]
        w.idx_keys[rows(gi), cols(gi)] = np.inf
        w.idx_keys[rows(gm), cols(gm)] = -np.inf
        w.idx_keys[rows(gn), cols(gn)] = np.nan
        c = cols(gp)
        w.idx_keys[base + 4 * gp, c] = np.inf
        w.idx_keys[base + 4 * gp + 1, c] = -np.inf
    db = qsa.DeviceBatch(w)
    gpu = run_decode(w, db=db)
    assert gpu["status"] == 0, f"device error flags {gpu['flags']:#x}"
    db.score()
    torch.cuda.synchronize()
    gpu["scores"] = db.scores.cpu().numpy()
    ref = oracle_run(w)
    assert_scores_equal(w, gpu, ref)
    assert np.isinf(ref["scores"][0, :5000]).sum() > 512  # the tie among +inf decides the set
    assert_ids_equal(w, gpu, ref)
    assert_attention_close(w, gpu, ref)
