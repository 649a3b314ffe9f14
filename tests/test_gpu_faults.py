"""Device-side error reporting without any GPU fault: bad inputs made on the
host are skipped by the kernels' own checks, recorded in the sticky error
word of the workspace, and read back by qsa_check_errors()."""
import numpy as np
import pytest

from gpu_helpers import need_gpu, oracle_run, assert_ids_equal, assert_attention_close
from top_group_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_slot_out_of_range_sets_flag_and_zero_fills():
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.make_workload("badslot", [3000, 40], idx_heads=4, idx_dim=32, q_heads=2, kv_heads=2,
                         head_dim=64, seed=5)
    w.slot_map[w.slot_offset[1] + 7] = w.num_slots + 11   # token 7 of query 1: beyond the cache
    db = qsa.DeviceBatch(w)
    db.score(); db.select(); db.gather(); db.attend()
    st, flags = db.check_errors()
    assert st == 5 and flags & qsa.QSA_DEVERR_SLOT_RANGE
    k_scr = db.k_scr.cpu().numpy()
    assert np.all(k_scr[1, 7] == 0)
    # query 0 is untouched by query 1's bad slot
    ref = oracle_run(w.subset([0]))
    gpu = {"ids": db.ids.cpu().numpy(), "n_ids": db.n_ids.cpu().numpy(), "out": db.out.cpu().numpy()}
    assert_ids_equal(w, gpu, ref, queries=[0])
    assert_attention_close(w, gpu, ref, queries=[0])
    # the word was cleared by the read
    assert db.check_errors() == (0, 0)


def test_visible_beyond_bound_gives_empty_row_and_flag():
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.make_workload("badT", [3000, 3000], idx_heads=4, idx_dim=32, q_heads=2, kv_heads=2,
                         head_dim=64, seed=6)
    db = qsa.DeviceBatch(w)
    db.visible[1] = 3001            # larger than max_visible = 3000
    db.decode()
    st, flags = db.check_errors()
    assert st == 5 and flags & qsa.QSA_DEVERR_VISIBLE_RANGE
    assert int(db.n_ids[1]) == 0
    assert torch.all(db.out[1] == 0)
    ref = oracle_run(w.subset([0]))
    gpu = {"ids": db.ids.cpu().numpy(), "n_ids": db.n_ids.cpu().numpy(), "out": db.out.cpu().numpy()}
    assert_ids_equal(w, gpu, ref, queries=[0])


def test_row_length_beyond_capacity_flagged():
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.make_workload("badn", [600, 600], idx_heads=4, idx_dim=32, q_heads=2, kv_heads=2,
                         head_dim=64, seed=7)
    db = qsa.DeviceBatch(w)
    db.score(); db.select()
    db.n_ids[0] = db.row_cap + 1
    db.gather(); db.attend()
    st, flags = db.check_errors()
    assert st == 5 and flags & qsa.QSA_DEVERR_ROW_RANGE
    assert torch.all(db.out[0] == 0)
    assert torch.all(torch.isfinite(db.out[1]))


def test_workspace_init_and_clean_tickets():
    """Tickets return to zero after every call, so repeated calls and a fresh
    qsa_workspace_init agree bit for bit."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.make_workload("ws", [5000, 123], idx_heads=4, idx_dim=32, q_heads=2, kv_heads=2,
                         head_dim=64, seed=8)
    db = qsa.DeviceBatch(w)
    db.decode()
    first = db.out.clone()
    qsa.qsa_workspace_init(db.ws)
    db.decode()
    db.decode()
    torch.cuda.synchronize()
    assert torch.equal(first, db.out)
    assert int(db.ws[:512].count_nonzero()) == 0  # error word and tickets


def test_copy_wait_timeout_is_reported_and_the_workspace_stays_usable():
    """Failure detection without a fault (the non-completion gate): the
    scorer runs with its copy producer switched off (qsa_selftest_copy_timeout),
    so every CTA's bounded wait runs out after 2 ms.  The error word reports
    QSA_DEVERR_WAIT_TIMEOUT, no score is written, and the read clears the
    word.  The same workspace then decodes exactly as one that never timed
    out (rows, counts and outputs bit for bit), and under its learned per-SM
    shares the scorer still writes every score, equal to the oracle's."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    from gpu_helpers import assert_scores_equal
    w = wl.make_workload("timeout", [65537, 40003, 2052], idx_heads=8, idx_dim=64, q_heads=16, kv_heads=2,
                         head_dim=128, seed=61, slots="paged16")
    db = qsa.DeviceBatch(w)
    fresh = qsa.DeviceBatch(w)
    for _ in range(3):  # both workspaces learn their per-SM scorer weights
        db.decode()
        fresh.decode()
    assert db.check_errors() == (0, 0) and fresh.check_errors() == (0, 0)
    db.scores.fill_(float("nan"))
    qsa.qsa_selftest_copy_timeout(db.dims, db.inputs, db.scores, db.ws, 2_000_000)
    st, flags = db.check_errors()
    assert st == qsa.QSA_ERR_DEVICE_FAULT and flags == qsa.QSA_DEVERR_WAIT_TIMEOUT
    assert bool(torch.isnan(db.scores).all())
    assert db.check_errors() == (0, 0)  # read and cleared
    for _ in range(3):
        db.decode()
        fresh.decode()
        assert db.check_errors() == (0, 0) and fresh.check_errors() == (0, 0)
        assert torch.equal(db.n_ids, fresh.n_ids)
        assert torch.equal(db.ids, fresh.ids)
        assert torch.equal(db.out, fresh.out)
    db.scores.fill_(float("nan"))
    db.score()
    assert db.check_errors() == (0, 0)
    ref = oracle_run(w)
    gpu = {"scores": db.scores.cpu().numpy(), "ids": db.ids.cpu().numpy(), "n_ids": db.n_ids.cpu().numpy(),
           "out": db.out.cpu().numpy()}
    assert_scores_equal(w, gpu, ref)
    assert_ids_equal(w, gpu, ref)
    assert_attention_close(w, gpu, ref)
