"""qsa_attend_noalloc against qsa_attend, through the C ABI.

qsa_attend_noalloc serves callers that cannot allocate device memory or pass
a workspace (a plugin whose host runtime owns all device memory and forbids
third-party allocations, or a loop that must not allocate once it runs): it
keeps its scratch in a fixed static device array instead.  It runs the same
kernel and merge as qsa_attend, so it must give the same output bit for bit,
call after call, although every call reuses the same array.  This file is collected last on purpose, so that a run
stopping at its first failure has already run every other test.
"""
import numpy as np
import pytest

from gpu_helpers import ATTN_TOL, need_gpu
from top_group_sparse_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _staged(w):
    from top_group_sparse_gb300 import qsa
    db = qsa.DeviceBatch(w)
    db.score()
    db.select()
    db.gather()
    db.attend()
    st, flags = db.check_errors()
    assert st == 0, f"device error word {flags:#x}"
    return db


def _rel_err(out, ref, v_scr):
    vmax = float(v_scr.abs().max())
    return float((out.double() - ref.double()).abs().max()) / vmax


def _two_calls_match(db):
    """Two qsa_attend_noalloc calls in a row, each bit-identical to qsa_attend
    on the same inputs (same kernel, same merge; ATTN_TOL only words the
    failure)."""
    import torch
    from top_group_sparse_gb300 import qsa
    ref = db.out.clone()
    for _ in range(2):
        out = torch.full_like(db.out, float("nan"))
        qsa.qsa_attend_noalloc(db.dims, db.q, db.k_scr, db.v_scr, db.n_ids, out)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"differs from qsa_attend: {_rel_err(out, ref, db.v_scr):.3e} (tol {ATTN_TOL})"
    return out


def test_attend_noalloc_matches_attend_on_two_calls_in_a_row():
    need_gpu()
    # two different batches, so the second call really reuses the array that
    # the first call left behind (different row lengths, ragged runs, an
    # empty row and a tail-only row)
    w1 = wl.make_workload("noalloc1", [9001, 2052, 0, 3, 40000, 2051, 777, 65537], idx_heads=8,
                          idx_dim=64, q_heads=16, kv_heads=2, head_dim=128, seed=101, slots="paged16")
    w2 = wl.make_workload("noalloc2", [30000, 5, 4100, 2049], idx_heads=8, idx_dim=64,
                          q_heads=16, kv_heads=2, head_dim=128, seed=102, slots="ring",
                          ring_size=40000, ring_shift=123)
    for w in (w1, w2):
        db = _staged(w)
        out = _two_calls_match(db)
        # empty row -> zero output, as qsa_attend
        n = db.n_ids.cpu().numpy()
        for b in np.flatnonzero(n == 0):
            assert bool((out[b] == 0).all())


def test_attend_noalloc_multi_wave_batch():
    """A batch whose attention grid does not fit on the GPU at once (17 runs x
    2 KV heads x 12 queries > 2 CTAs per SM on every SM): the runs' states are
    merged by the second launch, which reads them from the static array."""
    torch = need_gpu()
    vis = [9001 + 1013 * i for i in range(11)] + [65537]
    w = wl.make_workload("noalloc3", vis, idx_heads=8, idx_dim=64, q_heads=16, kv_heads=2, head_dim=128,
                         seed=103, slots="paged16")
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert 17 * w.kv_heads * w.batch > 2 * sms
    _two_calls_match(_staged(w))


def test_attend_noalloc_bad_row_length_gives_zero_output():
    """This call cannot report the device error word, so a row count outside
    [0, 4*budget + 3] must show as that query's zero output; the other
    queries still equal qsa_attend's bit for bit."""
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    w = wl.make_workload("noalloc4", [9001, 2052, 40000], idx_heads=8, idx_dim=64, q_heads=16, kv_heads=2,
                         head_dim=128, seed=104, slots="paged16")
    db = _staged(w)
    ref = db.out.clone()
    db.n_ids[0] = db.row_cap + 1
    out = torch.full_like(db.out, float("nan"))
    qsa.qsa_attend_noalloc(db.dims, db.q, db.k_scr, db.v_scr, db.n_ids, out)
    torch.cuda.synchronize()
    assert bool((out[0] == 0).all())
    assert torch.equal(out[1:], ref[1:])


def test_attend_noalloc_rejects_dims_beyond_its_scratch():
    need_gpu()
    from top_group_sparse_gb300 import qsa
    # 256 queries x 16 heads x 8 partials x 130 floats is ~17 MB > the fixed array
    dims = qsa.make_dims(256, 8, 64, 16, 2, 128, max_visible=100256)
    with pytest.raises(qsa.QsaError) as e:
        qsa.qsa_attend_noalloc(dims, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20)
    assert e.value.status == 3
