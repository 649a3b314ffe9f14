"""qsa_attend_noalloc against qsa_attend, through the C ABI.

qsa_attend_noalloc serves callers that cannot allocate device memory or pass
a workspace (a plugin whose host runtime owns all device memory and forbids
third-party allocations, or a loop that must not allocate once it runs): it
keeps its scratch in a fixed static device array instead.  It must give the
same attention output as qsa_attend, call after call, although every call
reuses the same array.  This file is collected last on purpose, so that a run
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


def _rel_err(torch, out, ref, v_scr):
    vmax = float(v_scr.abs().max())
    return float((out.double() - ref.double()).abs().max()) / vmax


def test_attend_noalloc_matches_attend_on_two_calls_in_a_row():
    torch = need_gpu()
    from top_group_sparse_gb300 import qsa
    # two different batches, so the second call really reuses the array that
    # the first call left behind (different row lengths, ragged chunks, an
    # empty row and a tail-only row)
    w1 = wl.make_workload("noalloc1", [9001, 2052, 0, 3, 40000, 2051, 777, 65537], idx_heads=8,
                          idx_dim=64, q_heads=16, kv_heads=2, head_dim=128, seed=101, slots="paged16")
    w2 = wl.make_workload("noalloc2", [30000, 5, 4100, 2049], idx_heads=8, idx_dim=64,
                          q_heads=16, kv_heads=2, head_dim=128, seed=102, slots="ring",
                          ring_size=40000, ring_shift=123)
    for w in (w1, w2):
        db = _staged(w)
        ref = db.out.clone()
        for _ in range(2):
            out = torch.full_like(db.out, float("nan"))
            qsa.qsa_attend_noalloc(db.dims, db.q, db.k_scr, db.v_scr, db.n_ids, out)
            torch.cuda.synchronize()
            assert bool(torch.isfinite(out).all())
            assert _rel_err(torch, out, ref, db.v_scr) <= ATTN_TOL
        # empty row -> zero output, as qsa_attend
        n = db.n_ids.cpu().numpy()
        for b in np.flatnonzero(n == 0):
            assert bool((out[b] == 0).all())


def test_attend_noalloc_rejects_dims_beyond_its_scratch():
    need_gpu()
    from top_group_sparse_gb300 import qsa
    # 256 queries x 16 heads x 8 partials x 130 floats is ~17 MB > the fixed array
    dims = qsa.make_dims(256, 8, 64, 16, 2, 128, max_visible=100256)
    with pytest.raises(qsa.QsaError) as e:
        qsa.qsa_attend_noalloc(dims, 1 << 20, 1 << 20, 1 << 20, 1 << 20, 1 << 20)
    assert e.value.status == 3
