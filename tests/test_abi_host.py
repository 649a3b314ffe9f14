"""The C-ABI library builds, loads and exports every symbol include/qsa.h
declares; its host-only logic (sizes, stats, validation) runs without a GPU.
No call here reaches a CUDA kernel: every compute call below is rejected by
host-side validation before anything is enqueued."""
import ctypes
import os

import pytest

from top_group_sparse_gb300 import build as qbuild
from top_group_sparse_gb300 import qsa

QSA_OK, INVALID, UNSUPPORTED, WS_SMALL = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    qbuild.build()
    return qsa.load()


def test_exports_every_declared_symbol(lib):
    names = qsa.exported_symbols()
    assert len(names) == 24
    for n in names:
        assert hasattr(lib, n), n
    for n in ("qsa_score_groups", "qsa_select", "qsa_gather", "qsa_attend", "qsa_gather_attend", "qsa_attend_state",
              "qsa_decode"):
        assert n in names
    # the failure-detection self-test, declared apart from the hot path
    selftest = qsa.exported_symbols(os.path.join(os.path.dirname(qsa.library_path()), "..", "..", "include",
                                                 "qsa_selftest.h"))
    assert selftest == ["qsa_selftest_copy_timeout"]
    assert hasattr(lib, selftest[0])


def test_status_strings(lib):
    for s in range(6):
        assert len(qsa.qsa_status_string(s)) >= 2
    assert qsa.qsa_status_string(99) == "unknown status"


def _dims(**kw):
    base = dict(batch=8, idx_heads=8, idx_dim=64, q_heads=16, kv_heads=2, head_dim=128,
                budget_groups=512, max_visible=262144)
    base.update(kw)
    return qsa.make_dims(**base)


def test_row_capacity_and_score_stride(lib):
    assert qsa.qsa_row_capacity(_dims()) == 2051
    assert qsa.qsa_row_capacity(_dims(budget_groups=1)) == 7
    assert qsa.qsa_score_stride(_dims()) == 65536
    assert qsa.qsa_score_stride(_dims(max_visible=65537)) == 16384
    assert qsa.qsa_score_stride(_dims(max_visible=37)) == 32
    assert qsa.qsa_score_stride(_dims(max_visible=0)) == 32


def _align(x, a=256):
    return (x + a - 1) // a * a


def test_workspace_formula(lib):
    """Scratch is groups + budget + selected width per query, never queries x
    keys ("A sparse mask is not sparse attention", What the checkpoint measures);
    the compact K/V row of the whole-path call stays on chip, so no K/V scratch."""
    d = _dims()
    B, nq, nkv, hd = 8, 16, 2, 128
    nch = 17  # attention partials per head: runs of 128 rows over at most 2051 rows
    bal = 7424  # the scorer's per-SM balance table
    want = 256 + _align(B * nkv * 4) + bal + 2 * _align(B * nq * nch * 4) + _align(B * nq * nch * hd * 4) \
        + _align(B * 16384 * 4) + _align(B * 65536 * 4) + _align(B * 2051 * 4) + _align(B * 4)
    assert qsa.qsa_workspace_size(d) == want
    # doubling the history adds exactly the scores (and per-quad maxima) of the new groups
    a = qsa.qsa_workspace_size(_dims(max_visible=1 << 20))
    b = qsa.qsa_workspace_size(_dims(max_visible=1 << 21))
    assert b - a == B * ((1 << 19) - (1 << 18)) * 4 + B * ((1 << 17) - (1 << 16)) * 4
    # and is linear in the batch
    assert qsa.qsa_workspace_size(_dims(batch=16)) < 2 * qsa.qsa_workspace_size(d) + 4096


def test_invalid_dims_give_zero_workspace(lib):
    assert qsa.qsa_workspace_size(_dims(group=3)) == 0
    assert qsa.qsa_workspace_size(_dims(budget_groups=0)) == 0
    assert qsa.qsa_workspace_size(_dims(budget_groups=513)) == 0
    assert qsa.qsa_workspace_size(_dims(q_heads=15)) == 0
    assert qsa.qsa_workspace_size(_dims(batch=-1)) == 0
    assert qsa.qsa_workspace_size(_dims(batch=65536)) == 0  # grids carry the query in a 16-bit dimension
    assert qsa.qsa_workspace_size(_dims(batch=65535, max_visible=64)) > 0
    assert qsa.qsa_workspace_size(_dims(max_visible=(1 << 26) + 1)) == 0


def test_stats_closed_forms(lib):
    d = _dims(batch=4, max_visible=300000)
    vis = [0, 37, 2052, 262144]
    st = qsa.qsa_get_stats(d, vis)
    G = [0, 9, 513, 65536]
    k = [0, 9, 512, 512]
    W = [0, 37, 2048, 2048]
    assert st["candidate_groups"] == sum(G)
    assert st["selected_groups"] == sum(k)
    assert st["selected_tokens"] == sum(W)
    assert st["raw_key_bytes"] == sum(vis) * 64 * 4
    assert st["kv_bytes"] == sum(W) * 2 * 128 * 4 * 2
    assert st["pooled_key_bytes"] == 0
    assert st["workspace_bytes"] == qsa.qsa_workspace_size(d)
    assert st["total_bytes"] == st["raw_key_bytes"] + st["kv_bytes"] + st["workspace_bytes"]
    assert st["dense_mask_bytes"] == 0
    with pytest.raises(qsa.QsaError):
        qsa.qsa_get_stats(d, [0, 1, 2, 300001])


def test_stats_of_the_incremental_form(lib):
    """Byte ownership of the incremental form ("A sparse mask is not sparse
    attention", What the checkpoint measures: raw-key, K/V, pooled-key,
    workspace and total bytes): the scorer streams no raw keys, and the
    pooled-key cache -- floor(T/4) rows of d_I floats per history, shared by
    the queries of one history -- is counted and included in the total."""
    # three chunked-prefill queries over one history of 100,256 tokens, and a
    # decode query with its own history of 262,144 tokens
    d = _dims(batch=4, max_visible=300000)
    vis = [100001, 100002, 100256, 262144]
    histories = {0: 100256, 1: 262144}  # history -> tokens it holds
    rows = sum(T // 4 for T in histories.values())
    full = qsa.qsa_get_stats(d, vis)
    st = qsa.qsa_get_stats_pooled(d, vis, rows)
    assert st["pooled_key_bytes"] == (100256 // 4 + 262144 // 4) * 64 * 4
    assert st["raw_key_bytes"] == 0
    for key in ("candidate_groups", "selected_groups", "selected_tokens", "kv_bytes", "workspace_bytes"):
        assert st[key] == full[key], key
    assert st["total_bytes"] == st["kv_bytes"] + st["pooled_key_bytes"] + st["workspace_bytes"]
    assert st["dense_mask_bytes"] == 0
    # the cache holds 4x fewer bytes than the raw keys of the same histories
    assert st["pooled_key_bytes"] * 4 == sum(histories.values()) * 64 * 4
    with pytest.raises(qsa.QsaError):
        qsa.qsa_get_stats_pooled(d, vis, -1)


def _raw(fn, *args):
    return getattr(qsa.load(), fn)(*args)


def test_validation_rejects_before_launch(lib):
    """Every one of these returns a status without touching the GPU."""
    d = _dims(batch=2, max_visible=4096)
    bad = _dims(group=5)
    fake = 1 << 20  # 256-aligned non-null address that is never dereferenced
    inp = qsa.QsaInputs(fake, fake, fake, fake, fake, fake, fake, 100, fake, fake)
    null_inp = qsa.QsaInputs(None, fake, fake, fake, fake, fake, fake, 100, fake, fake)
    mis_inp = qsa.QsaInputs(fake + 4, fake, fake, fake, fake, fake, fake, 100, fake, fake)
    ws_need = qsa.qsa_workspace_size(d)
    D, I = ctypes.byref, ctypes.byref
    assert _raw("qsa_decode", D(bad), I(inp), fake, fake, fake, fake, ws_need, None) == INVALID
    assert _raw("qsa_decode", D(d), I(null_inp), fake, fake, fake, fake, ws_need, None) == INVALID
    assert _raw("qsa_decode", D(d), I(mis_inp), fake, fake, fake, fake, ws_need, None) == INVALID
    assert _raw("qsa_decode", D(d), I(inp), fake, fake, fake, fake, ws_need - 1, None) == WS_SMALL
    assert _raw("qsa_decode", D(d), I(inp), fake, fake, fake, fake + 8, ws_need, None) == INVALID
    assert _raw("qsa_decode", D(d), I(inp), None, fake, fake, fake, ws_need, None) == INVALID
    uns = _dims(batch=2, max_visible=4096, idx_dim=48)
    assert _raw("qsa_decode", D(uns), I(inp), fake, fake, fake, fake, 1 << 30, None) == UNSUPPORTED
    uns = _dims(batch=2, max_visible=4096, head_dim=96)
    assert _raw("qsa_attend", D(uns), fake, fake, fake, fake, fake, fake, 1 << 30, None) == UNSUPPORTED
    uns = _dims(batch=2, max_visible=4096, q_heads=64, kv_heads=2)
    assert _raw("qsa_attend", D(uns), fake, fake, fake, fake, fake, fake, 1 << 30, None) == UNSUPPORTED
    assert _raw("qsa_score_groups", D(d), I(inp), None, fake, ws_need, None) == INVALID
    assert _raw("qsa_select", D(d), fake, fake, None, fake, fake, ws_need, None) == INVALID
    assert _raw("qsa_select", D(d), fake, fake + 4, fake, fake, fake, ws_need, None) == INVALID
    assert _raw("qsa_gather", D(d), I(inp), fake, fake, fake, fake + 4, fake, ws_need, None) == INVALID
    assert _raw("qsa_attend", D(d), fake, fake, fake, fake, fake, fake, 100, None) == WS_SMALL
    # qsa_attend_state(dims, in, ids, n_ids, acc, m, l, ws, ws_bytes, stream)
    st = "qsa_attend_state"
    assert _raw(st, D(d), I(inp), fake, fake, fake, fake, None, fake, ws_need, None) == INVALID
    assert _raw(st, D(d), I(inp), fake, fake, fake + 4, fake, fake, fake, ws_need, None) == INVALID
    no_q = qsa.QsaInputs(fake, fake, fake, fake, None, fake, fake, 100, fake, fake)
    assert _raw(st, D(d), I(no_q), fake, fake, fake, fake, fake, fake, ws_need, None) == INVALID
    assert _raw(st, D(d), I(inp), fake, fake, fake, fake, fake, fake, ws_need - 1, None) == WS_SMALL
    assert _raw(st, D(bad), I(inp), fake, fake, fake, fake, fake, fake, ws_need, None) == INVALID
    # qsa_merge_states(dims, n_parts, m, l, acc, out, stream)
    ms = "qsa_merge_states"
    assert _raw(ms, D(d), 0, fake, fake, fake, fake, None) == INVALID
    assert _raw(ms, D(d), 2, None, fake, fake, fake, None) == INVALID
    assert _raw(ms, D(d), 2, fake, fake, fake + 4, fake, None) == INVALID
    assert _raw(ms, D(d), 2, fake, fake, fake, fake + 8, None) == INVALID
    assert _raw(ms, D(d), 2, fake + 2, fake, fake, fake, None) == INVALID
    assert _raw(ms, D(bad), 2, fake, fake, fake, fake, None) == INVALID
    assert _raw(ms, D(_dims(batch=2, max_visible=4096, head_dim=96)), 2, fake, fake, fake, fake, None) == UNSUPPORTED
    # qsa_selftest_copy_timeout(dims, in, scores, ws, ws_bytes, wait_ns, stream)
    tst = "qsa_selftest_copy_timeout"
    assert _raw(tst, D(d), I(inp), fake, fake, ws_need, ctypes.c_uint64(0), None) == INVALID
    assert _raw(tst, D(d), I(inp), fake, fake, ws_need, ctypes.c_uint64(2_000_000_000), None) == INVALID
    assert _raw(tst, D(d), I(inp), fake, fake, ws_need - 1, ctypes.c_uint64(1000), None) == WS_SMALL
    assert _raw(tst, D(d), I(null_inp), fake, fake, ws_need, ctypes.c_uint64(1000), None) == INVALID
    assert _raw("qsa_workspace_init", None, 10, None) == INVALID
    assert _raw("qsa_check_errors", fake, 8, None, None) == INVALID


def test_ffma_probe_rejects_bad_arguments(lib):
    """Checked on the host before any launch: no GPU needed."""
    for bps, iters in ((0, 10), (9, 10), (4, 0)):
        with pytest.raises(qsa.QsaError):
            qsa.qsa_probe_ffma(bps, iters, None, stream=0)


def test_packed_step_buffers_layout():
    """A decode step's inputs (and outputs) share one buffer: every item on a
    16-byte boundary, typed views over its own bytes only, fills applied."""
    import numpy as np
    a = np.arange(6, dtype=np.float32).reshape(2, 3)
    b = np.array([5, -7, 9], dtype=np.int64)
    buf, v = qsa._packed([("a", a), ("b", b), ("c", ((3, 2), np.int32, -1)),
                          ("d", ((5,), np.float32, float("nan")))], "cpu")
    base = buf.data_ptr()
    for name in ("a", "b", "c", "d"):
        assert (v[name].data_ptr() - base) % 16 == 0, name
    assert v["a"].numpy().tobytes() == a.tobytes() and v["b"].numpy().tobytes() == b.tobytes()
    assert (v["c"].numpy() == -1).all() and np.isnan(v["d"].numpy()).all()
    # no overlap: writing one view leaves the others as they were
    v["c"].fill_(3)
    assert v["a"].numpy().tobytes() == a.tobytes() and v["b"].numpy().tobytes() == b.tobytes()
    ends = sorted((t.data_ptr() - base, t.data_ptr() - base + t.numel() * t.element_size()) for t in v.values())
    assert all(e0 <= s1 for (_, e0), (s1, _) in zip(ends, ends[1:])) and ends[-1][1] <= buf.numel()


_C_CLIENT = r"""
#include <stdio.h>
#include "qsa.h"

int main(void)
{
    qsa_dims d = {8, 8, 64, 16, 2, 128, 4, 512, 262144, 0.088388347648f};
    int32_t visible[8] = {262144, 262144, 262144, 262144, 262144, 262144, 262144, 262144};
    qsa_stats st;
    qsa_dims bad = d;
    bad.group = 5;
    if (qsa_get_stats(&d, visible, &st) != QSA_OK) return 2;
    printf("%zu %lld %d %lld %lld %lld %zu %s\n", qsa_workspace_size(&d), (long long)qsa_score_stride(&d),
           (int)qsa_row_capacity(&d), (long long)st.selected_tokens, (long long)st.raw_key_bytes,
           (long long)st.dense_mask_bytes, qsa_workspace_size(&bad),
           qsa_status_string(QSA_ERR_WORKSPACE_TOO_SMALL) != NULL ? "named" : "null");
    return 0;
}
"""


def test_plain_c_client_links_and_calls_the_abi(lib, tmp_path):
    """The boundary is a C ABI: a C99 program (no C++, no torch) includes
    qsa.h, links libqsa.so and calls its host-only entry points; the answers
    equal the binding's and the closed forms."""
    import shutil
    import subprocess
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "client.c"
    src.write_text(_C_CLIENT)
    exe = tmp_path / "client"
    libdir = os.path.dirname(qsa.library_path())
    inc = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(qsa.__file__))), "include")
    subprocess.run([gcc, "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", inc, str(src),
                    "-o", str(exe), "-L", libdir, "-lqsa", "-Wl,-rpath," + libdir], check=True)
    out = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split()
    d = _dims()
    assert int(out[0]) == qsa.qsa_workspace_size(d)
    assert int(out[1]) == qsa.qsa_score_stride(d) == 65536
    assert int(out[2]) == qsa.qsa_row_capacity(d) == 2051
    assert int(out[3]) == 8 * 2048                    # 512 groups x 4 tokens, no tail
    assert int(out[4]) == 8 * 262144 * 64 * 4         # the raw keys the scorer streams
    assert int(out[5]) == 0                           # no query-by-key mask
    assert int(out[6]) == 0 and out[7] == "named"


def test_empty_batch_enqueues_nothing(lib):
    """B = 0: every compute call checks its arguments and returns OK without
    any CUDA call -- so it succeeds on this machine, which has no GPU.  The
    device pointers (aligned, never dereferenced) and the workspace size are
    those a caller would pass."""
    import ctypes
    L = qsa.load()
    d = _dims(batch=0, max_visible=1000)
    fake = 1 << 20
    inp = qsa.QsaInputs(q_idx=fake, idx_keys=fake, key_offset=fake, visible=fake, q=fake, k_cache=fake,
                        v_cache=fake, num_slots=1000, slot_map=fake, slot_offset=fake)
    ws_bytes = L.qsa_workspace_size(ctypes.byref(d))
    assert ws_bytes > 0
    for name in ("qsa_score_groups", "qsa_select", "qsa_gather", "qsa_attend", "qsa_gather_attend",
                 "qsa_attend_state", "qsa_decode", "qsa_decode_pooled", "qsa_decode_shared", "qsa_pool_groups",
                 "qsa_score_pooled", "qsa_score_groups_shared"):
        fn = getattr(L, name)
        args = []
        for t in fn.argtypes:
            if t is ctypes.c_size_t:
                args.append(ws_bytes)
            elif t in (ctypes.c_int32, ctypes.c_int, ctypes.c_int64):
                args.append(0)
            elif getattr(t, "_type_", None) is qsa.QsaDims:
                args.append(ctypes.byref(d))
            elif getattr(t, "_type_", None) is qsa.QsaInputs:
                args.append(ctypes.byref(inp))
            else:
                args.append(ctypes.c_void_p(fake))
        args[-1] = None  # the legacy default stream
        assert fn(*args) == qsa.QSA_OK, name
