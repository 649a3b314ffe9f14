"""Thin ctypes binding of libqsa (``include/qsa.h``) -- argument marshalling only.

Every function carries the name of the C entry point it calls and does
nothing but turn torch tensors (device memory) and plain Python values into
the C arguments; every step of the path runs in the library's CUDA kernels.
The library is loaded on first use; if it is missing or fails to load, the
call raises -- there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

__all__ = [
    "QsaError", "QsaDims", "QsaInputs", "QsaStats", "load", "library_path", "exported_symbols",
    "qsa_workspace_size", "qsa_score_stride", "qsa_row_capacity", "qsa_get_stats", "qsa_get_stats_pooled",
    "qsa_status_string", "qsa_workspace_init", "qsa_check_errors", "qsa_score_groups",
    "qsa_select", "qsa_gather", "qsa_attend", "qsa_gather_attend", "qsa_attend_state", "qsa_merge_states", "qsa_selftest_copy_timeout", "qsa_decode",
    "qsa_decode_profiled", "qsa_attend_noalloc", "qsa_pool_groups", "qsa_score_pooled",
    "qsa_decode_pooled", "qsa_score_groups_shared", "qsa_decode_shared", "qsa_probe_ffma",
    "make_dims",
    "DeviceBatch",
    "QSA_DEVERR_VISIBLE_RANGE", "QSA_DEVERR_SLOT_RANGE", "QSA_DEVERR_ROW_RANGE", "QSA_DEVERR_NOT_SHARED",
    "QSA_DEVERR_WAIT_TIMEOUT",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG, "_build", "libqsa.so")

QSA_OK = 0
QSA_ERR_DEVICE_FAULT = 5
QSA_DEVERR_VISIBLE_RANGE = 0x1
QSA_DEVERR_SLOT_RANGE = 0x2
QSA_DEVERR_ROW_RANGE = 0x4
QSA_DEVERR_WAIT_TIMEOUT = 0x8
QSA_DEVERR_NOT_SHARED = 0x10


class QsaError(RuntimeError):
    def __init__(self, fn: str, status: int, msg: str):
        super().__init__(f"{fn}: status {status}: {msg}")
        self.status = status


class QsaDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("idx_heads", ctypes.c_int32),
                ("idx_dim", ctypes.c_int32), ("q_heads", ctypes.c_int32),
                ("kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("group", ctypes.c_int32), ("budget_groups", ctypes.c_int32),
                ("max_visible", ctypes.c_int32), ("scale", ctypes.c_float)]


class QsaInputs(ctypes.Structure):
    _fields_ = [("q_idx", ctypes.c_void_p), ("idx_keys", ctypes.c_void_p),
                ("key_offset", ctypes.c_void_p), ("visible", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("k_cache", ctypes.c_void_p),
                ("v_cache", ctypes.c_void_p), ("num_slots", ctypes.c_int64),
                ("slot_map", ctypes.c_void_p), ("slot_offset", ctypes.c_void_p)]


class QsaStats(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int64) for n in (
        "candidate_groups", "selected_groups", "selected_tokens", "raw_key_bytes", "kv_bytes",
        "pooled_key_bytes", "workspace_bytes", "total_bytes", "dense_mask_bytes")]

    def as_dict(self):
        return {n: int(getattr(self, n)) for n, _ in self._fields_}


_lib = None
_P = ctypes.c_void_p
_DP = ctypes.POINTER(QsaDims)
_IP = ctypes.POINTER(QsaInputs)


def library_path() -> str:
    return _LIB_PATH


def load(path: str | None = None):
    """Load libqsa.so (raises if it is not built or cannot be loaded)."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or _LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(f"libqsa.so is not built ({p}); run __graft_entry__.build() first")
    L = ctypes.CDLL(p)
    L.qsa_workspace_size.argtypes = [_DP]
    L.qsa_workspace_size.restype = ctypes.c_size_t
    L.qsa_score_stride.argtypes = [_DP]
    L.qsa_score_stride.restype = ctypes.c_int64
    L.qsa_row_capacity.argtypes = [_DP]
    L.qsa_row_capacity.restype = ctypes.c_int32
    L.qsa_get_stats.argtypes = [_DP, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(QsaStats)]
    L.qsa_get_stats.restype = ctypes.c_int
    L.qsa_get_stats_pooled.argtypes = [_DP, ctypes.POINTER(ctypes.c_int32), ctypes.c_int64, ctypes.POINTER(QsaStats)]
    L.qsa_get_stats_pooled.restype = ctypes.c_int
    L.qsa_status_string.argtypes = [ctypes.c_int]
    L.qsa_status_string.restype = ctypes.c_char_p
    L.qsa_workspace_init.argtypes = [_P, ctypes.c_size_t, _P]
    L.qsa_workspace_init.restype = ctypes.c_int
    L.qsa_check_errors.argtypes = [_P, ctypes.c_size_t, _P, ctypes.POINTER(ctypes.c_uint32)]
    L.qsa_check_errors.restype = ctypes.c_int
    L.qsa_score_groups.argtypes = [_DP, _IP, _P, _P, ctypes.c_size_t, _P]
    L.qsa_score_groups.restype = ctypes.c_int
    L.qsa_select.argtypes = [_DP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.qsa_select.restype = ctypes.c_int
    L.qsa_gather.argtypes = [_DP, _IP, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.qsa_gather.restype = ctypes.c_int
    L.qsa_attend.argtypes = [_DP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.qsa_attend.restype = ctypes.c_int
    L.qsa_gather_attend.argtypes = [_DP, _IP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.qsa_gather_attend.restype = ctypes.c_int
    L.qsa_attend_state.argtypes = [_DP, _IP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.qsa_attend_state.restype = ctypes.c_int
    L.qsa_merge_states.argtypes = [_DP, ctypes.c_int32, _P, _P, _P, _P, _P]
    L.qsa_selftest_copy_timeout.argtypes = [_DP, _IP, _P, _P, ctypes.c_size_t, ctypes.c_uint64, _P]
    L.qsa_selftest_copy_timeout.restype = ctypes.c_int
    L.qsa_merge_states.restype = ctypes.c_int
    L.qsa_decode.argtypes = [_DP, _IP, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.qsa_decode.restype = ctypes.c_int
    L.qsa_decode_profiled.argtypes = [_DP, _IP, _P, _P, _P, _P, ctypes.c_size_t, _P,
                                      ctypes.POINTER(ctypes.c_void_p), ctypes.c_int32]
    L.qsa_decode_profiled.restype = ctypes.c_int
    L.qsa_attend_noalloc.argtypes = [_DP, _P, _P, _P, _P, _P, _P]
    L.qsa_attend_noalloc.restype = ctypes.c_int
    L.qsa_pool_groups.argtypes = [_DP, _IP, _P, _P, ctypes.c_int32, _P, _P, _P, ctypes.c_size_t, _P]
    L.qsa_pool_groups.restype = ctypes.c_int
    L.qsa_score_pooled.argtypes = [_DP, _IP, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.qsa_score_pooled.restype = ctypes.c_int
    L.qsa_decode_pooled.argtypes = [_DP, _IP, _P, _P, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.qsa_decode_pooled.restype = ctypes.c_int
    L.qsa_score_groups_shared.argtypes = [_DP, _IP, _P, _P, ctypes.c_size_t, _P]
    L.qsa_score_groups_shared.restype = ctypes.c_int
    L.qsa_decode_shared.argtypes = [_DP, _IP, _P, _P, _P, _P, ctypes.c_size_t, _P]
    L.qsa_decode_shared.restype = ctypes.c_int
    L.qsa_probe_ffma.argtypes = [ctypes.c_int32, ctypes.c_int32, _P, ctypes.POINTER(ctypes.c_int64), _P]
    L.qsa_probe_ffma.restype = ctypes.c_int
    if path is None:
        _lib = L
    return L


def exported_symbols(header: str | None = None) -> list[str]:
    """Names of the functions include/qsa.h (or the given header) declares."""
    import re
    header = header or os.path.join(os.path.dirname(_PKG), "include", "qsa.h")
    text = open(header).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(qsa_[a-z_]+)\s*\(", text)))


# ---- marshalling helpers ----------------------------------------------------

def _ptr(x) -> int | None:
    if x is None:
        return None
    if isinstance(x, int):
        return x
    return int(x.data_ptr())


def _stream(stream) -> int | None:
    if stream is None:
        import torch
        return int(torch.cuda.current_stream().cuda_stream)
    if isinstance(stream, int):
        return stream
    return int(stream.cuda_stream)


def _ws(ws):
    """(pointer, bytes) of a workspace given as a tensor or a (ptr, bytes) pair."""
    if isinstance(ws, tuple):
        return ws
    return _ptr(ws), ws.numel() * ws.element_size()


def _check(fn: str, st: int):
    if st != QSA_OK:
        raise QsaError(fn, st, load().qsa_status_string(st).decode())
    return st


def make_dims(batch, idx_heads, idx_dim, q_heads, kv_heads, head_dim, budget_groups=512,
              max_visible=0, scale=None, group=4) -> QsaDims:
    if scale is None:
        scale = float(np.float32(1.0 / np.sqrt(head_dim)))
    return QsaDims(int(batch), int(idx_heads), int(idx_dim), int(q_heads), int(kv_heads),
                   int(head_dim), int(group), int(budget_groups), int(max_visible), float(scale))


# ---- the C entry points -----------------------------------------------------

def qsa_workspace_size(dims: QsaDims) -> int:
    return int(load().qsa_workspace_size(ctypes.byref(dims)))


def qsa_score_stride(dims: QsaDims) -> int:
    return int(load().qsa_score_stride(ctypes.byref(dims)))


def qsa_row_capacity(dims: QsaDims) -> int:
    return int(load().qsa_row_capacity(ctypes.byref(dims)))


def qsa_get_stats(dims: QsaDims, visible_host) -> dict:
    vis = np.ascontiguousarray(np.asarray(visible_host, dtype=np.int32))
    st = QsaStats()
    _check("qsa_get_stats", load().qsa_get_stats(
        ctypes.byref(dims), vis.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), ctypes.byref(st)))
    return st.as_dict()


def qsa_get_stats_pooled(dims: QsaDims, visible_host, pooled_rows: int) -> dict:
    vis = np.ascontiguousarray(np.asarray(visible_host, dtype=np.int32))
    st = QsaStats()
    _check("qsa_get_stats_pooled", load().qsa_get_stats_pooled(
        ctypes.byref(dims), vis.ctypes.data_as(ctypes.POINTER(ctypes.c_int32)), int(pooled_rows),
        ctypes.byref(st)))
    return st.as_dict()


def qsa_status_string(status: int) -> str:
    return load().qsa_status_string(int(status)).decode()


def qsa_workspace_init(ws, stream=None) -> int:
    p, n = _ws(ws)
    return _check("qsa_workspace_init", load().qsa_workspace_init(p, n, _stream(stream)))


def qsa_check_errors(ws, stream=None) -> tuple[int, int]:
    """Returns (status, flags); does not raise on QSA_ERR_DEVICE_FAULT."""
    p, n = _ws(ws)
    flags = ctypes.c_uint32(0)
    st = load().qsa_check_errors(p, n, _stream(stream), ctypes.byref(flags))
    if st not in (QSA_OK, QSA_ERR_DEVICE_FAULT):
        _check("qsa_check_errors", st)
    return int(st), int(flags.value)


def qsa_score_groups(dims, inputs, scores, ws, stream=None) -> int:
    p, n = _ws(ws)
    return _check("qsa_score_groups", load().qsa_score_groups(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(scores), p, n, _stream(stream)))


def qsa_select(dims, visible, scores, ids, n_ids, ws, stream=None) -> int:
    p, n = _ws(ws)
    return _check("qsa_select", load().qsa_select(
        ctypes.byref(dims), _ptr(visible), _ptr(scores), _ptr(ids), _ptr(n_ids), p, n,
        _stream(stream)))


def qsa_gather(dims, inputs, ids, n_ids, k_scr, v_scr, ws, stream=None) -> int:
    p, n = _ws(ws)
    return _check("qsa_gather", load().qsa_gather(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(ids), _ptr(n_ids), _ptr(k_scr),
        _ptr(v_scr), p, n, _stream(stream)))


def qsa_attend(dims, q, k_scr, v_scr, n_ids, out, ws, stream=None) -> int:
    p, n = _ws(ws)
    return _check("qsa_attend", load().qsa_attend(
        ctypes.byref(dims), _ptr(q), _ptr(k_scr), _ptr(v_scr), _ptr(n_ids), _ptr(out), p, n,
        _stream(stream)))


def qsa_gather_attend(dims, inputs, ids, n_ids, k_scr, v_scr, out, ws, stream=None) -> int:
    p, n = _ws(ws)
    return _check("qsa_gather_attend", load().qsa_gather_attend(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(ids), _ptr(n_ids), _ptr(k_scr), _ptr(v_scr),
        _ptr(out), p, n, _stream(stream)))


def qsa_attend_state(dims, inputs, ids, n_ids, acc, m, l, ws, stream=None) -> int:
    """Online-softmax state (acc [B, n_q, d], m [B, n_q], l [B, n_q]) of each
    query's rows ids[b, :n_ids[b]], resolved through the slot map."""
    p, n = _ws(ws)
    return _check("qsa_attend_state", load().qsa_attend_state(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(ids), _ptr(n_ids), _ptr(acc), _ptr(m), _ptr(l),
        p, n, _stream(stream)))


def qsa_selftest_copy_timeout(dims, inputs, scores, ws, wait_ns, stream=None) -> int:
    """The failure-detection self-test (include/qsa_selftest.h): the raw scorer
    with no copy issued, so that every CTA's bounded wait runs out after wait_ns."""
    p, n = _ws(ws)
    return _check("qsa_selftest_copy_timeout", load().qsa_selftest_copy_timeout(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(scores), p, n, int(wait_ns), _stream(stream)))


def qsa_merge_states(dims, n_parts, m, l, acc, out, stream=None) -> int:
    """Output [B, n_q, d] of rows whose consecutive slices' states are
    m, l [n_parts, B, n_q] and acc [n_parts, B, n_q, d], merged in slice order."""
    return _check("qsa_merge_states", load().qsa_merge_states(
        ctypes.byref(dims), int(n_parts), _ptr(m), _ptr(l), _ptr(acc), _ptr(out), _stream(stream)))


def qsa_decode(dims, inputs, ids, n_ids, out, ws, stream=None) -> int:
    p, n = _ws(ws)
    return _check("qsa_decode", load().qsa_decode(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(ids), _ptr(n_ids), _ptr(out), p, n,
        _stream(stream)))


def qsa_decode_profiled(dims, inputs, ids, n_ids, out, ws, events, stream=None) -> int:
    """events: four torch.cuda.Event(enable_timing=True) (or raw cudaEvent_t ints)."""
    handles = []
    for e in events:
        if isinstance(e, int):
            handles.append(e)
        else:
            if not e.cuda_event:  # torch creates the CUDA event on first record
                e.record()
            handles.append(int(e.cuda_event))
    arr = (ctypes.c_void_p * len(handles))(*handles)
    p, n = _ws(ws)
    return _check("qsa_decode_profiled", load().qsa_decode_profiled(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(ids), _ptr(n_ids), _ptr(out), p, n,
        _stream(stream), arr, len(handles)))


def qsa_pool_groups(dims, inputs, group_begin, group_end, max_groups, pooled, pool_offset, ws,
                    stream=None) -> int:
    p, n = _ws(ws)
    return _check("qsa_pool_groups", load().qsa_pool_groups(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(group_begin), _ptr(group_end), int(max_groups),
        _ptr(pooled), _ptr(pool_offset), p, n, _stream(stream)))


def qsa_score_pooled(dims, inputs, pooled, pool_offset, scores, ws, stream=None) -> int:
    p, n = _ws(ws)
    return _check("qsa_score_pooled", load().qsa_score_pooled(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(pooled), _ptr(pool_offset), _ptr(scores), p, n,
        _stream(stream)))


def qsa_decode_pooled(dims, inputs, pooled, pool_offset, ids, n_ids, out, ws, stream=None) -> int:
    p, n = _ws(ws)
    return _check("qsa_decode_pooled", load().qsa_decode_pooled(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(pooled), _ptr(pool_offset), _ptr(ids),
        _ptr(n_ids), _ptr(out), p, n, _stream(stream)))


def qsa_score_groups_shared(dims, inputs, scores, ws, stream=None) -> int:
    p, n = _ws(ws)
    return _check("qsa_score_groups_shared", load().qsa_score_groups_shared(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(scores), p, n, _stream(stream)))


def qsa_decode_shared(dims, inputs, ids, n_ids, out, ws, stream=None) -> int:
    p, n = _ws(ws)
    return _check("qsa_decode_shared", load().qsa_decode_shared(
        ctypes.byref(dims), ctypes.byref(inputs), _ptr(ids), _ptr(n_ids), _ptr(out), p, n,
        _stream(stream)))


def qsa_probe_ffma(blocks_per_sm, iters, sink, stream=None) -> int:
    """Launches the FFMA throughput probe; returns the FMAs it performs."""
    count = ctypes.c_int64(0)
    _check("qsa_probe_ffma", load().qsa_probe_ffma(int(blocks_per_sm), int(iters), _ptr(sink),
                                                   ctypes.byref(count), _stream(stream)))
    return int(count.value)


def qsa_attend_noalloc(dims, q, k_scr, v_scr, n_ids, out, stream=None) -> int:
    """Attention stage with the library's fixed static scratch instead of a
    workspace, for callers that cannot allocate device memory."""
    return _check("qsa_attend_noalloc", load().qsa_attend_noalloc(
        ctypes.byref(dims), _ptr(q), _ptr(k_scr), _ptr(v_scr), _ptr(n_ids), _ptr(out),
        _stream(stream)))


# ---- device-resident batch (plumbing: torch owns the memory) ----------------

def _packed(arrays, device):
    """One uint8 device buffer holding the given (name, numpy array or
    (shape, dtype, fill)) items back to back, each on a 16-byte boundary;
    returns (buffer, {name: typed view})."""
    import torch
    items, off = [], 0
    for name, a in arrays:
        if isinstance(a, tuple):
            shape, dtype, fill = a
            nbytes = int(np.prod(shape)) * np.dtype(dtype).itemsize
        else:
            a = np.ascontiguousarray(a)
            shape, dtype, fill, nbytes = a.shape, a.dtype, None, a.nbytes
        off = (off + 15) // 16 * 16
        items.append((name, off, shape, dtype, fill, a))
        off += nbytes
    buf = torch.zeros(max(off, 16), dtype=torch.uint8, device=device)
    views = {}
    tdt = {np.dtype(np.float32): torch.float32, np.dtype(np.int32): torch.int32,
           np.dtype(np.int64): torch.int64}
    for name, o, shape, dtype, fill, a in items:
        n = int(np.prod(shape)) * np.dtype(dtype).itemsize
        v = buf[o:o + n].view(tdt[np.dtype(dtype)]).view(tuple(shape))
        if fill is None:
            v.copy_(torch.from_numpy(a))
        else:
            v.fill_(fill)
        views[name] = v
    return buf, views


class DeviceBatch:
    """The arrays of one workload copied into device memory, with the output
    buffers and the workspace the library needs, all allocated by torch.

    A decode step's own inputs (q_idx, q, visible, key_offset, slot_offset)
    share one buffer, `step_in`, and its outputs (ids, n_ids, out) another,
    `step_out`: a step driven from host memory is one copy in and one copy
    out (`step_host_buffers`, `decode_from_host`)."""

    def __init__(self, w, device="cuda", budget=None, queries=None):
        import torch
        self.w = w
        sel = np.arange(w.batch) if queries is None else np.asarray(queries, np.int64)
        dev = torch.device(device)

        def put(a):
            return torch.from_numpy(np.ascontiguousarray(a)).to(dev)

        self.step_in, v = _packed([("q_idx", w.q_idx[sel]), ("q", w.q[sel]),
                                   ("visible", w.visible[sel]), ("key_offset", w.key_offset[sel]),
                                   ("slot_offset", w.slot_offset[sel])], dev)
        self.q_idx, self.q, self.visible = v["q_idx"], v["q"], v["visible"]
        self.key_offset, self.slot_offset = v["key_offset"], v["slot_offset"]
        self.idx_keys = put(w.idx_keys)
        self.k_cache = put(w.k_cache)
        self.v_cache = put(w.v_cache)
        self.slot_map = put(w.slot_map)
        B = len(sel)
        mv = int(w.visible[sel].max(initial=0))
        self.dims = make_dims(B, w.idx_heads, w.idx_dim, w.q_heads, w.kv_heads, w.head_dim,
                              budget_groups=w.budget if budget is None else budget,
                              max_visible=max(mv, w.max_visible if queries is None else mv),
                              scale=w.scale)
        self.inputs = QsaInputs(
            _ptr(self.q_idx), _ptr(self.idx_keys), _ptr(self.key_offset), _ptr(self.visible),
            _ptr(self.q), _ptr(self.k_cache), _ptr(self.v_cache), int(w.num_slots),
            _ptr(self.slot_map), _ptr(self.slot_offset))
        self.row_cap = qsa_row_capacity(self.dims)
        self.score_stride = qsa_score_stride(self.dims)
        nbytes = qsa_workspace_size(self.dims)
        if nbytes == 0:
            raise ValueError("invalid dims")
        # zero-filled: the workspace header must start clean
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
        self.step_out, v = _packed([("ids", ((B, self.row_cap), np.int32, -1)),
                                    ("n_ids", ((B,), np.int32, -1)),
                                    ("out", ((B, w.q_heads, w.head_dim), np.float32, float("nan")))], dev)
        self.ids, self.n_ids, self.out = v["ids"], v["n_ids"], v["out"]
        self.scores = torch.full((B, self.score_stride), float("nan"), dtype=torch.float32, device=dev)
        self.k_scr = torch.zeros((B, self.row_cap, w.kv_heads, w.head_dim), dtype=torch.float32, device=dev)
        self.v_scr = torch.zeros_like(self.k_scr)

    # a decode step driven from host memory: one copy in, one copy out
    def step_host_buffers(self):
        """Pinned host buffers laid out like step_in (holding this batch's
        current step inputs) and step_out."""
        import torch
        h_in = torch.empty(self.step_in.shape, dtype=torch.uint8).pin_memory()
        h_in.copy_(self.step_in)
        h_out = torch.empty(self.step_out.shape, dtype=torch.uint8).pin_memory()
        return h_in, h_out

    def step_slot(self):
        """A second device buffer laid out like step_in (holding the same step
        inputs) and the QsaInputs that point into it -- the history, the K/V
        caches and the slot map stay shared -- so that two host-driven steps
        can be in flight at once: one step's inputs copied in while the other
        step's kernels run.  Returns (buffer, inputs)."""
        buf = self.step_in.clone()
        base = self.step_in.data_ptr()

        def at(t):
            return buf.data_ptr() + (t.data_ptr() - base)

        inp = QsaInputs(at(self.q_idx), _ptr(self.idx_keys), at(self.key_offset), at(self.visible), at(self.q),
                        _ptr(self.k_cache), _ptr(self.v_cache), int(self.inputs.num_slots), _ptr(self.slot_map),
                        at(self.slot_offset))
        return buf, inp

    def decode_from_host(self, h_in, h_out, stream=None):
        """One step on the current torch stream (or `stream`): the step's
        inputs from h_in, qsa_decode, the ID rows, counts and outputs to
        h_out (both copies asynchronous; synchronise before reading h_out)."""
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        with torch.cuda.stream(s):
            self.step_in.copy_(h_in, non_blocking=True)
            self.decode(s)
            h_out.copy_(self.step_out, non_blocking=True)

    def decode_into_host(self, h_in, h_out, stream=None):
        """One step on the current torch stream (or `stream`): the step's
        inputs copied in from h_in, then qsa_decode with its ID rows, counts
        and outputs pointing straight into the pinned host buffer h_out (laid
        out like step_out): the last kernel stores them there, so no copy
        follows.  Synchronise before reading h_out."""
        import torch
        s = stream if stream is not None else torch.cuda.current_stream()
        hi, hn, ho = self.host_outputs(h_out)
        with torch.cuda.stream(s):
            self.step_in.copy_(h_in, non_blocking=True)
            qsa_decode(self.dims, self.inputs, hi, hn, ho, self.ws, s)

    def capture_decode_from_host(self, h_in, h_out, direct=False):
        """A CUDA graph of one host-driven step (copy in, qsa_decode, copy
        out), for a loop that repeats it: `g.replay()` on the current stream
        launches the whole step at once.  Run one eager step first (the
        library's one-time per-device setup must not happen during capture).
        The step reads the per-SM scorer weights from the workspace when it
        runs, so replays keep learning them."""
        import torch
        g = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            with torch.cuda.graph(g, stream=s):
                if direct:
                    self.decode_into_host(h_in, h_out, s)
                else:
                    self.decode_from_host(h_in, h_out, s)
        torch.cuda.current_stream().wait_stream(s)
        return g

    def host_outputs(self, h_out):
        """(ids, n_ids, out) views of a host buffer laid out like step_out."""
        import torch
        res = []
        for t in (self.ids, self.n_ids, self.out):
            o = t.data_ptr() - self.step_out.data_ptr()
            n = t.numel() * t.element_size()
            res.append(h_out[o:o + n].view(t.dtype).view(t.shape))
        return tuple(res)

    # the four stages and the whole path, on this batch's buffers
    def score(self, stream=None):
        return qsa_score_groups(self.dims, self.inputs, self.scores, self.ws, stream)

    def select(self, stream=None):
        return qsa_select(self.dims, self.visible, self.scores, self.ids, self.n_ids, self.ws, stream)

    def gather(self, stream=None):
        return qsa_gather(self.dims, self.inputs, self.ids, self.n_ids, self.k_scr, self.v_scr,
                          self.ws, stream)

    def attend(self, stream=None):
        return qsa_attend(self.dims, self.q, self.k_scr, self.v_scr, self.n_ids, self.out,
                          self.ws, stream)

    def gather_attend(self, stream=None):
        return qsa_gather_attend(self.dims, self.inputs, self.ids, self.n_ids, self.k_scr,
                                 self.v_scr, self.out, self.ws, stream)

    def decode(self, stream=None):
        return qsa_decode(self.dims, self.inputs, self.ids, self.n_ids, self.out, self.ws, stream)

    def decode_profiled(self, events, stream=None):
        return qsa_decode_profiled(self.dims, self.inputs, self.ids, self.n_ids, self.out, self.ws,
                                   events, stream)

    # ---- the incremental form: a pooled-key cache -----------------------------
    def make_pooled_cache(self):
        """Allocates the pooled-key cache: one block of rows per distinct
        history (queries that share a history share its rows), room for the
        longest T over the queries of that history."""
        import torch
        ko = self.key_offset.cpu().numpy()
        T = self.visible.cpu().numpy()
        base, rows = {}, 0
        for k in sorted(set(ko.tolist())):
            base[k] = rows
            rows += int(T[ko == k].max()) // 4
        self.pool_offset = torch.from_numpy(np.array([base[k] for k in ko.tolist()], np.int64)).to(self.q.device)
        self.pooled = torch.zeros((max(rows, 1), self.w.idx_dim), dtype=torch.float32, device=self.q.device)
        # the query of each history with the longest T pools the history's groups
        owner = {}
        for b, k in enumerate(ko.tolist()):
            if k not in owner or T[b] > T[owner[k]]:
                owner[k] = b
        self._pool_owner = np.array([owner[k] == b for b, k in enumerate(ko.tolist())])
        return self.pooled

    def pool(self, group_begin, group_end, stream=None):
        """Appends groups [group_begin[b], group_end[b]) of every query (host arrays)."""
        import torch
        gb = np.asarray(group_begin, np.int32)
        ge = np.asarray(group_end, np.int32)
        mg = int((ge - gb).max(initial=0))
        dev = self.q.device
        self._pool_args = (torch.from_numpy(gb).to(dev), torch.from_numpy(ge).to(dev))
        return qsa_pool_groups(self.dims, self.inputs, self._pool_args[0], self._pool_args[1], max(mg, 0),
                               self.pooled, self.pool_offset, self.ws, stream)

    def pool_all(self, stream=None):
        """Pools every complete group of every history (once per history)."""
        G = (self.visible.cpu().numpy() // 4).astype(np.int32)
        ge = np.where(self._pool_owner, G, 0).astype(np.int32)
        return self.pool(np.zeros_like(ge), ge, stream)

    def score_pooled(self, stream=None):
        return qsa_score_pooled(self.dims, self.inputs, self.pooled, self.pool_offset, self.scores,
                                self.ws, stream)

    def decode_pooled(self, stream=None):
        return qsa_decode_pooled(self.dims, self.inputs, self.pooled, self.pool_offset, self.ids,
                                 self.n_ids, self.out, self.ws, stream)

    # ---- queries over one shared history ------------------------------------
    def score_shared(self, stream=None):
        return qsa_score_groups_shared(self.dims, self.inputs, self.scores, self.ws, stream)

    def decode_shared(self, stream=None):
        return qsa_decode_shared(self.dims, self.inputs, self.ids, self.n_ids, self.out, self.ws, stream)

    def check_errors(self, stream=None):
        return qsa_check_errors(self.ws, stream)
