"""ctypes wrapper of the plain C oracle (``qsa_oracle.c``) -- test infrastructure.

The oracle is the slow, sequential CPU definition of physically sparse QSA
decode written from the notes "Top-k chooses the set; time chooses the
order" (AFN-017) and "A sparse mask is not sparse attention" (AFN-016).
Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may use it; it shares no code with the CUDA library.

Everything here is argument marshalling around the C functions, plus the
build step (gcc, ``-O2 -ffp-contract=off``).
"""
from __future__ import annotations

import ctypes
import os
import platform
import shutil
import subprocess
import tempfile

import numpy as np

__all__ = [
    "build", "lib", "num_groups", "tail_len", "row_width", "pool_group",
    "score_groups", "score_groups_incremental", "pool_cache", "select", "dense_ids",
    "resolve", "attend", "attend_partial", "merge_states", "decode", "threads", "GROUP",
]

GROUP = 4
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qsa_oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_SO = os.path.join(_OUT_DIR, "libqsa_oracle.so")

_lib = None


def _cflags() -> list[str]:
    flags = ["-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]
    if _has_openmp():
        flags.append("-fopenmp")  # the per-group scoring loop, shared among host threads
    # fmaf() is correctly rounded by definition; on x86-64 the FMA extension
    # only turns the libm call into one instruction with the same result.
    if platform.machine() in ("x86_64", "AMD64"):
        flags.append("-mfma")
    return flags


def _has_openmp() -> bool:
    """Whether gcc here builds and links OpenMP code."""
    global _omp
    if _omp is None:
        d = tempfile.mkdtemp()
        try:
            c = os.path.join(d, "t.c")
            open(c, "w").write("#include <omp.h>\nint f(void){return omp_get_max_threads();}\n")
            r = subprocess.run(["gcc", "-fopenmp", "-fPIC", "-shared", c, "-o", os.path.join(d, "t.so")],
                               capture_output=True)
            _omp = r.returncode == 0
        finally:
            shutil.rmtree(d, ignore_errors=True)
    return _omp


_omp = None


def build(force: bool = False, sanitize: bool = False, out: str | None = None,
          src: str | None = None) -> str:
    """Compile ``qsa_oracle.c`` (or ``src``) into a shared library; return its path."""
    so = out or _SO
    src = src or _SRC
    if not force and os.path.exists(so) and os.path.getmtime(so) >= os.path.getmtime(src):
        return so
    os.makedirs(os.path.dirname(so), exist_ok=True)
    flags = _cflags()
    if sanitize:  # (single-threaded: the sanitizers see the plain loops)
        flags = [f for f in flags if f not in ("-O2", "-fopenmp")] + [
            "-O1", "-g", "-fsanitize=address,undefined", "-fno-omit-frame-pointer",
            "-fno-sanitize-recover=all"]
    fd, tmp = tempfile.mkstemp(suffix=".so", dir=os.path.dirname(so))
    os.close(fd)
    try:
        subprocess.run(["gcc", *flags, src, "-o", tmp, "-lm"], check=True)
        os.replace(tmp, so)
    finally:
        if os.path.exists(tmp):
            os.unlink(tmp)
    return so


_F32P = ctypes.POINTER(ctypes.c_float)
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)
_i32, _i64, _f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float


def _declare(L):
    L.qsao_num_groups.argtypes = [_i32]
    L.qsao_num_groups.restype = _i32
    L.qsao_tail_len.argtypes = [_i32]
    L.qsao_tail_len.restype = _i32
    L.qsao_row_width.argtypes = [_i32, _i32]
    L.qsao_row_width.restype = _i32
    L.qsao_pool_group.argtypes = [_F32P, _i32, _f32, _F32P]
    L.qsao_pool_group.restype = None
    L.qsao_score_pooled.argtypes = [_F32P, _i32, _i32, _F32P]
    L.qsao_score_pooled.restype = _f32
    L.qsao_score_groups.argtypes = [_F32P, _i32, _i32, _F32P, _i32, _f32, _F32P]
    L.qsao_score_groups.restype = None
    L.qsao_pool_cache_append.argtypes = [_F32P, _F32P, _i32, _F32P, _i32, _f32]
    L.qsao_pool_cache_append.restype = None
    L.qsao_score_from_pooled.argtypes = [_F32P, _i32, _i32, _F32P, _i32, _F32P]
    L.qsao_score_from_pooled.restype = None
    L.qsao_select.argtypes = [_F32P, _i32, _i32, _I32P, _I32P]
    L.qsao_select.restype = _i32
    L.qsao_dense_ids.argtypes = [_i32, _I32P]
    L.qsao_dense_ids.restype = _i32
    L.qsao_resolve.argtypes = [_I32P, _i32, _I32P, _i64, _I32P]
    L.qsao_resolve.restype = _i32
    L.qsao_attend.argtypes = [_F32P, _i32, _i32, _i32, _f32, _F32P, _F32P, _I32P, _i32, _F32P]
    L.qsao_attend.restype = None
    L.qsao_threads.argtypes = [_i32]
    L.qsao_threads.restype = _i32
    L.qsao_attend_partial.argtypes = [_F32P, _i32, _i32, _i32, _f32, _F32P, _F32P, _I32P, _i32,
                                      _F32P, _F32P, _F32P]
    L.qsao_attend_partial.restype = None
    L.qsao_merge_states.argtypes = [_i32, _i32, _i32, _F32P, _F32P, _F32P, _F32P]
    L.qsao_merge_states.restype = None
    L.qsao_decode.argtypes = [
        _i32, _i32, _i32, _i32, _i32, _i32, _i32, _f32,
        _F32P, _F32P, _I64P, _I32P, _F32P, _F32P, _F32P, _i64, _I32P, _I64P,
        _F32P, _i32, _I32P, _i32, _I32P, _F32P]
    L.qsao_decode.restype = _i32


def lib():
    """Load (building first if needed) the oracle shared library.

    QSA_ORACLE_LIB names another build of the same source to load instead;
    the mutation test uses it to run the pins against planted mistakes."""
    global _lib
    if _lib is None:
        L = ctypes.CDLL(os.environ.get("QSA_ORACLE_LIB") or build())
        _declare(L)
        _lib = L
    return _lib


def _fa(a):
    a = np.ascontiguousarray(a, dtype=np.float32)
    return a, a.ctypes.data_as(_F32P)


def _ia(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(_I32P)


def _la(a):
    a = np.ascontiguousarray(a, dtype=np.int64)
    return a, a.ctypes.data_as(_I64P)


def num_groups(T: int) -> int:
    return int(lib().qsao_num_groups(int(T)))


def tail_len(T: int) -> int:
    return int(lib().qsao_tail_len(int(T)))


def row_width(T: int, budget: int = 512) -> int:
    return int(lib().qsao_row_width(int(T), int(budget)))


def pool_group(k4: np.ndarray, pool_scale: float = 0.25) -> np.ndarray:
    """k4: [4, d] raw index keys of one group -> pooled key [d]."""
    k4, pk = _fa(k4)
    d = k4.shape[-1]
    p = np.empty(d, np.float32)
    lib().qsao_pool_group(pk, d, pool_scale, p.ctypes.data_as(_F32P))
    return p


def score_groups(q_idx: np.ndarray, keys: np.ndarray, T: int | None = None,
                 pool_scale: float = 0.25) -> np.ndarray:
    """q_idx [H, d], keys [>=T, d] (logical order) -> scores [floor(T/4)]."""
    q_idx, pq = _fa(q_idx)
    keys, pk = _fa(keys)
    H, d = q_idx.shape
    T = keys.shape[0] if T is None else int(T)
    assert keys.shape[0] >= T and keys.shape[1] == d
    G = T // GROUP
    s = np.empty(max(G, 1), np.float32)
    lib().qsao_score_groups(pq, H, d, pk, T, pool_scale, s.ctypes.data_as(_F32P))
    return s[:G]


def pool_cache(keys: np.ndarray, T: int, pool_scale: float = 0.25) -> np.ndarray:
    """The pooled-key cache of one history after T tokens, built one token at
    a time as a decode loop would ("full-raw / incremental identity"):
    [floor(T/4), d] pooled keys of the complete groups."""
    keys = np.ascontiguousarray(keys, dtype=np.float32)
    d = keys.shape[1]
    G = T // GROUP
    pooled = np.zeros((max(G, 1), d), np.float32)
    pending = np.zeros((GROUP, d), np.float32)
    L = lib()
    pp, pe = pooled.ctypes.data_as(_F32P), pending.ctypes.data_as(_F32P)
    for t in range(T):
        row = keys[t]
        L.qsao_pool_cache_append(pp, pe, d, row.ctypes.data_as(_F32P), t, pool_scale)
    return pooled[:G]


def score_groups_incremental(q_idx: np.ndarray, keys: np.ndarray, T: int,
                             pool_scale: float = 0.25) -> np.ndarray:
    """Same scores, read from a pooled-key cache built one token at a time."""
    q_idx, pq = _fa(q_idx)
    H, d = q_idx.shape
    G = T // GROUP
    pooled = np.ascontiguousarray(pool_cache(keys, T, pool_scale))
    if G == 0:
        pooled = np.zeros((1, d), np.float32)
    s = np.empty(max(G, 1), np.float32)
    lib().qsao_score_from_pooled(pq, H, d, pooled.ctypes.data_as(_F32P), G, s.ctypes.data_as(_F32P))
    return s[:G]


def select(scores: np.ndarray, T: int, budget: int = 512, return_chosen: bool = False):
    """scores [floor(T/4)] -> emitted logical token IDs (int32 [W])."""
    G = T // GROUP
    scores = np.ascontiguousarray(scores, dtype=np.float32)
    assert scores.shape[0] >= G
    cap = max(row_width(T, budget), 1)
    ids = np.empty(cap, np.int32)
    chosen = np.empty(max(min(G, budget), 1), np.int32)
    n = lib().qsao_select(scores.ctypes.data_as(_F32P), int(T), int(budget),
                          ids.ctypes.data_as(_I32P), chosen.ctypes.data_as(_I32P))
    if return_chosen:
        return ids[:n], chosen[:min(G, budget)]
    return ids[:n]


def dense_ids(T: int) -> np.ndarray:
    ids = np.empty(max(T, 1), np.int32)
    n = lib().qsao_dense_ids(int(T), ids.ctypes.data_as(_I32P))
    return ids[:n]


def resolve(ids: np.ndarray, slot_map: np.ndarray, num_slots: int):
    """Returns (status, slots); status 0 or -(i+1) for the first bad row."""
    ids, pi = _ia(ids)
    slot_map, ps = _ia(slot_map)
    slots = np.empty(max(len(ids), 1), np.int32)
    st = lib().qsao_resolve(pi, len(ids), ps, int(num_slots), slots.ctypes.data_as(_I32P))
    return int(st), slots[:len(ids)]


def attend(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
           slots: np.ndarray, scale: float) -> np.ndarray:
    """q [n_q, d]; caches [num_slots, n_kv, d]; slots in emitted order -> [n_q, d]."""
    q, pq = _fa(q)
    k_cache, pk = _fa(k_cache)
    v_cache, pv = _fa(v_cache)
    slots, ps = _ia(slots)
    n_q, d = q.shape
    n_kv = k_cache.shape[1]
    out = np.empty((n_q, d), np.float32)
    lib().qsao_attend(pq, n_q, n_kv, d, float(scale), pk, pv, ps, len(slots),
                      out.ctypes.data_as(_F32P))
    return out


def threads(n: int = 0) -> int:
    """Host threads the scoring loop uses (n > 0 sets it); 1 without OpenMP."""
    return int(lib().qsao_threads(int(n)))


def attend_partial(q: np.ndarray, k_cache: np.ndarray, v_cache: np.ndarray,
                   slots: np.ndarray, scale: float):
    """The online-softmax state (m [n_q], l [n_q], acc [n_q, d]) after the
    rows `slots` in order; attend() is acc / l of it."""
    q, pq = _fa(q)
    k_cache, pk = _fa(k_cache)
    v_cache, pv = _fa(v_cache)
    slots, ps = _ia(slots)
    n_q, d = q.shape
    n_kv = k_cache.shape[1]
    m = np.empty(n_q, np.float32)
    l = np.empty(n_q, np.float32)
    acc = np.empty((n_q, d), np.float32)
    lib().qsao_attend_partial(pq, n_q, n_kv, d, float(scale), pk, pv, ps, len(slots),
                              m.ctypes.data_as(_F32P), l.ctypes.data_as(_F32P),
                              acc.ctypes.data_as(_F32P))
    return m, l, acc


def merge_states(parts):
    """Output [n_q, d] of one row from the online-softmax states (m [n_q],
    l [n_q], acc [n_q, d]) of its consecutive slices, given in row order:
    each slice folded in as one more block of the online softmax."""
    n = len(parts)
    m = np.ascontiguousarray(np.stack([np.asarray(p[0], np.float32) for p in parts]))
    l = np.ascontiguousarray(np.stack([np.asarray(p[1], np.float32) for p in parts]))
    acc = np.ascontiguousarray(np.stack([np.asarray(p[2], np.float32) for p in parts]))
    n_q, d = acc.shape[1], acc.shape[2]
    out = np.empty((n_q, d), np.float32)
    lib().qsao_merge_states(n, n_q, d, m.ctypes.data_as(_F32P), l.ctypes.data_as(_F32P),
                            acc.ctypes.data_as(_F32P), out.ctypes.data_as(_F32P))
    return out


def decode(w, with_scores: bool = False, queries=None):
    """Whole decode of a workload (any object with the workload fields).

    queries: optional list of query indices to run (a sample of the batch).
    Returns dict(ids [b, row_cap], n_ids [b], out [b, n_q, d], status[, scores]).
    """
    sel = np.arange(w.batch) if queries is None else np.asarray(queries, np.int64)
    Bs = len(sel)
    H, dI = w.idx_heads, w.idx_dim
    n_q, n_kv, hd = w.q_heads, w.kv_heads, w.head_dim
    row_cap = GROUP * w.budget + GROUP - 1
    gstride = max(w.max_visible // GROUP, 1)
    q_idx, p_qidx = _fa(w.q_idx[sel])
    keys, p_keys = _fa(w.idx_keys)
    koff, p_koff = _la(w.key_offset[sel])
    vis, p_vis = _ia(w.visible[sel])
    q, p_q = _fa(w.q[sel])
    kc, p_kc = _fa(w.k_cache)
    vc, p_vc = _fa(w.v_cache)
    sm, p_sm = _ia(w.slot_map)
    soff, p_soff = _la(w.slot_offset[sel])
    ids = np.zeros((Bs, row_cap), np.int32)
    n_ids = np.zeros(Bs, np.int32)
    out = np.zeros((Bs, n_q, hd), np.float32)
    scores = np.zeros((Bs, gstride), np.float32) if with_scores else None
    st = lib().qsao_decode(
        Bs, H, dI, n_q, n_kv, hd, w.budget, float(w.scale),
        p_qidx, p_keys, p_koff, p_vis, p_q, p_kc, p_vc, int(w.num_slots), p_sm, p_soff,
        scores.ctypes.data_as(_F32P) if with_scores else None, gstride,
        ids.ctypes.data_as(_I32P), row_cap, n_ids.ctypes.data_as(_I32P),
        out.ctypes.data_as(_F32P))
    res = {"ids": ids, "n_ids": n_ids, "out": out, "status": int(st)}
    if with_scores:
        res["scores"] = scores
    return res
