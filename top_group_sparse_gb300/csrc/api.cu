// api.cu -- the extern "C" boundary of libqsa (declared in include/qsa.h).
//
// Host side only: argument validation (every host-detectable error returns a
// status before anything is enqueued), the workspace layout, and the launch
// of each stage's kernel on the caller's stream.  The library allocates
// nothing; all buffers, the workspace included, belong to the caller.
#include <cuda_runtime.h>

#include <cstring>

#include "qsa_internal.cuh"
#include "qsa_selftest.h"

namespace qsa {

bool dims_valid(const qsa_dims *d)
{
    if (!d) return false;
    if (d->batch < 0 || d->batch > 65535) return false;
    if (d->group != kGroup) return false;
    if (d->budget_groups < 1 || d->budget_groups > QSA_MAX_BUDGET) return false;
    if (d->max_visible < 0 || d->max_visible > QSA_MAX_VISIBLE) return false;
    if (d->idx_heads <= 0 || d->idx_dim <= 0 || d->q_heads <= 0 || d->kv_heads <= 0 || d->head_dim <= 0)
        return false;
    if (d->q_heads % d->kv_heads != 0) return false;
    if (!(d->scale == d->scale)) return false;  // NaN scale
    return true;
}

Layout make_layout(const qsa_dims *d)
{
    Layout L{};
    const int64_t gmax = d->max_visible / kGroup;
    L.score_stride = ((gmax + 31) / 32) * 32;
    if (L.score_stride == 0) L.score_stride = 32;
    L.row_cap = kGroup * d->budget_groups + (kGroup - 1);
    L.nparts = kAttendParts;
    const size_t B = size_t(d->batch);
    size_t off = 0;
    L.off_err = off;
    off += kWsAlign;
    L.off_tickets = off;
    off = align_up(off + B * size_t(d->kv_heads) * 4, kWsAlign);
    L.off_bal = off;
    off = align_up(off + sizeof(ScoreBalance), kWsAlign);
    const size_t nparts = B * size_t(d->q_heads) * size_t(L.nparts);
    L.off_part_m = off;
    off = align_up(off + nparts * 4, kWsAlign);
    L.off_part_l = off;
    off = align_up(off + nparts * 4, kWsAlign);
    L.off_part_acc = off;
    off = align_up(off + nparts * size_t(d->head_dim) * 4, kWsAlign);
    L.qmax_stride = ((gmax + 3) / 4 + 31) / 32 * 32;
    if (L.qmax_stride == 0) L.qmax_stride = 32;
    L.off_qmax = off;
    off = align_up(off + B * size_t(L.qmax_stride) * 4, kWsAlign);
    L.off_scores = off;
    off = align_up(off + B * size_t(L.score_stride) * 4, kWsAlign);
    L.off_ids = off;   // the whole-path call's ID rows and counts, before the caller's copy
    off = align_up(off + B * size_t(L.row_cap) * 4, kWsAlign);
    L.off_nids = off;
    off = align_up(off + B * 4, kWsAlign);
    L.total = off;
    return L;
}

namespace {

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int num_sms_of_current_device()
{
    static int cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev < 0 || dev >= 64) return 0;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cache[dev] = n;
    }
    return cache[dev];
}

qsa_status check_ws(const qsa_dims *d, void *ws, size_t ws_bytes)
{
    if (!ws || !aligned(ws, kWsAlign)) return QSA_ERR_INVALID_ARG;
    if (ws_bytes < make_layout(d).total) return QSA_ERR_WORKSPACE_TOO_SMALL;
    return QSA_OK;
}

qsa_status check_inputs_score(const qsa_inputs *in)
{
    if (!in || !in->q_idx || !in->idx_keys || !in->key_offset || !in->visible) return QSA_ERR_INVALID_ARG;
    if (!aligned(in->q_idx, 16) || !aligned(in->idx_keys, 16) || !aligned(in->key_offset, 8) ||
        !aligned(in->visible, 4))
        return QSA_ERR_INVALID_ARG;
    return QSA_OK;
}

// Scoring from the pooled-key cache reads q_idx and visible from `in`.
qsa_status check_inputs_pooled(const qsa_inputs *in, const float *pooled, const int64_t *pool_offset)
{
    if (!in || !in->q_idx || !in->visible || !pooled || !pool_offset) return QSA_ERR_INVALID_ARG;
    if (!aligned(in->q_idx, 16) || !aligned(in->visible, 4) || !aligned(pooled, 16) || !aligned(pool_offset, 8))
        return QSA_ERR_INVALID_ARG;
    return QSA_OK;
}

qsa_status check_inputs_gather(const qsa_inputs *in)
{
    if (!in || !in->visible || !in->k_cache || !in->v_cache || !in->slot_map || !in->slot_offset)
        return QSA_ERR_INVALID_ARG;
    if (in->num_slots < 0) return QSA_ERR_INVALID_ARG;
    if (!aligned(in->k_cache, 16) || !aligned(in->v_cache, 16) || !aligned(in->slot_map, 4) ||
        !aligned(in->slot_offset, 8) || !aligned(in->visible, 4))
        return QSA_ERR_INVALID_ARG;
    return QSA_OK;
}

qsa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? QSA_OK : QSA_ERR_CUDA; }

uint32_t *err_word(void *ws, const Layout &L)
{
    return reinterpret_cast<uint32_t *>(static_cast<unsigned char *>(ws) + L.off_err);
}

template <typename T>
T *ws_at(void *ws, size_t off)
{
    return reinterpret_cast<T *>(static_cast<unsigned char *>(ws) + off);
}

// pooled != nullptr: score from the pooled-key cache instead of the raw keys;
// shared: every query reads the history at key_offset[0] (one pooled tile for all).
qsa_status do_score(const qsa_dims *d, const qsa_inputs *in, float *scores, int64_t stride, void *ws,
                    const Layout &L, cudaStream_t s, const float *pooled = nullptr,
                    const int64_t *pool_offset = nullptr, bool shared = false)
{
    if (d->batch == 0) return QSA_OK;
    const int sms = num_sms_of_current_device();
    if (sms <= 0) return QSA_ERR_CUDA;
    ScoreArgs a{in->q_idx, in->idx_keys, in->key_offset, in->visible, scores, stride,
                d->batch, d->idx_heads, d->idx_dim, d->max_visible, err_word(ws, L),
                ws_at<uint32_t>(ws, L.off_qmax), L.qmax_stride, pooled, pool_offset,
                (pooled == nullptr && !shared) ? ws_at<ScoreBalance>(ws, L.off_bal) : nullptr, 0};
    return from_cuda(shared ? launch_score_shared(a, sms, s) : launch_score(a, sms, s));
}

// use_hint: the quad maxima in the workspace were written by the scorer for
// exactly these scores (only inside qsa_decode).
qsa_status do_select(const qsa_dims *d, const int32_t *visible, const float *scores, int64_t stride,
                     int32_t *ids, int32_t *n_ids, void *ws, const Layout &L, cudaStream_t s, bool use_hint,
                     bool pdl = false, bool balance = false, const qsa_inputs *prefetch_for = nullptr)
{
    if (d->batch == 0) return QSA_OK;
    SelectArgs a{visible, scores, stride, ids, n_ids, L.row_cap, d->budget_groups, d->max_visible,
                 d->batch, err_word(ws, L), use_hint ? ws_at<uint32_t>(ws, L.off_qmax) : nullptr,
                 L.qmax_stride, balance ? ws_at<ScoreBalance>(ws, L.off_bal) : nullptr,
                 prefetch_for ? prefetch_for->slot_map : nullptr, prefetch_for ? prefetch_for->slot_offset : nullptr};
    return from_cuda(launch_select(a, s, pdl));
}

qsa_status do_gather(const qsa_dims *d, const qsa_inputs *in, const int32_t *ids, const int32_t *n_ids,
                     float *k_scr, float *v_scr, void *ws, const Layout &L, cudaStream_t s)
{
    if (d->batch == 0) return QSA_OK;
    GatherArgs a{in->visible, ids, n_ids, in->slot_map, in->slot_offset, in->k_cache, in->v_cache,
                 in->num_slots, k_scr, v_scr, L.row_cap, d->kv_heads * d->head_dim, d->batch,
                 err_word(ws, L)};
    return from_cuda(launch_gather(a, s));
}

qsa_status do_attend(const qsa_dims *d, const float *q, const float *k_scr, const float *v_scr,
                     const int32_t *n_ids, float *out, void *ws, const Layout &L, cudaStream_t s)
{
    if (d->batch == 0) return QSA_OK;
    AttendArgs a{q, k_scr, v_scr, n_ids, out,
                 ws_at<float>(ws, L.off_part_m), ws_at<float>(ws, L.off_part_l),
                 ws_at<float>(ws, L.off_part_acc), ws_at<uint32_t>(ws, L.off_tickets),
                 L.row_cap, L.nparts, d->batch, d->q_heads, d->kv_heads, d->head_dim,
                 d->scale, err_word(ws, L)};
    return from_cuda(launch_attend(a, s));
}

qsa_status do_gather_attend(const qsa_dims *d, const qsa_inputs *in, const int32_t *ids, const int32_t *n_ids,
                            float *k_scr, float *v_scr, float *out, void *ws, const Layout &L, cudaStream_t s,
                            bool pdl = false, int32_t *ids_out = nullptr, int32_t *n_ids_out = nullptr,
                            float *m_out = nullptr, float *l_out = nullptr)
{
    if (d->batch == 0) return QSA_OK;
    AttendArgs a{in->q, nullptr, nullptr, n_ids, out,
                 ws_at<float>(ws, L.off_part_m), ws_at<float>(ws, L.off_part_l),
                 ws_at<float>(ws, L.off_part_acc), ws_at<uint32_t>(ws, L.off_tickets),
                 L.row_cap, L.nparts, d->batch, d->q_heads, d->kv_heads, d->head_dim,
                 d->scale, err_word(ws, L),
                 ids, in->visible, in->slot_map, in->slot_offset, in->k_cache, in->v_cache, in->num_slots,
                 k_scr, v_scr, /*defer_merge (the launcher's)*/ 0, ids_out, n_ids_out, m_out, l_out};
    return from_cuda(launch_attend(a, s, pdl));
}

qsa_status check_shapes(const qsa_dims *d, bool score, bool attend)
{
    if (score && !score_shape_supported(d->idx_heads, d->idx_dim)) return QSA_ERR_UNSUPPORTED_SHAPE;
    if (attend && !attend_shape_supported(d->head_dim, d->q_heads, d->kv_heads))
        return QSA_ERR_UNSUPPORTED_SHAPE;
    return QSA_OK;
}

}  // namespace
}  // namespace qsa

using namespace qsa;

extern "C" {

size_t qsa_workspace_size(const qsa_dims *dims)
{
    if (!dims_valid(dims)) return 0;
    return make_layout(dims).total;
}

int64_t qsa_score_stride(const qsa_dims *dims)
{
    if (!dims_valid(dims)) return 0;
    return make_layout(dims).score_stride;
}

int32_t qsa_row_capacity(const qsa_dims *dims)
{
    if (!dims_valid(dims)) return 0;
    return make_layout(dims).row_cap;
}

namespace {
// pooled_rows < 0: the full-raw form; else the incremental form with a cache
// of pooled_rows rows.
qsa_status fill_stats(const qsa_dims *dims, const int32_t *visible_host, int64_t pooled_rows, qsa_stats *out)
{
    if (!dims_valid(dims) || !out || (dims->batch > 0 && !visible_host)) return QSA_ERR_INVALID_ARG;
    qsa_stats st;
    std::memset(&st, 0, sizeof st);
    for (int32_t b = 0; b < dims->batch; ++b) {
        const int64_t T = visible_host[b];
        if (T < 0 || T > dims->max_visible) return QSA_ERR_INVALID_ARG;
        const int64_t G = T / kGroup;
        const int64_t k = G < dims->budget_groups ? G : dims->budget_groups;
        const int64_t W = kGroup * k + T % kGroup;
        st.candidate_groups += G;
        st.selected_groups += k;
        st.selected_tokens += W;
        if (pooled_rows < 0) st.raw_key_bytes += T * dims->idx_dim * 4;
        st.kv_bytes += W * int64_t(dims->kv_heads) * dims->head_dim * 4 * 2;
    }
    st.pooled_key_bytes = pooled_rows < 0 ? 0 : pooled_rows * dims->idx_dim * 4;
    st.workspace_bytes = int64_t(make_layout(dims).total);
    st.total_bytes = st.raw_key_bytes + st.kv_bytes + st.pooled_key_bytes + st.workspace_bytes;
    st.dense_mask_bytes = 0;  // no entry point allocates or writes a query-by-key mask
    *out = st;
    return QSA_OK;
}
}  // namespace

qsa_status qsa_get_stats(const qsa_dims *dims, const int32_t *visible_host, qsa_stats *out)
{
    return fill_stats(dims, visible_host, -1, out);
}

qsa_status qsa_get_stats_pooled(const qsa_dims *dims, const int32_t *visible_host, int64_t pooled_rows,
                                qsa_stats *out)
{
    if (pooled_rows < 0) return QSA_ERR_INVALID_ARG;
    return fill_stats(dims, visible_host, pooled_rows, out);
}

const char *qsa_status_string(qsa_status status)
{
    switch (status) {
    case QSA_OK: return "ok";
    case QSA_ERR_INVALID_ARG: return "invalid argument (NULL or misaligned pointer, or bad value)";
    case QSA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (no kernel built for these dimensions)";
    case QSA_ERR_WORKSPACE_TOO_SMALL: return "workspace smaller than qsa_workspace_size(dims)";
    case QSA_ERR_CUDA: return "a CUDA runtime call or kernel launch failed";
    case QSA_ERR_DEVICE_FAULT: return "the device error word was set (see QSA_DEVERR_* bits)";
    }
    return "unknown status";
}

qsa_status qsa_workspace_init(void *ws, size_t ws_bytes, void *stream)
{
    if (!ws || !aligned(ws, kWsAlign)) return QSA_ERR_INVALID_ARG;
    if (ws_bytes == 0) return QSA_OK;
    return from_cuda(cudaMemsetAsync(ws, 0, ws_bytes, static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_check_errors(void *ws, size_t ws_bytes, void *stream, uint32_t *flags_out)
{
    if (!ws || !aligned(ws, kWsAlign) || ws_bytes < kWsAlign) return QSA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint32_t flags = 0;
    if (cudaStreamSynchronize(s) != cudaSuccess) return QSA_ERR_CUDA;
    if (cudaMemcpy(&flags, ws, sizeof flags, cudaMemcpyDeviceToHost) != cudaSuccess) return QSA_ERR_CUDA;
    if (flags != 0 && cudaMemset(ws, 0, sizeof flags) != cudaSuccess) return QSA_ERR_CUDA;
    if (flags_out) *flags_out = flags;
    return flags ? QSA_ERR_DEVICE_FAULT : QSA_OK;
}

qsa_status qsa_score_groups(const qsa_dims *dims, const qsa_inputs *in, float *scores, void *ws,
                            size_t ws_bytes, void *stream)
{
    if (!dims_valid(dims)) return QSA_ERR_INVALID_ARG;
    qsa_status st;
    if ((st = check_shapes(dims, true, false)) != QSA_OK) return st;
    if ((st = check_inputs_score(in)) != QSA_OK) return st;
    if (!scores || !aligned(scores, 16)) return QSA_ERR_INVALID_ARG;
    if ((st = check_ws(dims, ws, ws_bytes)) != QSA_OK) return st;
    const Layout L = make_layout(dims);
    return do_score(dims, in, scores, L.score_stride, ws, L, static_cast<cudaStream_t>(stream));
}

qsa_status qsa_select(const qsa_dims *dims, const int32_t *visible, const float *scores, int32_t *ids,
                      int32_t *n_ids, void *ws, size_t ws_bytes, void *stream)
{
    if (!dims_valid(dims)) return QSA_ERR_INVALID_ARG;
    if (!visible || !scores || !ids || !n_ids) return QSA_ERR_INVALID_ARG;
    if (!aligned(visible, 4) || !aligned(scores, 16) || !aligned(ids, 4) || !aligned(n_ids, 4))
        return QSA_ERR_INVALID_ARG;
    qsa_status st;
    if ((st = check_ws(dims, ws, ws_bytes)) != QSA_OK) return st;
    const Layout L = make_layout(dims);
    return do_select(dims, visible, scores, L.score_stride, ids, n_ids, ws, L,
                     static_cast<cudaStream_t>(stream), false);
}

qsa_status qsa_gather(const qsa_dims *dims, const qsa_inputs *in, const int32_t *ids, const int32_t *n_ids,
                      float *k_scr, float *v_scr, void *ws, size_t ws_bytes, void *stream)
{
    if (!dims_valid(dims)) return QSA_ERR_INVALID_ARG;
    qsa_status st;
    if ((st = check_inputs_gather(in)) != QSA_OK) return st;
    if (!ids || !n_ids || !k_scr || !v_scr) return QSA_ERR_INVALID_ARG;
    if (!aligned(ids, 4) || !aligned(n_ids, 4) || !aligned(k_scr, 16) || !aligned(v_scr, 16))
        return QSA_ERR_INVALID_ARG;
    if ((dims->kv_heads * dims->head_dim) % 4 != 0) return QSA_ERR_UNSUPPORTED_SHAPE;
    if ((st = check_ws(dims, ws, ws_bytes)) != QSA_OK) return st;
    const Layout L = make_layout(dims);
    return do_gather(dims, in, ids, n_ids, k_scr, v_scr, ws, L, static_cast<cudaStream_t>(stream));
}

qsa_status qsa_attend(const qsa_dims *dims, const float *q, const float *k_scr, const float *v_scr,
                      const int32_t *n_ids, float *out, void *ws, size_t ws_bytes, void *stream)
{
    if (!dims_valid(dims)) return QSA_ERR_INVALID_ARG;
    qsa_status st;
    if ((st = check_shapes(dims, false, true)) != QSA_OK) return st;
    if (!q || !k_scr || !v_scr || !n_ids || !out) return QSA_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_scr, 16) || !aligned(v_scr, 16) || !aligned(n_ids, 4) ||
        !aligned(out, 16))
        return QSA_ERR_INVALID_ARG;
    if ((st = check_ws(dims, ws, ws_bytes)) != QSA_OK) return st;
    const Layout L = make_layout(dims);
    return do_attend(dims, q, k_scr, v_scr, n_ids, out, ws, L, static_cast<cudaStream_t>(stream));
}

qsa_status qsa_gather_attend(const qsa_dims *dims, const qsa_inputs *in, const int32_t *ids, const int32_t *n_ids,
                             float *k_scr, float *v_scr, float *out, void *ws, size_t ws_bytes, void *stream)
{
    if (!dims_valid(dims)) return QSA_ERR_INVALID_ARG;
    qsa_status st;
    if ((st = check_shapes(dims, false, true)) != QSA_OK) return st;
    if ((st = check_inputs_gather(in)) != QSA_OK) return st;
    if (!in->q || !aligned(in->q, 16)) return QSA_ERR_INVALID_ARG;
    if (!ids || !n_ids || !k_scr || !v_scr || !out) return QSA_ERR_INVALID_ARG;
    if (!aligned(ids, 4) || !aligned(n_ids, 4) || !aligned(k_scr, 16) || !aligned(v_scr, 16) || !aligned(out, 16))
        return QSA_ERR_INVALID_ARG;
    if ((st = check_ws(dims, ws, ws_bytes)) != QSA_OK) return st;
    const Layout L = make_layout(dims);
    return do_gather_attend(dims, in, ids, n_ids, k_scr, v_scr, out, ws, L, static_cast<cudaStream_t>(stream));
}

qsa_status qsa_selftest_copy_timeout(const qsa_dims *dims, const qsa_inputs *in, float *scores, void *ws,
                                     size_t ws_bytes, uint64_t wait_ns, void *stream)
{
    if (!dims_valid(dims) || wait_ns == 0 || wait_ns > kWaitLimitNs) return QSA_ERR_INVALID_ARG;
    qsa_status st;
    if ((st = check_shapes(dims, true, false)) != QSA_OK) return st;
    if ((st = check_inputs_score(in)) != QSA_OK) return st;
    if (!scores || !aligned(scores, 16)) return QSA_ERR_INVALID_ARG;
    if ((st = check_ws(dims, ws, ws_bytes)) != QSA_OK) return st;
    if (dims->batch == 0) return QSA_OK;
    const Layout L = make_layout(dims);
    const int sms = num_sms_of_current_device();
    if (sms <= 0) return QSA_ERR_CUDA;
    // equal shares (no per-SM weights), no copy issued, short waits
    ScoreArgs a{in->q_idx, in->idx_keys, in->key_offset, in->visible, scores, L.score_stride,
                dims->batch, dims->idx_heads, dims->idx_dim, dims->max_visible, err_word(ws, L),
                ws_at<uint32_t>(ws, L.off_qmax), L.qmax_stride, nullptr, nullptr, nullptr, 0, 1, wait_ns};
    return from_cuda(launch_score(a, sms, static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_attend_state(const qsa_dims *dims, const qsa_inputs *in, const int32_t *ids, const int32_t *n_ids,
                            float *acc, float *m, float *l, void *ws, size_t ws_bytes, void *stream)
{
    if (!dims_valid(dims)) return QSA_ERR_INVALID_ARG;
    qsa_status st;
    if ((st = check_shapes(dims, false, true)) != QSA_OK) return st;
    if ((st = check_inputs_gather(in)) != QSA_OK) return st;
    if (!in->q || !aligned(in->q, 16)) return QSA_ERR_INVALID_ARG;
    if (!ids || !n_ids || !acc || !m || !l) return QSA_ERR_INVALID_ARG;
    if (!aligned(ids, 4) || !aligned(n_ids, 4) || !aligned(acc, 16) || !aligned(m, 4) || !aligned(l, 4))
        return QSA_ERR_INVALID_ARG;
    if ((st = check_ws(dims, ws, ws_bytes)) != QSA_OK) return st;
    const Layout L = make_layout(dims);
    return do_gather_attend(dims, in, ids, n_ids, nullptr, nullptr, acc, ws, L, static_cast<cudaStream_t>(stream),
                            false, nullptr, nullptr, m, l);
}

qsa_status qsa_merge_states(const qsa_dims *dims, int32_t n_parts, const float *m, const float *l, const float *acc,
                            float *out, void *stream)
{
    if (!dims_valid(dims)) return QSA_ERR_INVALID_ARG;
    qsa_status st;
    if ((st = check_shapes(dims, false, true)) != QSA_OK) return st;
    if (n_parts < 1 || !m || !l || !acc || !out) return QSA_ERR_INVALID_ARG;
    if (!aligned(m, 4) || !aligned(l, 4) || !aligned(acc, 16) || !aligned(out, 16)) return QSA_ERR_INVALID_ARG;
    const long long bh = (long long)dims->batch * dims->q_heads;
    if (bh > 0x7fffffffLL / (long long)n_parts) return QSA_ERR_INVALID_ARG;
    return from_cuda(launch_merge_states(m, l, acc, out, n_parts, int(bh), dims->head_dim,
                                         static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace {
// The whole path; pooled != nullptr scores from the pooled-key cache.
qsa_status decode_impl(const qsa_dims *dims, const qsa_inputs *in, const float *pooled,
                       const int64_t *pool_offset, int32_t *ids, int32_t *n_ids, float *out, void *ws,
                       size_t ws_bytes, void *stream, void *const *events, int32_t n_events,
                       bool shared = false)
{
    if (!dims_valid(dims)) return QSA_ERR_INVALID_ARG;
    qsa_status st;
    if ((st = check_shapes(dims, true, true)) != QSA_OK) return st;
    if ((st = pooled ? check_inputs_pooled(in, pooled, pool_offset) : check_inputs_score(in)) != QSA_OK) return st;
    if ((st = check_inputs_gather(in)) != QSA_OK) return st;
    if (!in->q || !aligned(in->q, 16)) return QSA_ERR_INVALID_ARG;
    if (!ids || !n_ids || !out || !aligned(ids, 4) || !aligned(n_ids, 4) || !aligned(out, 16))
        return QSA_ERR_INVALID_ARG;
    if ((st = check_ws(dims, ws, ws_bytes)) != QSA_OK) return st;
    if (n_events != 0 && (n_events != 4 || !events)) return QSA_ERR_INVALID_ARG;
    for (int32_t i = 0; i < n_events; ++i)
        if (!events[i]) return QSA_ERR_INVALID_ARG;
    const Layout L = make_layout(dims);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float *scores = ws_at<float>(ws, L.off_scores);
    auto mark = [&](int i) -> bool {
        return n_events == 0 || cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) == cudaSuccess;
    };
    if (!mark(0)) return QSA_ERR_CUDA;
    if ((st = do_score(dims, in, scores, L.score_stride, ws, L, s, pooled, pool_offset, shared)) != QSA_OK)
        return st;
    if (!mark(1)) return QSA_ERR_CUDA;
    // The three launches overlap their launch latency with the predecessor's
    // tail (programmatic dependent launch) unless timing marks separate them.
    const bool pdl = n_events == 0;
    // (after the raw scorer: one spare selection CTA updates its per-SM weights)
    // The rows go to the workspace; the attention kernel, which finishes the
    // path, stores them with `out` to the caller's buffers (device or mapped
    // host memory alike: no separate copy of the results).
    int32_t *ids_ws = ws_at<int32_t>(ws, L.off_ids);
    int32_t *n_ws = ws_at<int32_t>(ws, L.off_nids);
    // (the chosen groups' slot-map entries are prefetched into L2 for the attention)
    if ((st = do_select(dims, in->visible, scores, L.score_stride, ids_ws, n_ws, ws, L, s, true, pdl,
                        pooled == nullptr && !shared, in)) != QSA_OK)
        return st;
    if (!mark(2)) return QSA_ERR_CUDA;
    // K/V rows go from the cache to shared memory and nowhere else: no scratch
    if ((st = do_gather_attend(dims, in, ids_ws, n_ws, nullptr, nullptr, out, ws, L, s, pdl, ids, n_ids)) != QSA_OK)
        return st;
    if (!mark(3)) return QSA_ERR_CUDA;
    return QSA_OK;
}

}  // namespace

extern "C" {

qsa_status qsa_decode_profiled(const qsa_dims *dims, const qsa_inputs *in, int32_t *ids, int32_t *n_ids,
                               float *out, void *ws, size_t ws_bytes, void *stream, void *const *events,
                               int32_t n_events)
{
    return decode_impl(dims, in, nullptr, nullptr, ids, n_ids, out, ws, ws_bytes, stream, events, n_events);
}

qsa_status qsa_decode_pooled(const qsa_dims *dims, const qsa_inputs *in, const float *pooled,
                             const int64_t *pool_offset, int32_t *ids, int32_t *n_ids, float *out, void *ws,
                             size_t ws_bytes, void *stream)
{
    if (!pooled || !pool_offset) return QSA_ERR_INVALID_ARG;
    return decode_impl(dims, in, pooled, pool_offset, ids, n_ids, out, ws, ws_bytes, stream, nullptr, 0);
}

qsa_status qsa_decode_shared(const qsa_dims *dims, const qsa_inputs *in, int32_t *ids, int32_t *n_ids,
                             float *out, void *ws, size_t ws_bytes, void *stream)
{
    return decode_impl(dims, in, nullptr, nullptr, ids, n_ids, out, ws, ws_bytes, stream, nullptr, 0, true);
}

qsa_status qsa_score_groups_shared(const qsa_dims *dims, const qsa_inputs *in, float *scores, void *ws,
                                   size_t ws_bytes, void *stream)
{
    if (!dims_valid(dims)) return QSA_ERR_INVALID_ARG;
    qsa_status st;
    if ((st = check_shapes(dims, true, false)) != QSA_OK) return st;
    if ((st = check_inputs_score(in)) != QSA_OK) return st;
    if (!scores || !aligned(scores, 16)) return QSA_ERR_INVALID_ARG;
    if ((st = check_ws(dims, ws, ws_bytes)) != QSA_OK) return st;
    const Layout L = make_layout(dims);
    return do_score(dims, in, scores, L.score_stride, ws, L, static_cast<cudaStream_t>(stream), nullptr, nullptr,
                    true);
}

qsa_status qsa_score_pooled(const qsa_dims *dims, const qsa_inputs *in, const float *pooled,
                            const int64_t *pool_offset, float *scores, void *ws, size_t ws_bytes, void *stream)
{
    if (!dims_valid(dims)) return QSA_ERR_INVALID_ARG;
    qsa_status st;
    if ((st = check_shapes(dims, true, false)) != QSA_OK) return st;
    if ((st = check_inputs_pooled(in, pooled, pool_offset)) != QSA_OK) return st;
    if (!scores || !aligned(scores, 16)) return QSA_ERR_INVALID_ARG;
    if ((st = check_ws(dims, ws, ws_bytes)) != QSA_OK) return st;
    const Layout L = make_layout(dims);
    return do_score(dims, in, scores, L.score_stride, ws, L, static_cast<cudaStream_t>(stream), pooled, pool_offset);
}

qsa_status qsa_pool_groups(const qsa_dims *dims, const qsa_inputs *in, const int32_t *group_begin,
                           const int32_t *group_end, int32_t max_groups, float *pooled, const int64_t *pool_offset,
                           void *ws, size_t ws_bytes, void *stream)
{
    if (!dims_valid(dims)) return QSA_ERR_INVALID_ARG;
    if (!score_shape_supported(dims->idx_heads, dims->idx_dim)) return QSA_ERR_UNSUPPORTED_SHAPE;
    if (!in || !in->idx_keys || !in->key_offset || !aligned(in->idx_keys, 16) || !aligned(in->key_offset, 8))
        return QSA_ERR_INVALID_ARG;
    if (!group_begin || !group_end || !pooled || !pool_offset || !aligned(group_begin, 4) ||
        !aligned(group_end, 4) || !aligned(pooled, 16) || !aligned(pool_offset, 8))
        return QSA_ERR_INVALID_ARG;
    const int32_t g_max = dims->max_visible / kGroup;
    if (max_groups < 0 || max_groups > g_max) return QSA_ERR_INVALID_ARG;
    qsa_status st;
    if ((st = check_ws(dims, ws, ws_bytes)) != QSA_OK) return st;
    const Layout L = make_layout(dims);
    PoolArgs a{in->idx_keys, in->key_offset, group_begin, group_end, pooled, pool_offset,
               dims->batch, dims->idx_dim, max_groups, g_max, err_word(ws, L)};
    return from_cuda(launch_pool(a, static_cast<cudaStream_t>(stream)));
}

qsa_status qsa_decode(const qsa_dims *dims, const qsa_inputs *in, int32_t *ids, int32_t *n_ids, float *out,
                      void *ws, size_t ws_bytes, void *stream)
{
    return qsa_decode_profiled(dims, in, ids, n_ids, out, ws, ws_bytes, stream, nullptr, 0);
}

}  // extern "C"
