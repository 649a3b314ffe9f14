/*
 * qsa.h -- C ABI of libqsa, physically sparse QSA decode on GB300 (sm_103a).
 *
 * The method is the one defined by two notes of the Hebrus project:
 *   [AFN-017] "Top-k chooses the set; time chooses the order"
 *   [AFN-016] "A sparse mask is not sparse attention"
 * Per decode query with T visible tokens, the path
 *   scores every complete four-token group g (tokens 4g..4g+3) as
 *     sum over indexer heads h of ReLU(q_h . mean(k_4g..k_4g+3)),
 *   chooses the top min(G, budget) groups by (score desc, position asc),
 *   emits them in ascending position, each expanded to 4 token IDs, and
 *     appends the raw tail of T mod 4 tokens (at most 2,051 IDs),
 *   resolves the IDs through a slot map, gathers only those K/V rows into
 *     bounded scratch, and
 *   runs an online softmax over that compact row in emitted order.
 * No query-by-key mask is ever built ([AFN-016] What the checkpoint measures).
 *
 * Conventions shared by every call
 * --------------------------------
 * - All pointers except `dims`, `stats` and host-side arguments named
 *   `*_host` are DEVICE pointers of the current CUDA device.  The library
 *   never allocates or frees memory: the caller owns every buffer,
 *   including the workspace ([AFN-016] What the checkpoint measures: byte
 *   ownership is visible).
 * - Float arrays are IEEE binary32, row-major, and must start on a 16-byte
 *   boundary; the workspace on a 256-byte boundary.
 * - `stream` is a cudaStream_t (NULL = the legacy default stream).  Every
 *   compute call is asynchronous on `stream` and returns after enqueueing.
 * - Host-detectable errors (NULL or misaligned pointers, bad dimensions,
 *   unsupported shapes, a workspace that is too small) return a status
 *   before anything is enqueued.  A failed launch returns QSA_ERR_CUDA.
 *   An empty batch (B = 0) with valid arguments enqueues nothing and
 *   returns QSA_OK.
 * - Errors that only the device can see (a T_b outside [0, max_visible],
 *   a slot outside [0, num_slots), an ID row longer than its capacity, a
 *   bounded wait that ran out) never trap: the kernel skips the bad access,
 *   writes zeros / an empty row for that query, and sets a bit in a sticky
 *   error word in the workspace, which qsa_check_errors() reads and clears.
 * - Results are deterministic: the same inputs give bit-identical outputs,
 *   whatever the batch composition or the number of SMs.
 * - Calls that share one workspace must not overlap on the GPU.
 */
#ifndef QSA_H
#define QSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    QSA_OK = 0,
    QSA_ERR_INVALID_ARG = 1,          /* NULL/misaligned pointer, bad value     */
    QSA_ERR_UNSUPPORTED_SHAPE = 2,    /* no kernel built for these dimensions  */
    QSA_ERR_WORKSPACE_TOO_SMALL = 3,  /* ws_bytes < qsa_workspace_size(dims)   */
    QSA_ERR_CUDA = 4,                 /* a CUDA runtime call or launch failed  */
    QSA_ERR_DEVICE_FAULT = 5          /* the device error word was non-zero    */
} qsa_status;

/* Bits of the device error word (see qsa_check_errors). */
#define QSA_DEVERR_VISIBLE_RANGE 0x1u  /* some T_b < 0 or T_b > max_visible   */
#define QSA_DEVERR_SLOT_RANGE    0x2u  /* a slot-map entry outside the cache  */
#define QSA_DEVERR_ROW_RANGE     0x4u  /* n_ids[b] or an ID outside its row   */
#define QSA_DEVERR_WAIT_TIMEOUT  0x8u  /* a bounded copy wait ran out         */
#define QSA_DEVERR_NOT_SHARED    0x10u /* a shared-history call whose queries  */
                                       /* do not all have key_offset[0]       */

/* Problem dimensions.  Supported builds: (idx_heads, idx_dim) in
 * {(4,32), (8,32), (4,64), (8,64)}; head_dim in {64, 128};
 * q_heads = kv_heads * r with r in 1..16; group == 4; 1 <= budget_groups
 * <= 512; 0 <= max_visible <= QSA_MAX_VISIBLE; 0 <= batch <= 65535 (the
 * attention's grids carry the query in a dimension of at most 65,535). */
typedef struct {
    int32_t batch;          /* B: decode queries in this call (0..65535)          */
    int32_t idx_heads;      /* H_I: indexer query heads                          */
    int32_t idx_dim;        /* d_I: width of one raw index key                   */
    int32_t q_heads;        /* n_q: attention query heads                        */
    int32_t kv_heads;       /* n_kv: K/V heads; q head h reads KV head h/(n_q/n_kv) */
    int32_t head_dim;       /* d: attention head width                           */
    int32_t group;          /* tokens per scored group; must be 4 ([AFN-017] Decision) */
    int32_t budget_groups;  /* groups kept per query; 512 in the notes           */
    int32_t max_visible;    /* upper bound on every T_b; sizes scores and grids  */
    float scale;            /* softmax scale, usually 1/sqrt(head_dim)           */
} qsa_dims;

#define QSA_MAX_VISIBLE (1 << 26)
#define QSA_MAX_BUDGET 512

/* Inputs of one decode batch (device pointers). */
typedef struct {
    const float *q_idx;          /* [B, H_I, d_I] indexer queries                        */
    const float *idx_keys;       /* [total_tokens, d_I] raw index keys, LOGICAL order:   */
                                 /*   query b's token t is row key_offset[b] + t         */
    const int64_t *key_offset;   /* [B] first row of query b's history in idx_keys       */
    const int32_t *visible;      /* [B] T_b, visible tokens of query b                   */
    const float *q;              /* [B, n_q, d] attention queries                        */
    const float *k_cache;        /* [num_slots, n_kv, d] K rows by PHYSICAL slot         */
    const float *v_cache;        /* [num_slots, n_kv, d] V rows by PHYSICAL slot         */
    int64_t num_slots;           /* physical slots in k_cache / v_cache                  */
    const int32_t *slot_map;     /* logical -> physical: query b's token t lives in slot */
                                 /*   slot_map[slot_offset[b] + t]                        */
    const int64_t *slot_offset;  /* [B] first slot-map entry of query b's history        */
} qsa_inputs;

/* Work and byte ownership of one batch ([AFN-016] What the checkpoint
 * measures: candidate groups scored, selected groups and expanded width,
 * raw-key / K/V / pooled-key / workspace / total bytes, zero dense mask). */
typedef struct {
    int64_t candidate_groups;   /* sum_b floor(T_b/4)                            */
    int64_t selected_groups;    /* sum_b min(floor(T_b/4), budget)               */
    int64_t selected_tokens;    /* sum_b (4*selected groups + T_b mod 4)         */
    int64_t raw_key_bytes;      /* raw index-key bytes the scorer streams:       */
                                /*   sum_b T_b*d_I*4 (full-raw form), 0 for the  */
                                /*   incremental form, which reads pooled keys   */
    int64_t kv_bytes;           /* K and V bytes the gather reads                */
    int64_t pooled_key_bytes;   /* pooled keys held in device memory: 0 in the   */
                                /*   full-raw form (its pooled tiles live in     */
                                /*   shared memory only); the caller's pooled-   */
                                /*   key cache in the incremental form           */
    int64_t workspace_bytes;    /* qsa_workspace_size(dims)                      */
    int64_t total_bytes;        /* raw_key + kv + pooled_key + workspace         */
    int64_t dense_mask_bytes;   /* bytes of any query-by-key mask: 0 by          */
                                /*   construction -- no entry point allocates or */
                                /*   writes one, and the workspace formula below */
                                /*   has no queries x keys term                  */
} qsa_stats;

/* ---- sizes (host only, no CUDA call) ---------------------------------- */

/* Bytes of workspace every call below needs for these dims (0 if the dims
 * are invalid).  Sized as groups + budget + selected width per query,
 * never queries x keys ([AFN-016] What the checkpoint measures):
 *   header (256 + align256(B*n_kv*4) attention tickets + 7,424 for the
 *   scorer's per-SM balance: weights learned from its own timings) +
 *   B*score_stride*4 (scores) + B*qstride*4 (the largest score of
 *   every four groups, a selection aid; qstride = ceil(G_max/4) rounded up
 *   to 32, G_max = max_visible/4) +
 *   B*n_q*17*(d+2)*4 (attention partials: 17 runs of 128 rows per head) +
 *   B*(4*budget+3)*4 + B*4 (qsa_decode's ID rows and counts, which its last
 *   kernel then stores to the caller's ids / n_ids).
 * The compact K/V row of qsa_decode never reaches device memory, so the
 * workspace holds no K/V scratch. */
size_t qsa_workspace_size(const qsa_dims *dims);

/* Row stride, in floats, of a scores buffer: max_visible/4 rounded up to 32. */
int64_t qsa_score_stride(const qsa_dims *dims);

/* Capacity of one emitted ID row: 4*budget_groups + 3 (2,051 at budget 512,
 * [AFN-016] Decision). */
int32_t qsa_row_capacity(const qsa_dims *dims);

/* Fills *out for the full-raw form (qsa_decode) from the dims and the host
 * copy of visible ([B] T_b). */
qsa_status qsa_get_stats(const qsa_dims *dims, const int32_t *visible_host, qsa_stats *out);

/* Fills *out for the incremental form (qsa_decode_pooled): the scorer streams
 * sum_b floor(T_b/4)*d_I*4 bytes of pooled keys instead of raw keys
 * (raw_key_bytes = 0), and pooled_key_bytes counts the caller's pooled-key
 * cache of pooled_rows rows of d_I floats (queries that share a history
 * share its rows, so pooled_rows is the sum of floor(T/4) over the distinct
 * histories when the cache holds exactly their complete groups). */
qsa_status qsa_get_stats_pooled(const qsa_dims *dims, const int32_t *visible_host, int64_t pooled_rows,
                                qsa_stats *out);

const char *qsa_status_string(qsa_status status);

/* ---- workspace ---------------------------------------------------------- */

/* Zeroes the ws_bytes of the workspace, whose header holds the error word,
 * the attention tickets and the scorer's per-SM weights.  Call once after
 * allocating a workspace, before its first use; a zero-filled allocation
 * needs no call.  Afterwards every call leaves the tickets clean, and the
 * weights are learned from the scorer's own timings. */
qsa_status qsa_workspace_init(void *ws, size_t ws_bytes, void *stream);

/* Synchronises `stream`, then reads and clears the sticky device error word
 * of `ws`.  *flags_out (may be NULL) receives the QSA_DEVERR_* bits.
 * Returns QSA_ERR_DEVICE_FAULT if any bit was set, else QSA_OK. */
qsa_status qsa_check_errors(void *ws, size_t ws_bytes, void *stream, uint32_t *flags_out);

/* ---- the hot path, one stage per call ----------------------------------- */

/* Stage 1 -- group scoring ([AFN-016] Decision: score complete groups in
 * bounded tiles; Why a sparse mask can still be dense: pooled groups and
 * sum(ReLU(dot_h))).  For each query b and each complete group
 * g < floor(T_b/4):
 *   p[j] = (((k[4g][j] + k[4g+1][j]) + k[4g+2][j]) + k[4g+3][j]) * 0.25
 *   scores[b*score_stride + g] = sum_{h=0..H_I-1, in order} ReLU(dot_h),
 *   dot_h = fma chain over j = 0..d_I-1 starting from +0, ReLU(x) = x>0 ? x : +0,
 * every step binary32 round-to-nearest in exactly that order, so scores are
 * bit-identical to any implementation of that order.
 * scores: [B, qsa_score_stride(dims)]; entries g >= floor(T_b/4) untouched.
 * When the tiles fill every SM, the launch is cooperative and each SM's
 * share of the tiles follows its streaming speed as measured in earlier
 * launches on this workspace (the weights qsa_decode keeps up to date); the
 * shares move work between SMs and never change a score. */
qsa_status qsa_score_groups(const qsa_dims *dims, const qsa_inputs *in, float *scores,
                            void *ws, size_t ws_bytes, void *stream);

/* Stage 2 -- set choice and chronological emission ([AFN-017] Decision;
 * Tie handling belongs to membership).  Chooses the top
 * k = min(floor(T_b/4), budget) groups of scores[b] by (score descending,
 * group position ascending) -- ties resolved while choosing membership --
 * then writes their IDs in ascending logical position, each group expanded
 * to 4 consecutive token IDs, followed by the raw tail 4*floor(T_b/4)..T_b-1:
 *   ids:   [B, qsa_row_capacity(dims)] int32, entries >= n_ids[b] untouched
 *   n_ids: [B] int32, = 4k + T_b mod 4
 * Scores must not be NaN (-0 counts as +0).  Below budget the row is exactly
 * 0..T_b-1, the dense causal row ([AFN-017] The dense-parity property). */
qsa_status qsa_select(const qsa_dims *dims, const int32_t *visible, const float *scores,
                      int32_t *ids, int32_t *n_ids, void *ws, size_t ws_bytes, void *stream);

/* Stage 3 -- slot resolution and compact gather ([AFN-016] Decision: only
 * the gather crosses from logical identity into the physical layout; Why
 * compact gather comes before fusion).  For i < n_ids[b]:
 *   s = slot_map[slot_offset[b] + ids[b][i]]
 *   k_scr[b][i][:][:] = k_cache[s][:][:],  v_scr[b][i][:][:] = v_cache[s][:][:]
 * k_scr, v_scr: [B, qsa_row_capacity(dims), n_kv, d]; rows >= n_ids[b]
 * untouched.  A slot outside [0, num_slots) zero-fills that row and sets
 * QSA_DEVERR_SLOT_RANGE. */
qsa_status qsa_gather(const qsa_dims *dims, const qsa_inputs *in, const int32_t *ids,
                      const int32_t *n_ids, float *k_scr, float *v_scr,
                      void *ws, size_t ws_bytes, void *stream);

/* Stage 4 -- online softmax over the compact row ([AFN-017] Floating point
 * makes order observable; [AFN-016] Decision).  For each query b and head h
 * (KV head h / (n_q/n_kv)):
 *   out[b][h] = sum_i softmax_i(scale * q[b][h] . k_scr[b][i]) v_scr[b][i],
 * rows i < n_ids[b] visited in emitted order: the row is cut into runs of
 * 128 rows (17 at most), each run into steps of 4 consecutive rows dealt
 * to 8 running states in turn; each state is a running
 * max / rescale / denominator / accumulator, and the states are merged in a
 * fixed order, then the runs in row order.  The split depends only on
 * n_ids[b], so results do not depend on the batch.  n_ids[b] = 0 gives a
 * zero output.  out: [B, n_q, d]. */
qsa_status qsa_attend(const qsa_dims *dims, const float *q, const float *k_scr,
                      const float *v_scr, const int32_t *n_ids, float *out,
                      void *ws, size_t ws_bytes, void *stream);

/* Stages 3 and 4 in one launch: each attention CTA resolves its rows'
 * slots, copies exactly those K/V rows from the cache into shared memory,
 * writes them from there to k_scr / v_scr (the same bytes as qsa_gather) and
 * runs the attention of qsa_attend on them.  Outputs: k_scr, v_scr (as
 * qsa_gather) and out (as qsa_attend), bit-identical to qsa_gather followed
 * by qsa_attend. */
qsa_status qsa_gather_attend(const qsa_dims *dims, const qsa_inputs *in, const int32_t *ids,
                             const int32_t *n_ids, float *k_scr, float *v_scr, float *out,
                             void *ws, size_t ws_bytes, void *stream);

/* The attention of qsa_gather_attend (rows resolved through the slot map and
 * copied from the cache, visited in the order of qsa_attend) with its
 * online-softmax state as the result instead of the normalised output, so
 * that consecutive slices of one emitted row, attended separately (e.g. on
 * the ranks that hold those tokens), combine into the row's attention
 * ([AFN-017] Floating point makes order observable: the slices are merged in
 * row order, a fixed order).  For each query b and head h, over the rows
 * ids[b*row_cap + i], i < n_ids[b] (row_cap = qsa_row_capacity(dims); token
 * IDs below visible[b], resolved as slot_map[slot_offset[b] + id]), with
 * s_i = scale * q[b][h] . k_i:
 *   m[b*n_q + h]    = max_i s_i                           (-inf for no rows)
 *   l[b*n_q + h]    = sum_i e^(s_i - m)                   (0 for no rows)
 *   acc[b][h][0..d) = sum_i e^(s_i - m) v_i               (0 for no rows)
 * each sum taken in qsa_attend's order, so acc / l is qsa_attend's output
 * bit for bit.  Slices r = 0, 1, ... of one row combine, in that order, as
 * M = max m_r, L = sum_r l_r e^(m_r - M), out = (sum_r acc_r e^(m_r - M)) / L.
 * acc: [B, n_q, d] (16-byte aligned); m, l: [B, n_q]; all device memory,
 * caller-owned.  A row whose ID is outside [0, visible[b]) or whose slot is
 * outside [0, num_slots) is taken as a zero K/V row and flagged
 * (QSA_DEVERR_ROW_RANGE / QSA_DEVERR_SLOT_RANGE), as in qsa_decode; a count
 * outside [0, row_cap] gives the empty state and QSA_DEVERR_ROW_RANGE. */
qsa_status qsa_attend_state(const qsa_dims *dims, const qsa_inputs *in, const int32_t *ids,
                            const int32_t *n_ids, float *acc, float *m, float *l,
                            void *ws, size_t ws_bytes, void *stream);

/* Joins the attention states of consecutive slices of one emitted row -- as
 * qsa_attend_state returns them, e.g. one slice per rank holding those
 * tokens -- into the row's output ([AFN-017] Floating point makes order
 * observable: the slices merge in row order, a fixed order).  For each query
 * b and head h, with slices r = 0 .. n_parts-1 in that order:
 *   M = max_r m_r,  w_r = e^(m_r - M)  (0 when M = -inf),  L = sum_r l_r w_r,
 *   out[b][h] = (sum_r acc_r w_r) / L   (0 when L = 0),
 * both sums taken in slice order with the arithmetic the attention kernels
 * use to merge their own runs, so one slice holding a whole row gives
 * qsa_decode's output bit for bit.  m, l: [n_parts, B, n_q] (4-byte
 * aligned); acc: [n_parts, B, n_q, d] and out: [B, n_q, d] (16-byte
 * aligned); all device memory, caller-owned; n_parts >= 1.  Reads dims->
 * batch, q_heads, kv_heads and head_dim; needs no workspace. */
qsa_status qsa_merge_states(const qsa_dims *dims, int32_t n_parts, const float *m, const float *l,
                            const float *acc, float *out, void *stream);

/* The whole path on `stream`: qsa_score_groups, qsa_select, then the
 * gather fused into the attention ([AFN-016] Why compact gather comes before
 * fusion: fusion once the compact path is measured, keeping logical IDs and
 * zero dense-mask bytes) -- each attention CTA copies its selected K/V rows
 * from the cache straight into shared memory, so the compact row is never
 * written to device memory.  Outputs: ids, n_ids (as qsa_select) and out,
 * bit-identical to qsa_attend over qsa_gather's scratch.  The selection
 * launch has one spare CTA that turns the scorer's recorded times into its
 * per-SM shares for the next call on this workspace.  The selection writes
 * its rows to the workspace and the attention kernel, the last one of the
 * call, stores them to ids / n_ids together with out: the three outputs may
 * point to mapped (pinned) host memory, and then the results reach the host
 * with no separate copy. */
qsa_status qsa_decode(const qsa_dims *dims, const qsa_inputs *in, int32_t *ids,
                      int32_t *n_ids, float *out, void *ws, size_t ws_bytes, void *stream);

/* qsa_decode with timing marks: `events` holds n_events = 4 cudaEvent_t
 * handles (created by the caller) recorded on `stream` before the scoring
 * launch, before the selection launch, before the gather + attention launch
 * and after it; n_events = 0 is plain qsa_decode.  The launches and results
 * are those of qsa_decode. */
qsa_status qsa_decode_profiled(const qsa_dims *dims, const qsa_inputs *in, int32_t *ids,
                               int32_t *n_ids, float *out, void *ws, size_t ws_bytes, void *stream,
                               void *const *events, int32_t n_events);

/* ---- the incremental form: a pooled-key cache --------------------------- */

/* The notes pair the full-raw indexer with an incremental one ([AFN-017]
 * capsule and Evidence: the full-raw / incremental identity): instead of
 * pooling every group's raw keys at every decode step, keep the pooled key
 * of each complete group in device memory and append groups as they
 * complete.  The pooling arithmetic is the same binary32 sequence as in
 * qsa_score_groups, so scores from the cache equal full-raw scores bit for
 * bit, and so do the ID rows and outputs of qsa_decode_pooled.
 *
 * Cache layout (caller-owned, device): pooled[row][d_I] f32; group g of query
 * b lives at row pool_offset[b] + g, with its 16-byte chunks permuted within
 * the row: elements 4c..4c+3 of the pooled key sit at 4(c ^ (g & 7))..+3
 * (g the query's own group index; d_I is a multiple of 32), so that whole
 * rows copied into shared memory are read without bank conflicts.  Queries
 * that share a history may share rows (chunked prefill). */

/* Appends pooled keys: for each query b and g in [group_begin[b],
 * group_end[b]) (device int32 arrays),
 *   pooled key element j = (((k0[j]+k1[j])+k2[j])+k3[j]) * 0.25,
 *   k_u = idx_keys[key_offset[b] + 4g + u]          (reads in->idx_keys,
 * in->key_offset only), stored at row pool_offset[b] + g in the layout above.
 * max_groups (host) bounds group_end[b] -
 * group_begin[b] for every b and sizes the launch: a decode step that
 * completes one group per query passes 1.  The caller guarantees the raw rows
 * exist.  A range outside [0, max_visible/4] or longer than max_groups is
 * skipped and sets QSA_DEVERR_VISIBLE_RANGE. */
qsa_status qsa_pool_groups(const qsa_dims *dims, const qsa_inputs *in, const int32_t *group_begin,
                           const int32_t *group_end, int32_t max_groups, float *pooled,
                           const int64_t *pool_offset, void *ws, size_t ws_bytes, void *stream);

/* qsa_score_groups with the pooled keys read from the cache (rows
 * pool_offset[b] + g, g < floor(T_b/4)) instead of pooled from the raw keys:
 * G*d_I*4 bytes streamed per query instead of T*d_I*4.  Reads in->q_idx and
 * in->visible; in->idx_keys and in->key_offset may be NULL.  Its kernel is
 * launched with programmatic dependent launch: it may start while the kernel
 * before it on `stream` (e.g. qsa_pool_groups) finishes, and waits for that
 * kernel to complete before it reads anything, so stream order holds. */
qsa_status qsa_score_pooled(const qsa_dims *dims, const qsa_inputs *in, const float *pooled,
                            const int64_t *pool_offset, float *scores, void *ws, size_t ws_bytes,
                            void *stream);

/* qsa_decode with the scorer reading the pooled-key cache: same launches
 * otherwise, same outputs bit for bit when the cache holds every complete
 * group of each query's history.  in->idx_keys and in->key_offset may be
 * NULL. */
qsa_status qsa_decode_pooled(const qsa_dims *dims, const qsa_inputs *in, const float *pooled,
                             const int64_t *pool_offset, int32_t *ids, int32_t *n_ids, float *out,
                             void *ws, size_t ws_bytes, void *stream);

/* ---- queries over one shared history (chunked prefill) ------------------ */

/* qsa_score_groups for a batch whose queries all read one key history
 * (key_offset[b] == key_offset[0] for every b; T_b may differ), e.g. the
 * consecutive positions of a chunked prefill ([AFN-017] capsule: chunk =
 * decode).  Each tile of raw keys is pooled once and scored for every query
 * that needs it, instead of once per query; the scores are bit-identical to
 * qsa_score_groups.  A query whose key_offset differs gets no scores and
 * sets QSA_DEVERR_NOT_SHARED. */
qsa_status qsa_score_groups_shared(const qsa_dims *dims, const qsa_inputs *in, float *scores,
                                   void *ws, size_t ws_bytes, void *stream);

/* qsa_decode with the shared-history scorer: same launches otherwise, and
 * outputs bit-identical to qsa_decode (and so to one single-query decode per
 * query). */
qsa_status qsa_decode_shared(const qsa_dims *dims, const qsa_inputs *in, int32_t *ids,
                             int32_t *n_ids, float *out, void *ws, size_t ws_bytes, void *stream);

/* ---- attention without a workspace -------------------------------------- */

/* Fixed size of the device scratch behind qsa_attend_noalloc (4 MiB); every
 * GPU that loads the library holds it until the process exits. */
#define QSA_ATTEND_NOALLOC_SCRATCH_BYTES ((size_t)4 << 20)

/* Stage 4 without a workspace.  The notes have no counterpart to this call:
 * it exists for callers that cannot allocate device memory or pass a
 * workspace -- e.g. a plugin whose host runtime owns all device memory and
 * forbids third-party allocations, or a loop that must not allocate once it
 * runs.  Same arguments, kernel and results as qsa_attend, minus `ws`: the
 * error word, merge tickets and chunk partials live in one static device
 * array of QSA_ATTEND_NOALLOC_SCRATCH_BYTES.  Nothing is allocated or freed.
 *  - Size limit: 256 + align256(B*n_kv*4) + 2*align256(B*n_q*17*4)
 *    + align256(B*n_q*17*d*4) bytes must fit; larger dims return
 *    QSA_ERR_WORKSPACE_TOO_SMALL before anything is enqueued (e.g. B=8,
 *    n_q=16, d=128 needs 1.1 MB: fits; B=32 at the same shape does not).
 *  - The first call on each device, with that device current, looks up the
 *    array's device address (cudaGetSymbolAddress) and keeps it for the
 *    life of the process; make that first call before any stream capture.
 *    A cudaDeviceReset() can reload the library's device code at another
 *    address, so do not use this call after resetting the device in the
 *    same process.
 *  - Every call shares the array and it keeps the last call's contents: each
 *    call clears the error word and tickets on `stream` first.  Calls that
 *    overlap on the GPU (other streams, other threads) race on it.
 *  - Device-detected errors (an n_ids[b] outside [0, 4*budget+3]) zero that
 *    query's output; the error word is not reported by this call. */
qsa_status qsa_attend_noalloc(const qsa_dims *dims, const float *q, const float *k_scr,
                              const float *v_scr, const int32_t *n_ids, float *out, void *stream);

/* ---- measurement -------------------------------------------------------- */

/* Launches a binary32 FFMA throughput probe on `stream`: blocks_per_sm (1..8)
 * blocks of 256 threads per SM, each thread running 8 independent FMA chains
 * for iters x 16 steps; *fma_count (host) receives the FMAs the launch
 * performs.  The caller times it (events on `stream`): 2 * fma_count / time
 * is the FFMA peak that an FFMA-bound kernel of this library is reported
 * against.  sink: >= sms * blocks_per_sm floats of device memory, written
 * only to keep the chains from being optimised away (in practice never). */
qsa_status qsa_probe_ffma(int32_t blocks_per_sm, int32_t iters, float *sink, int64_t *fma_count,
                          void *stream);

#ifdef __cplusplus
}
#endif

#endif /* QSA_H */
