/*
 * qsa_oracle.c -- plain, slow, obviously-correct CPU reference for
 * physically sparse QSA decode.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: only the tests, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no code, header, table or helper with the
 * CUDA library; it is written from the two notes that define the method:
 *
 *   [AFN-017] "Top-k chooses the set; time chooses the order"
 *   [AFN-016] "A sparse mask is not sparse attention"
 *
 * Precision: the notes fix the path as model-free F32 ([AFN-016] Retrieval
 * capsule, claim boundary), so every floating-point step here is IEEE
 * binary32 with round-to-nearest, in one fixed order written out below.
 * Build with -ffp-contract=off so that no a*b+c is fused behind our back;
 * the only fused multiply-adds are the explicit fmaf() calls.
 *
 * Per query with T visible tokens:
 *   1. split   G = floor(T/4) complete groups [4g, 4g+4), tail [4G, T)
 *              ([AFN-017] Decision; [AFN-016] Decision)
 *   2. pool    p[j] = (((k0[j]+k1[j])+k2[j])+k3[j]) * 0.25   (mean)
 *              ([AFN-016] Why a sparse mask can still be dense: the
 *              indexer pools complete groups of raw index keys)
 *   3. score   s = sum_h ReLU(q_h . p), ReLU per head *before* the head
 *              sum; dot = fmaf chain j = 0..d-1 from +0; ReLU(x) = x>0?x:+0;
 *              head sum left to right from +0   (same section, "sum(ReLU(dot_h))")
 *   4. choose  the top min(G, budget) groups by (score desc, position asc),
 *              a full comparator sort -- ties resolved during membership
 *              ([AFN-017] Decision; Tie handling belongs to membership)
 *   5. emit    chosen groups sorted by ascending position, each expanded
 *              to 4 consecutive token IDs, then the raw tail appended
 *              ([AFN-017] Decision)
 *   6. resolve slot = slot_map[id], once, at one boundary
 *              ([AFN-016] Decision: only the gather crosses into the
 *              physical cache layout)
 *   7. attend  sequential online softmax over the emitted row in emitted
 *              (chronological) order: running max, rescale, exp,
 *              denominator and accumulator updates
 *              ([AFN-017] Floating point makes order observable;
 *              [AFN-016] Decision: online softmax over at most 2,051 rows)
 *
 * Readings where the notes are silent (each restated in the design notes):
 *   - pooling is the mean (sum would scale every score by exactly 4 and
 *     leave the selection unchanged; the tests check that);
 *   - one index key per token, shared by all indexer heads;
 *   - the FP32 summation orders above are this library's contract;
 *   - ReLU maps -0 and NaN to +0, so scores lie in [+0, +inf];
 *   - the tail is never scored and always appended;
 *   - T = 0 gives an empty row and a zero output vector;
 *   - index keys are addressed in logical order; the slot map applies to
 *     K/V only;
 *   - GQA: q head h reads KV head h / (n_q / n_kv).
 *
 * Parity pins: every function here is pinned by a CPU test against
 * something other than itself (closed forms on an exact integer grid,
 * brute-force enumeration, float64 definitions, invariants).  None is
 * "parity unpinned".
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define QSAO_GROUP 4

/* ---- 1. split ----------------------------------------------------------- */

int32_t qsao_num_groups(int32_t T) { return T > 0 ? T / QSAO_GROUP : 0; }
int32_t qsao_tail_len(int32_t T) { return T > 0 ? T % QSAO_GROUP : 0; }

/* Width of the emitted row: 4 * min(G, budget) + tail. */
int32_t qsao_row_width(int32_t T, int32_t budget)
{
    int32_t G = qsao_num_groups(T);
    int32_t k = G < budget ? G : budget;
    return QSAO_GROUP * k + qsao_tail_len(T);
}

/* ---- 2. pool ------------------------------------------------------------ */

/* k4 points at the 4 consecutive raw index keys of one group, each d floats.
 * pool_scale is 0.25f for the mean (1.0f gives the sum, used only by the
 * test that checks the mean/sum reading leaves the selection unchanged). */
void qsao_pool_group(const float *k4, int32_t d, float pool_scale, float *p)
{
    for (int32_t j = 0; j < d; ++j) {
        float acc = k4[j];
        acc = acc + k4[d + j];
        acc = acc + k4[2 * d + j];
        acc = acc + k4[3 * d + j];
        p[j] = acc * pool_scale;
    }
}

/* ---- 3. score ----------------------------------------------------------- */

/* q: [H, d] indexer query heads; p: [d] pooled group key. */
float qsao_score_pooled(const float *q, int32_t H, int32_t d, const float *p)
{
    float s = 0.0f;
    for (int32_t h = 0; h < H; ++h) {
        float acc = 0.0f;
        for (int32_t j = 0; j < d; ++j)
            acc = fmaf(q[(int64_t)h * d + j], p[j], acc);
        float r = acc > 0.0f ? acc : 0.0f;
        s = s + r;
    }
    return s;
}

/* Full-raw scoring: keys [T, d] are the query's raw index keys in logical
 * order; writes scores[0..G).  Each group's score depends on that group
 * alone, so when built with OpenMP the groups are shared out among the host
 * threads (same arithmetic per group, same results). */
void qsao_score_groups(const float *q, int32_t H, int32_t d, const float *keys,
                       int32_t T, float pool_scale, float *scores)
{
    int32_t G = qsao_num_groups(T);
#ifdef _OPENMP
#pragma omp parallel
#endif
    {
        float *p = (float *)malloc(sizeof(float) * (size_t)(d > 0 ? d : 1));
#ifdef _OPENMP
#pragma omp for schedule(static)
#endif
        for (int32_t g = 0; g < G; ++g) {
            qsao_pool_group(keys + (int64_t)g * QSAO_GROUP * d, d, pool_scale, p);
            scores[g] = qsao_score_pooled(q, H, d, p);
        }
        free(p);
    }
}

/* Host threads the scoring uses (1 without OpenMP); n <= 0 keeps the current
 * setting.  Returns the setting in force. */
int32_t qsao_threads(int32_t n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return (int32_t)omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* Incremental pooled-key cache ([AFN-017] Retrieval capsule names
 * "full-raw/incremental identity"): tokens arrive one at a time; the raw key
 * of token t is staged in pending[(t % 4) * d]; when t completes a group, that
 * group's pooled key is written to pooled[(t / 4) * d].  Scores are then read
 * from the cache instead of re-pooling the raw keys. */
void qsao_pool_cache_append(float *pooled, float *pending, int32_t d,
                            const float *key, int32_t t, float pool_scale)
{
    memcpy(pending + (int64_t)(t % QSAO_GROUP) * d, key, sizeof(float) * (size_t)d);
    if (t % QSAO_GROUP == QSAO_GROUP - 1)
        qsao_pool_group(pending, d, pool_scale, pooled + (int64_t)(t / QSAO_GROUP) * d);
}

void qsao_score_from_pooled(const float *q, int32_t H, int32_t d,
                            const float *pooled, int32_t G, float *scores)
{
    for (int32_t g = 0; g < G; ++g)
        scores[g] = qsao_score_pooled(q, H, d, pooled + (int64_t)g * d);
}

/* ---- 4./5. choose the set, emit in time order --------------------------- */

typedef struct {
    float s;
    int32_t g;
} qsao_cand;

/* Rank order: score descending, then group position ascending. */
static int qsao_cmp_rank(const void *a, const void *b)
{
    const qsao_cand *x = (const qsao_cand *)a, *y = (const qsao_cand *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->g > y->g) - (x->g < y->g);
}

static int qsao_cmp_pos(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* scores[0..G) for G = floor(T/4); writes the emitted logical token IDs to
 * ids (capacity >= qsao_row_width(T, budget)) and returns their count.
 * chosen (optional, capacity >= min(G, budget)) receives the chosen group
 * IDs in ascending position.  Scores must not be NaN. */
int32_t qsao_select(const float *scores, int32_t T, int32_t budget,
                    int32_t *ids, int32_t *chosen_out)
{
    int32_t G = qsao_num_groups(T);
    int32_t k = G < budget ? G : budget;
    if (k < 0) k = 0;
    qsao_cand *c = (qsao_cand *)malloc(sizeof(qsao_cand) * (size_t)(G > 0 ? G : 1));
    int32_t *chosen = (int32_t *)malloc(sizeof(int32_t) * (size_t)(k > 0 ? k : 1));
    for (int32_t g = 0; g < G; ++g) {
        c[g].s = scores[g];
        c[g].g = g;
    }
    qsort(c, (size_t)G, sizeof(qsao_cand), qsao_cmp_rank);   /* membership */
    for (int32_t r = 0; r < k; ++r) chosen[r] = c[r].g;
    qsort(chosen, (size_t)k, sizeof(int32_t), qsao_cmp_pos); /* time order */
    int32_t n = 0;
    for (int32_t r = 0; r < k; ++r)
        for (int32_t u = 0; u < QSAO_GROUP; ++u)
            ids[n++] = QSAO_GROUP * chosen[r] + u;              /* expand   */
    for (int32_t t = QSAO_GROUP * G; t < T; ++t) ids[n++] = t;  /* raw tail */
    if (chosen_out)
        for (int32_t r = 0; r < k; ++r) chosen_out[r] = chosen[r];
    free(chosen);
    free(c);
    return n;
}

/* The bounded dense row (AFN-011, named in [AFN-016] Failure boundary as the
 * dense oracle through 2,051 keys): every visible token, in order. */
int32_t qsao_dense_ids(int32_t T, int32_t *ids)
{
    int32_t n = 0;
    for (int32_t t = 0; t < T; ++t) ids[n++] = t;
    return n;
}

/* ---- 6. resolve --------------------------------------------------------- */

/* slot_map points at the query's region (logical token 0).  Returns 0, or
 * -(i+1) for the first row i whose slot is outside [0, num_slots). */
int32_t qsao_resolve(const int32_t *ids, int32_t n, const int32_t *slot_map,
                     int64_t num_slots, int32_t *slots)
{
    for (int32_t i = 0; i < n; ++i) {
        int32_t s = slot_map[ids[i]];
        if (s < 0 || (int64_t)s >= num_slots) return -(i + 1);
        slots[i] = s;
    }
    return 0;
}

/* ---- 7. attend ---------------------------------------------------------- */

/* The online-softmax state after visiting rows slots[0..n) in the given
 * order, for every q head h: m_out[h] the running maximum (-inf before any
 * row), l_out[h] the denominator, acc_out[h][0..d) the unnormalised output.
 * q: [n_q, d]; k_cache, v_cache: [num_slots, n_kv, d].  Sequential, one
 * visit per row. */
void qsao_attend_partial(const float *q, int32_t n_q, int32_t n_kv, int32_t d, float scale,
                         const float *k_cache, const float *v_cache,
                         const int32_t *slots, int32_t n,
                         float *m_out, float *l_out, float *acc_out)
{
    int32_t group = n_q / n_kv;
    /* heads are independent: shared among host threads under OpenMP */
#ifdef _OPENMP
#pragma omp parallel for schedule(static)
#endif
    for (int32_t h = 0; h < n_q; ++h) {
        int32_t kvh = h / group;
        const float *qh = q + (int64_t)h * d;
        float *acc = acc_out + (int64_t)h * d;
        float m = -INFINITY, l = 0.0f;
        for (int32_t j = 0; j < d; ++j) acc[j] = 0.0f;
        for (int32_t i = 0; i < n; ++i) {
            const float *k = k_cache + ((int64_t)slots[i] * n_kv + kvh) * d;
            const float *v = v_cache + ((int64_t)slots[i] * n_kv + kvh) * d;
            float dot = 0.0f;
            for (int32_t j = 0; j < d; ++j) dot = fmaf(qh[j], k[j], dot);
            float x = scale * dot;
            float m_new = x > m ? x : m;
            float alpha = (m == -INFINITY) ? 0.0f : expf(m - m_new);
            float p = expf(x - m_new);
            l = l * alpha + p;
            for (int32_t j = 0; j < d; ++j) acc[j] = acc[j] * alpha + p * v[j];
            m = m_new;
        }
        m_out[h] = m;
        l_out[h] = l;
    }
}

/* Online-softmax states of consecutive slices of one row merged in slice
 * order -- the step that joins slices attended apart ("Top-k chooses the set;
 * time chooses the order", Floating point makes order observable: the merge
 * keeps the row's time order).  m, l: [n_parts, n_q]; acc: [n_parts, n_q, d].
 * Starting from slice 0, slice r is folded in as one more block of the
 * online softmax:
 *   m' = max(m, m_r),  a = e^(m - m'),  a_r = e^(m_r - m')   (0 for m = -inf),
 *   l  = l a + l_r a_r,  acc = acc a + acc_r a_r,  m = m'.
 * out: [n_q, d] = acc / l (0 when l = 0). */
void qsao_merge_states(int32_t n_parts, int32_t n_q, int32_t d, const float *m_in, const float *l_in,
                       const float *acc_in, float *out)
{
    for (int32_t h = 0; h < n_q; ++h) {
        float m = -INFINITY, l = 0.0f;
        float *acc = out + (int64_t)h * d;
        for (int32_t j = 0; j < d; ++j) acc[j] = 0.0f;
        for (int32_t r = 0; r < n_parts; ++r) {
            const float mr = m_in[(int64_t)r * n_q + h];
            const float lr = l_in[(int64_t)r * n_q + h];
            const float *ar = acc_in + ((int64_t)r * n_q + h) * d;
            const float mn = mr > m ? mr : m;
            const float a = (m == -INFINITY) ? 0.0f : expf(m - mn);
            const float b = (mr == -INFINITY) ? 0.0f : expf(mr - mn);
            l = l * a + lr * b;
            for (int32_t j = 0; j < d; ++j) acc[j] = acc[j] * a + ar[j] * b;
            m = mn;
        }
        for (int32_t j = 0; j < d; ++j) acc[j] = l > 0.0f ? acc[j] / l : 0.0f;
    }
}

/* out: [n_q, d] = acc / l of the state above (0 for an empty row): the
 * attention of the q heads over the rows in the given order. */
void qsao_attend(const float *q, int32_t n_q, int32_t n_kv, int32_t d, float scale,
                 const float *k_cache, const float *v_cache,
                 const int32_t *slots, int32_t n, float *out)
{
    float *m = (float *)malloc(sizeof(float) * (size_t)(n_q > 0 ? n_q : 1));
    float *l = (float *)malloc(sizeof(float) * (size_t)(n_q > 0 ? n_q : 1));
    float *acc = (float *)malloc(sizeof(float) * (size_t)(n_q > 0 ? n_q : 1) * (size_t)d);
    qsao_attend_partial(q, n_q, n_kv, d, scale, k_cache, v_cache, slots, n, m, l, acc);
    for (int32_t h = 0; h < n_q; ++h) {
        float *o = out + (int64_t)h * d;
        for (int32_t j = 0; j < d; ++j) o[j] = l[h] > 0.0f ? acc[(int64_t)h * d + j] / l[h] : 0.0f;
    }
    free(acc);
    free(l);
    free(m);
}

/* ---- whole decode over a batch ------------------------------------------ */

/* Runs steps 1-7 for every query b of a batch, one after the other.
 *   q_idx     [B, H, dI]          idx_keys  [total_tokens, dI] logical order
 *   key_offset[B] first logical row of query b's history in idx_keys
 *   visible   [B] T_b             q [B, n_q, hd]
 *   k_cache, v_cache [num_slots, n_kv, hd]
 *   slot_map  [total_tokens]      slot_offset [B] first entry of b's region
 *   scores    [B, gstride] or NULL; ids [B, row_cap]; n_ids [B]; out [B, n_q, hd]
 * Returns 0, or 1 + b for the first query whose slot lookup was out of range
 * (that query's output is zero), or -1 for a T_b that does not fit. */
int32_t qsao_decode(int32_t B, int32_t H, int32_t dI, int32_t n_q, int32_t n_kv,
                    int32_t hd, int32_t budget, float scale,
                    const float *q_idx, const float *idx_keys, const int64_t *key_offset,
                    const int32_t *visible, const float *q,
                    const float *k_cache, const float *v_cache, int64_t num_slots,
                    const int32_t *slot_map, const int64_t *slot_offset,
                    float *scores, int32_t gstride,
                    int32_t *ids, int32_t row_cap, int32_t *n_ids, float *out)
{
    for (int32_t b = 0; b < B; ++b) {
        int32_t T = visible[b];
        if (T < 0 || qsao_row_width(T, budget) > row_cap ||
            (scores && qsao_num_groups(T) > gstride))
            return -1;
    }
    /* Queries are independent: under OpenMP they are shared among the host
     * threads, and the threads left over (fewer queries than threads) share
     * each query's groups and heads one level down.  Per-query results are
     * those of the sequential loop. */
    int32_t *st_b = (int32_t *)calloc((size_t)(B > 0 ? B : 1), sizeof(int32_t));
#ifdef _OPENMP
    int n_thr = omp_get_max_threads();
    int outer = B < n_thr ? (B > 0 ? B : 1) : n_thr;
    int inner = n_thr / outer > 0 ? n_thr / outer : 1;
    int levels = omp_get_max_active_levels();
    omp_set_max_active_levels(2);
#pragma omp parallel for num_threads(outer) schedule(dynamic, 1)
#endif
    for (int32_t b = 0; b < B; ++b) {
#ifdef _OPENMP
        omp_set_num_threads(inner);
#endif
        int32_t T = visible[b];
        int32_t G = qsao_num_groups(T);
        float *sc = (float *)malloc(sizeof(float) * (size_t)(G > 0 ? G : 1));
        qsao_score_groups(q_idx + (int64_t)b * H * dI, H, dI,
                          idx_keys + key_offset[b] * dI, T, 0.25f, sc);
        if (scores)
            for (int32_t g = 0; g < G; ++g) scores[(int64_t)b * gstride + g] = sc[g];
        int32_t *row = ids + (int64_t)b * row_cap;
        int32_t n = qsao_select(sc, T, budget, row, NULL);
        n_ids[b] = n;
        int32_t *slots = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n > 0 ? n : 1));
        float *ob = out + (int64_t)b * n_q * hd;
        if (qsao_resolve(row, n, slot_map + slot_offset[b], num_slots, slots) != 0) {
            for (int64_t e = 0; e < (int64_t)n_q * hd; ++e) ob[e] = 0.0f;
            st_b[b] = 1;
        } else {
            qsao_attend(q + (int64_t)b * n_q * hd, n_q, n_kv, hd, scale,
                        k_cache, v_cache, slots, n, ob);
        }
        free(slots);
        free(sc);
    }
#ifdef _OPENMP
    omp_set_max_active_levels(levels);
#endif
    int32_t status = 0;
    for (int32_t b = 0; b < B && status == 0; ++b)
        if (st_b[b]) status = 1 + b;
    free(st_b);
    return status;
}
