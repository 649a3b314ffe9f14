// qsa_internal.cuh -- internal declarations and device helpers of libqsa.
//
// Everything here is private to the library: the public boundary is
// include/qsa.h.  Kernels never trap: a bad index is skipped and recorded in
// the sticky device error word; every wait on an mbarrier is bounded in time.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "qsa.h"

namespace qsa {

// ---- workspace layout -----------------------------------------------------

constexpr int kGroup = 4;            // tokens per scored group
constexpr int kAttendRowsPerPart = 128;  // emitted rows per attention CTA (32 steps of 4)
constexpr int kAttendParts =             // attention CTAs (and partials) per (query, KV head) at
    (kGroup * QSA_MAX_BUDGET + kGroup - 1 + kAttendRowsPerPart - 1) / kAttendRowsPerPart;  // most: 17
constexpr int kMaxGqa = 16;          // q heads per KV head supported by attend

// The raw scorer's per-SM balance (in the workspace; all zero at first).
// The SMs do not stream equally fast -- the spread is mostly a property of
// each SM, stable from launch to launch -- so each scorer CTA, launched two
// per SM by a cooperative launch, takes a share of the tiles sized by the
// measured speed of the SM it runs on.  Each CTA records its time; one spare
// CTA of the following selection turns the times into the weights of the
// next launch.  The weights only move work between CTAs: the scores do not
// depend on them.
constexpr int kBalSlots = 256;                 // SM ids covered (larger ids: equal shares)
constexpr uint32_t kBalMagic = 0x51534231u;    // the weights below are complete
struct ScoreBalance {
    uint32_t magic;                  // kBalMagic once the weights are filled in
    uint32_t nsm;                    // SMs with a weight
    uint32_t w_total;                // sum of the weights
    uint32_t pad;
    uint32_t w_before[kBalSlots];    // sum of the weights of the lower SM ids
    uint32_t w[kBalSlots];           // weight of each SM id (0: none)
    uint32_t ctr[kBalSlots];         // CTAs ever started on the SM: tells its two CTAs apart
    uint32_t el_ns[kBalSlots][2];    // the last cooperative launch: each CTA's time (ns) ...
    uint32_t tiles[kBalSlots][2];    // ... and its tile count
};
constexpr size_t kWsAlign = 256;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Launches kernel<<<grid, block, smem, s>>>(args...), optionally with the
// programmatic stream-serialization attribute (see wait_for_predecessor).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                          bool pdl, Args &&...args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct Layout {
    int64_t score_stride;   // floats per scores row
    int64_t qmax_stride;    // entries per row of quad maxima (selection hint)
    int32_t row_cap;        // IDs per row: 4*budget + 3
    int32_t nparts;         // attention partials per (query, head): kAttendParts
    size_t off_err, off_tickets, off_bal, off_part_m, off_part_l, off_part_acc;
    size_t off_qmax, off_scores, off_ids, off_nids;
    size_t total;
};

bool dims_valid(const qsa_dims *d);
Layout make_layout(const qsa_dims *d);

// ---- launchers (one per stage) --------------------------------------------

struct ScoreArgs {
    const float *q_idx;
    const float *idx_keys;
    const int64_t *key_offset;
    const int32_t *visible;
    float *scores;
    int64_t score_stride;
    int32_t batch, idx_heads, idx_dim, max_visible;
    uint32_t *err;
    uint32_t *qmax;          // [B, qmax_stride]: order key of the max score of groups 4j..4j+3
    int64_t qmax_stride;
    // pooled != nullptr: score from the pooled-key cache, group g of query b
    // at row pool_offset[b] + g (idx_keys, key_offset unused)
    const float *pooled;
    const int64_t *pool_offset;
    // raw keys only: the per-SM balance (nullptr: equal shares per CTA)
    ScoreBalance *bal;
    int32_t bal_coop;        // set by the launcher: a cooperative launch, two CTAs on every SM
    // the failure-detection self-test: the producer issues no copy (no_issue)
    // and each copy wait gives up after wait_ns (0: the normal limit)
    int32_t no_issue;
    uint64_t wait_ns;
};
bool score_shape_supported(int idx_heads, int idx_dim);
cudaError_t launch_score(const ScoreArgs &a, int num_sms, cudaStream_t s);
// every query of the batch reads the history at key_offset[0] (checked on the device)
cudaError_t launch_score_shared(const ScoreArgs &a, int num_sms, cudaStream_t s);

struct PoolArgs {
    const float *idx_keys;
    const int64_t *key_offset;
    const int32_t *group_begin, *group_end;
    float *pooled;
    const int64_t *pool_offset;
    int32_t batch, idx_dim, max_groups, g_max;
    uint32_t *err;
};
cudaError_t launch_pool(const PoolArgs &a, cudaStream_t s);

// pdl: launch programmatically after the previous kernel in the stream
// (used only inside qsa_decode, where the order of the launches is fixed).

struct SelectArgs {
    const int32_t *visible;
    const float *scores;
    int64_t score_stride;
    int32_t *ids;
    int32_t *n_ids;
    int32_t row_cap, budget, max_visible, batch;
    uint32_t *err;
    const uint32_t *qmax;    // hint only: quad maxima as written by the scorer (may be stale)
    int64_t qmax_stride;
    // non-null: one CTA more than the batch turns the scorer's recorded
    // times into its next per-SM weights, once the scorer has finished
    ScoreBalance *bal;
    // non-null: the slot-map entries of the chosen groups are prefetched into
    // L2 for the attention kernel that follows (slot_map[slot_offset[b] + t])
    const int32_t *slot_map;
    const int64_t *slot_offset;
};
cudaError_t launch_select(const SelectArgs &a, cudaStream_t s, bool pdl = false);

struct GatherArgs {
    const int32_t *visible;
    const int32_t *ids;
    const int32_t *n_ids;
    const int32_t *slot_map;
    const int64_t *slot_offset;
    const float *k_cache, *v_cache;
    int64_t num_slots;
    float *k_scr, *v_scr;
    int32_t row_cap, row_floats, batch;
    uint32_t *err;
};
cudaError_t launch_gather(const GatherArgs &a, cudaStream_t s);

struct AttendArgs {
    const float *q;
    const float *k_scr, *v_scr;      // rows read from the gathered scratch (k_cache == nullptr)
    const int32_t *n_ids;
    float *out;
    float *part_m, *part_l, *part_acc;
    uint32_t *tickets;
    int32_t row_cap, nparts, batch, q_heads, kv_heads, head_dim;
    float scale;
    uint32_t *err;
    // fused gather: when k_cache != nullptr, rows are resolved through the slot
    // map and copied from the cache; when k_scr_out != nullptr they are also
    // written to k_scr_out / v_scr_out (the gather's output)
    const int32_t *ids;
    const int32_t *visible;
    const int32_t *slot_map;
    const int64_t *slot_offset;
    const float *k_cache, *v_cache;
    int64_t num_slots;
    float *k_scr_out, *v_scr_out;
    // set by the launcher (grids of more than one wave): every run CTA writes
    // its state and leaves; a second, small launch merges the runs (the same
    // arithmetic as the last CTA's merge, so the same bits)
    int32_t defer_merge;
    // the whole-path call: ids / n_ids are the selection's rows in the
    // workspace; each run CTA of KV head 0 also stores its rows (and CTA
    // (run 0, KV head 0) the count) to the caller's ids_out / n_ids_out, as
    // it stores `out` -- so the results reach the caller's memory, wherever it
    // is, from the kernel that finishes the path (nullptr: not wanted)
    int32_t *ids_out, *n_ids_out;
    // the state export: when m_out != nullptr, `out` receives the unnormalised
    // accumulator sum_i e^(s_i - m) v_i of each head, m_out the running max m
    // and l_out the denominator sum_i e^(s_i - m), instead of the output
    float *m_out, *l_out;
};
bool attend_shape_supported(int head_dim, int q_heads, int kv_heads);
cudaError_t launch_attend(const AttendArgs &a, cudaStream_t s, bool pdl = false);
// states [n_parts, bh] (m, l) and [n_parts, bh, head_dim] (acc) -> out [bh, head_dim]
cudaError_t launch_merge_states(const float *m, const float *l, const float *acc, float *out, int n_parts,
                                int bh, int head_dim, cudaStream_t s);

// ---- device helpers ---------------------------------------------------------

// Order-preserving uint32 image of a score: larger float, larger key; -0 is
// folded to +0 first.  Scores from the scorer are in [+0, +inf].
__device__ __forceinline__ uint32_t order_key(float x)
{
    const uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ void set_error(uint32_t *err, uint32_t bit)
{
    atomicOr(err, bit);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_mbar_init()
{
    // make the initialised barriers visible to the async (bulk copy) proxy
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// Waits for the given phase parity of an mbarrier for at most limit_ns
// nanoseconds of wall time.  Returns false if the time ran out.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint64_t limit_ns)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// One-dimensional bulk copy global -> shared, completing on an mbarrier.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// An L2 policy that marks the lines a load brings in as first to evict: for
// data streamed once, so that it does not push out data that is read again soon.
__device__ __forceinline__ uint64_t l2_evict_first_policy()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// bulk_copy_g2s with an L2 cache policy for the source lines.
__device__ __forceinline__ void bulk_copy_g2s_hint(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                                   uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
        : "memory");
}

// One-dimensional bulk copy shared -> global in this thread's bulk async-group.
// dst, src 16-byte aligned; bytes a multiple of 16.
__device__ __forceinline__ void bulk_copy_s2g(void *dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// This thread's committed bulk stores have finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
// ... and have completed their writes.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Orders this thread's generic-proxy writes to shared memory before later
// async-proxy (bulk copy) accesses of the same bytes.
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while its predecessor drains; it
// must wait here before touching anything the predecessor writes.  Both
// instructions are no-ops for a kernel launched the ordinary way.
__device__ __forceinline__ void wait_for_predecessor()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Lets the next kernel in the stream (if launched programmatically) begin
// launching; its CTAs still wait in wait_for_predecessor() for this grid.
__device__ __forceinline__ void allow_successor_launch()
{
    asm volatile("griddepcontrol.launch_dependents;" :::);
}

// Asks L2 to fetch the 128-byte line holding p (no data returned, nothing
// waits).  Only for addresses the caller's own loads will touch.
__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

constexpr uint64_t kWaitLimitNs = 1000000000ull;     // 1 s for a copy to land
constexpr uint64_t kDrainLimitNs = 100000000ull;     // 0.1 s per copy when draining

}  // namespace qsa
