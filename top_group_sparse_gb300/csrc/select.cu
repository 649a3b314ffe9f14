// select.cu -- stage 2: choose the set, emit it in time order.
//
// "Top-k chooses the set; time chooses the order" (AFN-017), Decision and
// Tie handling belongs to membership: the top k = min(G, budget) groups by
// (score descending, group position ascending) form the set -- ties decided
// while choosing membership -- and the set is emitted in ascending position,
// each group expanded to 4 consecutive token IDs, then the raw tail appended.
//
// GPU design (no sort anywhere):
//  * One thread-block cluster of kCl CTAs per query; CTA r owns a contiguous
//    slice of the query's G scores, cached in shared memory as order-preserving
//    uint32 keys (float bits, sign-folded; -0 folded to +0).
//  * Radix select of the k-th largest key in three passes (11/11/10 bits):
//    each CTA histograms its slice into shared memory, the cluster sums the
//    eight histograms through distributed shared memory, and every CTA finds
//    the same digit.  Result: threshold key s* and need = k - #(key > s*).
//  * Membership: key > s*, or key == s* and among the first `need` equal keys
//    in ascending position (the tie rule, applied during membership).
//  * Emission: output position of a chosen group g is
//      #(key > s* before g) + min(need, #(key == s* before g)),
//    from one block scan per CTA plus the lower CTAs' totals (again through
//    distributed shared memory), so the row comes out in ascending position.
// Below budget (G <= budget) every group is chosen and the row is 0..T-1.
#include <cooperative_groups.h>

#include "qsa_internal.cuh"

namespace cg = cooperative_groups;

namespace qsa {
namespace {

constexpr int kCl = 8;             // CTAs per query (one cluster)
constexpr int kThreads = 512;
constexpr int kBins = 2048;        // widest radix digit: 11 bits
constexpr int kWarps = kThreads / 32;
constexpr int kCacheKeys = 49152;  // slice keys kept in shared memory (192 KB)

__device__ __forceinline__ uint32_t order_key(float x)
{
    uint32_t u = __float_as_uint(x == 0.0f ? 0.0f : x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Block-wide exclusive scan of a 64-bit value; *total receives the sum.
__device__ __forceinline__ uint64_t block_excl_scan_u64(uint64_t v, uint64_t *warp_tmp, uint64_t *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint64_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint64_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tmp[warp] = x;
    __syncthreads();
    if (warp == 0) {
        uint64_t w = lane < kWarps ? warp_tmp[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint64_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kWarps) warp_tmp[lane] = w;  // inclusive warp prefix
    }
    __syncthreads();
    const uint64_t warp_before = warp == 0 ? 0 : warp_tmp[warp - 1];
    *total = warp_tmp[kWarps - 1];
    const uint64_t r = warp_before + x - v;
    __syncthreads();  // warp_tmp may be reused by the caller
    return r;
}

template <bool kCached>
__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kThreads, 1)
select_emit_kernel(const SelectArgs a)
{
    extern __shared__ __align__(16) uint32_t keys[];  // [slice] when kCached
    __shared__ __align__(16) uint32_t hist[2][kBins];
    __shared__ uint64_t warp_tmp[kWarps];
    __shared__ uint32_t found_digit, found_above;
    __shared__ uint32_t cta_gt, cta_eq;

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int b = blockIdx.x / kCl;
    const int tid = threadIdx.x;

    const int T = __ldg(a.visible + b);
    int32_t *row = a.ids + int64_t(b) * a.row_cap;
    if (T < 0 || T > a.max_visible) {
        if (rank == 0 && tid == 0) {
            a.n_ids[b] = 0;
            set_error(a.err, QSA_DEVERR_VISIBLE_RANGE);
        }
        return;  // uniform across the cluster: every CTA read the same T
    }
    const int G = T >> 2;
    const int tail = T & 3;
    const int k = G < a.budget ? G : a.budget;
    if (G <= a.budget) {
        // Every complete group is chosen: the row is the dense causal row.
        for (int i = rank * kThreads + tid; i < T; i += kCl * kThreads) row[i] = i;
        if (rank == 0 && tid == 0) a.n_ids[b] = T;
        return;
    }

    const int slice = (G + kCl - 1) / kCl;
    const int lo = min(G, rank * slice);
    const int cnt = min(G, lo + slice) - lo;
    const float *src = a.scores + int64_t(b) * a.score_stride + lo;
    if (kCached) {
        for (int i = tid; i < cnt; i += kThreads) keys[i] = order_key(__ldg(src + i));
    }
    auto key_at = [&](int i) -> uint32_t { return kCached ? keys[i] : order_key(__ldg(src + i)); };

    // ---- radix select of the k-th largest key --------------------------------
    uint32_t prefix = 0, pmask = 0, remaining = uint32_t(k);
    if (tid == 0) {
        found_digit = 0;
        found_above = 0;
    }
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        uint32_t *h = hist[pass & 1];
        for (int i = tid; i < kBins; i += kThreads) h[i] = 0;
        __syncthreads();
        const int sh = shifts[pass];
        const uint32_t dmask = (1u << widths[pass]) - 1u;
        for (int i = tid; i < cnt; i += kThreads) {
            const uint32_t key = key_at(i);
            if ((key & pmask) == prefix) atomicAdd(&h[(key >> sh) & dmask], 1u);
        }
        // All eight local histograms complete.  (Two buffers: the one zeroed
        // next pass was last read remotely before this barrier.)
        cluster.sync();
        uint32_t c[4] = {0, 0, 0, 0};
#pragma unroll 1
        for (int r = 0; r < kCl; ++r) {
            const uint4 v = *reinterpret_cast<const uint4 *>(cluster.map_shared_rank(h, r) + 4 * tid);
            c[0] += v.x;
            c[1] += v.y;
            c[2] += v.z;
            c[3] += v.w;
        }
        // above(d) = number of keys matching the prefix with digit > d.
        uint64_t total;
        const uint64_t below_me = block_excl_scan_u64(uint64_t(c[0] + c[1] + c[2] + c[3]), warp_tmp, &total);
        uint32_t above = uint32_t(total - below_me - (c[0] + c[1] + c[2] + c[3]));
#pragma unroll
        for (int q = 3; q >= 0; --q) {
            if (above < remaining && remaining <= above + c[q]) {
                found_digit = uint32_t(4 * tid + q);
                found_above = above;
            }
            above += c[q];
        }
        __syncthreads();
        prefix |= found_digit << sh;
        pmask |= dmask << sh;
        remaining -= found_above;
        __syncthreads();
    }
    const uint32_t thr = prefix;    // the k-th largest key
    const uint32_t need = remaining; // equal keys to take, in ascending position

    // ---- membership and emission in ascending position ---------------------
    const int run = (cnt + kThreads - 1) / kThreads;
    const int a0 = min(cnt, tid * run);
    const int a1 = min(cnt, a0 + run);
    uint32_t n_gt = 0, n_eq = 0;
    for (int i = a0; i < a1; ++i) {
        const uint32_t key = key_at(i);
        n_gt += key > thr;
        n_eq += key == thr;
    }
    uint64_t cta_total;
    const uint64_t excl = block_excl_scan_u64((uint64_t(n_eq) << 32) | n_gt, warp_tmp, &cta_total);
    if (tid == 0) {
        cta_gt = uint32_t(cta_total);
        cta_eq = uint32_t(cta_total >> 32);
    }
    cluster.sync();
    uint32_t gt_c = 0, eq_c = 0;
    for (int r = 0; r < rank; ++r) {
        gt_c += *cluster.map_shared_rank(&cta_gt, r);
        eq_c += *cluster.map_shared_rank(&cta_eq, r);
    }
    gt_c += uint32_t(excl);
    eq_c += uint32_t(excl >> 32);
    for (int i = a0; i < a1; ++i) {
        const uint32_t key = key_at(i);
        int pos = -1;
        if (key > thr) {
            pos = int(gt_c + min(need, eq_c));
            ++gt_c;
        } else if (key == thr) {
            if (eq_c < need) pos = int(gt_c + eq_c);
            ++eq_c;
        }
        if (pos >= k) {  // cannot happen for a correct threshold; never write past the row
            set_error(a.err, QSA_DEVERR_ROW_RANGE);
            pos = -1;
        }
        if (pos >= 0) {
            const int g = lo + i;
            int32_t *o = row + kGroup * pos;
            o[0] = kGroup * g;
            o[1] = kGroup * g + 1;
            o[2] = kGroup * g + 2;
            o[3] = kGroup * g + 3;
        }
    }
    if (rank == 0) {
        if (tid < tail) row[kGroup * k + tid] = kGroup * G + tid;
        if (tid == 0) a.n_ids[b] = kGroup * k + tail;
    }
    cluster.sync();  // keep this CTA's shared memory alive for remote readers
}

}  // namespace

cudaError_t launch_select(const SelectArgs &a, cudaStream_t s)
{
    if (a.batch == 0) return cudaSuccess;
    const int gmax = a.max_visible / kGroup;
    const int slice = (gmax + kCl - 1) / kCl;
    const bool cached = slice <= kCacheKeys;
    const size_t dyn = cached ? size_t(slice > 0 ? slice : 1) * 4 : 0;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(select_emit_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             kCacheKeys * 4);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const dim3 grid(unsigned(a.batch) * kCl);
    if (cached)
        select_emit_kernel<true><<<grid, kThreads, dyn, s>>>(a);
    else
        select_emit_kernel<false><<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa
