// select.cu -- stage 2: choose the set, emit it in time order.
//
// "Top-k chooses the set; time chooses the order" (AFN-017), Decision and
// Tie handling belongs to membership: the top k = min(G, budget) groups by
// (score descending, group position ascending) form the set -- ties decided
// while choosing membership -- and the set is emitted in ascending position,
// each group expanded to 4 consecutive token IDs, then the raw tail appended.
//
// GPU design (no sort anywhere).  One thread-block cluster of kCl CTAs per
// query; CTA r owns a contiguous slice of the query's G scores, cached in
// shared memory as order-preserving uint32 keys (float bits, sign-folded; -0
// folded to +0).  Membership is `key > s*`, or `key == s*` among the first
// `need` equal keys in ascending position (the tie rule applied during
// membership), where s* is the k-th largest key and need = k - #(key > s*);
// a chosen group's output slot is #(key > s* before it) + min(need,
// #(key == s* before it)), so the row comes out in ascending position.
//
// Fast path (exact): every CTA cuts its slice into ceil(k / kCl) disjoint
// blocks, so the cluster has at least k blocks; L = min over blocks of the
// block maximum is then a lower bound of s* (each block holds a key >= L).
// Keys >= L -- typically a few thousand of 65,536 -- are compacted in
// position order into rank 0's shared memory through distributed shared
// memory, and rank 0 alone finishes: radix select of s* on 12-bit digits of
// (key - L), then the ordered emission, with no further cluster barriers.
//
// Full path (when the candidates do not fit, e.g. when everything ties): a
// cluster-wide radix select in three passes (11/11/10 bits) -- per-CTA shared
// histograms summed over distributed shared memory -- then the ordered
// emission over every key, using per-CTA totals exchanged the same way.
// Below budget (G <= budget) every group is chosen and the row is 0..T-1.
#include <cooperative_groups.h>

#include "qsa_internal.cuh"

namespace cg = cooperative_groups;

namespace qsa {
namespace {

constexpr int kCl = 8;             // CTAs per query (one cluster)
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;        // full path: widest radix digit, 11 bits
constexpr int kLocalBits = 12;     // fast path: digits of (key - L)
constexpr int kLocalBins = 1 << kLocalBits;
constexpr int kCacheKeys = 24576;  // slice keys kept in shared memory (96 KB)
constexpr int kCandCap = 8192;     // fast-path candidates held by rank 0 (64 KB)

// Scores per cluster CTA: ceil(G / kCl) rounded up to 32, so every slice
// starts on a 128-byte boundary of the scores row.
__host__ __device__ __forceinline__ int slice_len(int G)
{
    return ((G + kCl - 1) / kCl + 31) & ~31;
}

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

// Each thread holds NB consecutive bin counts (thread t: bins NB*t..NB*t+NB-1).
// Finds the digit d with above(d) < remaining <= above(d) + count(d), where
// above(d) counts the keys in bins > d, and publishes it.
template <int NB>
__device__ __forceinline__ void find_digit(const uint32_t (&c)[NB], uint32_t remaining, uint64_t *warp_tmp,
                                           uint32_t *found_digit, uint32_t *found_above)
{
    uint32_t mine = 0;
#pragma unroll
    for (int q = 0; q < NB; ++q) mine += c[q];
    uint64_t total;
    const uint64_t below_me = block_excl_scan_u64(uint64_t(mine), warp_tmp, &total);
    uint32_t above = uint32_t(total - below_me - mine);
#pragma unroll
    for (int q = NB - 1; q >= 0; --q) {
        if (above < remaining && remaining <= above + c[q]) {
            *found_digit = uint32_t(NB * threadIdx.x + q);
            *found_above = above;
        }
        above += c[q];
    }
}

// Ordered emission over keys [0, n) (any key source): the keys > thr and the
// first `need` keys == thr, each written as 4 token IDs at its output slot.
// gt_base / eq_base count the keys of each kind that precede key 0.
template <typename KeyAt, typename GroupAt>
__device__ __forceinline__ void emit_in_order(KeyAt key_at, GroupAt group_at, int n, uint32_t thr, uint32_t need,
                                              int k, uint32_t gt_base, uint32_t eq_base, uint64_t *warp_tmp,
                                              int32_t *row, uint32_t *err, uint32_t *cta_gt, uint32_t *cta_eq,
                                              bool publish_only)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int run = ((n + kWarps - 1) / kWarps + 31) & ~31;
    const int w0 = min(n, warp * run);
    const int w1 = min(n, w0 + run);
    uint32_t n_gt = 0, n_eq = 0;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < w1 ? key_at(i) : 0u;
        n_gt += __popc(__ballot_sync(0xffffffffu, i < w1 && key > thr));
        n_eq += __popc(__ballot_sync(0xffffffffu, i < w1 && key == thr));
    }
    uint64_t tot;
    const uint64_t excl = block_excl_scan_u64(lane == 0 ? ((uint64_t(n_eq) << 32) | n_gt) : 0, warp_tmp, &tot);
    if (publish_only) {
        if (threadIdx.x == 0) {
            *cta_gt = uint32_t(tot);
            *cta_eq = uint32_t(tot >> 32);
        }
        return;
    }
    const uint64_t mine = __shfl_sync(0xffffffffu, excl, 0);  // lane 0 holds the warp's prefix
    uint32_t gt_c = gt_base + uint32_t(mine);
    uint32_t eq_c = eq_base + uint32_t(mine >> 32);
    const uint32_t lt_mask = (1u << lane) - 1u;
    for (int base = w0; base < w1; base += 32) {
        const int i = base + lane;
        const uint32_t key = i < w1 ? key_at(i) : 0u;
        const bool is_gt = i < w1 && key > thr;
        const bool is_eq = i < w1 && key == thr;
        const uint32_t bg = __ballot_sync(0xffffffffu, is_gt);
        const uint32_t be = __ballot_sync(0xffffffffu, is_eq);
        const uint32_t my_gt = gt_c + __popc(bg & lt_mask);  // greater keys before this one
        const uint32_t my_eq = eq_c + __popc(be & lt_mask);  // equal keys before this one
        int pos = -1;
        if (is_gt) pos = int(my_gt + min(need, my_eq));
        else if (is_eq && my_eq < need) pos = int(my_gt + my_eq);
        if (pos >= k) {  // cannot happen for a correct threshold; never write past the row
            set_error(err, QSA_DEVERR_ROW_RANGE);
            pos = -1;
        }
        if (pos >= 0) {
            const int g = group_at(i);
            int32_t *o = row + kGroup * pos;
            o[0] = kGroup * g;
            o[1] = kGroup * g + 1;
            o[2] = kGroup * g + 2;
            o[3] = kGroup * g + 3;
        }
        gt_c += __popc(bg);
        eq_c += __popc(be);
    }
}

template <bool kCached>
__global__ void __cluster_dims__(kCl, 1, 1) __launch_bounds__(kThreads, 1)
select_emit_kernel(const SelectArgs a)
{
    extern __shared__ __align__(16) uint32_t dyn[];
    uint32_t *cand_key = dyn;                                          // [kCandCap], rank 0
    int32_t *cand_g = reinterpret_cast<int32_t *>(dyn + kCandCap);     // [kCandCap], rank 0
    uint32_t *keys = dyn + 2 * kCandCap;                               // [slice] when kCached
    __shared__ __align__(16) uint32_t hist[2][kLocalBins];
    __shared__ uint64_t warp_tmp[kWarps];
    __shared__ uint32_t warp_red[kWarps];
    __shared__ uint32_t found_digit, found_above;
    __shared__ uint32_t cta_gt, cta_eq, cta_min, cta_cand, bcast[2];

    cg::cluster_group cluster = cg::this_cluster();
    const int rank = int(cluster.block_rank());
    const int b = blockIdx.x / kCl;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;

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

    const int slice = slice_len(G);
    const int lo = min(G, rank * slice);
    const int cnt = min(G, lo + slice) - lo;
    const float *src = a.scores + int64_t(b) * a.score_stride + lo;
    if (kCached) {
        // slices start on 128-byte boundaries: 16-byte loads, all in flight
        const float4 *src4 = reinterpret_cast<const float4 *>(src);
        const int n4 = cnt >> 2;
        int i = tid;
        for (; i + 3 * kThreads < n4; i += 4 * kThreads) {
            float4 x[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) x[u] = __ldg(src4 + i + u * kThreads);
#pragma unroll
            for (int u = 0; u < 4; ++u)
                *reinterpret_cast<uint4 *>(keys + 4 * (i + u * kThreads)) =
                    make_uint4(order_key(x[u].x), order_key(x[u].y), order_key(x[u].z), order_key(x[u].w));
        }
        for (; i < n4; i += kThreads) {
            const float4 x = __ldg(src4 + i);
            *reinterpret_cast<uint4 *>(keys + 4 * i) =
                make_uint4(order_key(x.x), order_key(x.y), order_key(x.z), order_key(x.w));
        }
        for (int j = 4 * n4 + tid; j < cnt; j += kThreads) keys[j] = order_key(__ldg(src + j));
        __syncthreads();
    }
    auto key_at = [&](int i) -> uint32_t { return kCached ? keys[i] : order_key(__ldg(src + i)); };
    auto group_at = [&](int i) -> int { return lo + i; };

    // ---- fast path: lower bound L, candidates, rank 0 finishes -------------------
    const int kb = (k + kCl - 1) / kCl;  // blocks per CTA; kCl * kb >= k
    if (slice >= kb && G - (kCl - 1) * slice >= kb) {  // every CTA can form kb blocks (uniform)
        const int bsz = cnt / kb;
        uint32_t wmin = 0xffffffffu;
        for (int j = warp; j < kb; j += kWarps) {
            uint32_t m = 0;
            for (int i = j * bsz + lane; i < (j + 1) * bsz; i += 32) m = max(m, key_at(i));
            m = __reduce_max_sync(0xffffffffu, m);
            wmin = min(wmin, m);
        }
        if (lane == 0) warp_red[warp] = wmin;
        __syncthreads();
        if (tid == 0) {
            uint32_t m = 0xffffffffu;
            for (int w = 0; w < kWarps; ++w) m = min(m, warp_red[w]);
            cta_min = m;
        }
        cluster.sync();
        if (warp == 0) {
            uint32_t m = lane < kCl ? *cluster.map_shared_rank(&cta_min, lane) : 0xffffffffu;
            m = __reduce_min_sync(0xffffffffu, m);
            if (lane == 0) bcast[0] = m;
        }
        __syncthreads();
        const uint32_t L = bcast[0];  // <= the k-th largest key of the query

        // candidates (key >= L) of this CTA, counted per warp range in order
        const int run = ((cnt + kWarps - 1) / kWarps + 31) & ~31;
        const int w0 = min(cnt, warp * run);
        const int w1 = min(cnt, w0 + run);
        uint32_t n_c = 0;
        for (int base = w0; base < w1; base += 32) {
            const int i = base + lane;
            n_c += __popc(__ballot_sync(0xffffffffu, i < w1 && key_at(i) >= L));
        }
        uint64_t tot;
        const uint64_t excl = block_excl_scan_u64(lane == 0 ? uint64_t(n_c) : 0, warp_tmp, &tot);
        if (tid == 0) cta_cand = uint32_t(tot);
        cluster.sync();
        if (warp == 0) {
            const uint32_t c_r = lane < kCl ? *cluster.map_shared_rank(&cta_cand, lane) : 0u;
            const uint32_t before = __reduce_add_sync(0xffffffffu, lane < rank ? c_r : 0u);
            const uint32_t total_c = __reduce_add_sync(0xffffffffu, c_r);
            if (lane == 0) {
                bcast[0] = before;
                bcast[1] = total_c;
            }
        }
        __syncthreads();
        const uint32_t total_c = bcast[1];
        if (total_c <= uint32_t(kCandCap)) {  // uniform: every CTA read the same totals
            uint32_t *rk = cluster.map_shared_rank(cand_key, 0);
            int32_t *rg = cluster.map_shared_rank(cand_g, 0);
            uint32_t pos = bcast[0] + uint32_t(__shfl_sync(0xffffffffu, excl, 0));
            const uint32_t lt_mask = (1u << lane) - 1u;
            for (int base = w0; base < w1; base += 32) {
                const int i = base + lane;
                const uint32_t key = i < w1 ? key_at(i) : 0u;
                const bool c = i < w1 && key >= L;
                const uint32_t bc = __ballot_sync(0xffffffffu, c);
                if (c) {
                    const uint32_t at = pos + __popc(bc & lt_mask);
                    rk[at] = key;
                    rg[at] = lo + i;
                }
                pos += __popc(bc);
            }
            cluster.sync();  // candidates are in rank 0; nobody reads another CTA after this
            if (rank != 0) return;

            // rank 0: radix select of the k-th largest candidate on (key - L)
            const int n = int(total_c);
            uint32_t mx = 0;
            for (int i = tid; i < n; i += kThreads) mx = max(mx, cand_key[i]);
            mx = __reduce_max_sync(0xffffffffu, mx);
            if (lane == 0) warp_red[warp] = mx;
            __syncthreads();
            if (tid == 0) {
                uint32_t m = 0;
                for (int w = 0; w < kWarps; ++w) m = max(m, warp_red[w]);
                bcast[0] = m;
            }
            __syncthreads();
            const uint32_t range = bcast[0] - L;
            const int nbits = range == 0 ? 0 : 32 - __clz(range);
            uint32_t prefix = 0, pmask = 0, remaining = uint32_t(k);
            int pass = 0;
            for (int hi = nbits; hi > 0; hi -= kLocalBits, ++pass) {
                const int lo_bit = max(hi - kLocalBits, 0);
                const uint32_t dmask = (1u << (hi - lo_bit)) - 1u;
                uint32_t *h = hist[pass & 1];
                for (int i = tid; i < kLocalBins; i += kThreads) h[i] = 0;
                __syncthreads();
                for (int base = warp * 32; base < n; base += kThreads) {
                    const int i = base + lane;
                    uint32_t bin = 0xffffffffu;
                    if (i < n) {
                        const uint32_t off = cand_key[i] - L;
                        if ((off & pmask) == prefix) bin = (off >> lo_bit) & dmask;
                    }
                    const uint32_t peers = __match_any_sync(0xffffffffu, bin);
                    if (bin != 0xffffffffu && lane == __ffs(peers) - 1) atomicAdd(&h[bin], uint32_t(__popc(peers)));
                }
                __syncthreads();
                constexpr int NB = kLocalBins / kThreads;
                uint32_t c[NB];
#pragma unroll
                for (int q = 0; q < NB; ++q) c[q] = h[NB * tid + q];
                find_digit<NB>(c, remaining, warp_tmp, &found_digit, &found_above);
                __syncthreads();
                prefix |= found_digit << lo_bit;
                pmask |= dmask << lo_bit;
                remaining -= found_above;
                __syncthreads();
            }
            emit_in_order([&](int i) { return cand_key[i]; }, [&](int i) { return cand_g[i]; }, n, L + prefix,
                          remaining, k, 0u, 0u, warp_tmp, row, a.err, &cta_gt, &cta_eq, false);
            if (tid < tail) row[kGroup * k + tid] = kGroup * G + tid;
            if (tid == 0) a.n_ids[b] = kGroup * k + tail;
            return;
        }
        // too many candidates (heavy ties): every CTA takes the full path
    }

    // ---- full path: cluster-wide radix select of the k-th largest key -------------
    uint32_t prefix = 0, pmask = 0, remaining = uint32_t(k);
    if (tid == 0) {
        found_digit = 0;
        found_above = 0;
    }
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        uint32_t *h = hist[pass & 1];
        for (int i = tid; i < kBins; i += kThreads) h[i] = 0;
        __syncthreads();
        const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const uint32_t dmask = pass == 2 ? 0x3ffu : 0x7ffu;
        // Warp-aggregated increments: lanes holding the same digit add once.
        for (int base = warp * 32; base < cnt; base += kThreads) {
            const int i = base + lane;
            uint32_t bin = 0xffffffffu;
            if (i < cnt) {
                const uint32_t key = key_at(i);
                if ((key & pmask) == prefix) bin = (key >> sh) & dmask;
            }
            const uint32_t peers = __match_any_sync(0xffffffffu, bin);
            if (bin != 0xffffffffu && lane == __ffs(peers) - 1) atomicAdd(&h[bin], uint32_t(__popc(peers)));
        }
        // All eight local histograms complete.  (Two buffers: the one zeroed
        // next pass was last read remotely before this barrier.)
        cluster.sync();
        uint4 v[kCl];
#pragma unroll
        for (int r = 0; r < kCl; ++r) v[r] = *reinterpret_cast<const uint4 *>(cluster.map_shared_rank(h, r) + 4 * tid);
        uint32_t c[4] = {0, 0, 0, 0};
#pragma unroll
        for (int r = 0; r < kCl; ++r) {
            c[0] += v[r].x;
            c[1] += v[r].y;
            c[2] += v[r].z;
            c[3] += v[r].w;
        }
        find_digit<4>(c, remaining, warp_tmp, &found_digit, &found_above);
        __syncthreads();
        prefix |= found_digit << sh;
        pmask |= dmask << sh;
        remaining -= found_above;
        __syncthreads();
    }
    const uint32_t thr = prefix;     // the k-th largest key
    const uint32_t need = remaining; // equal keys to take, in ascending position

    // ---- membership and emission in ascending position -----------------------
    emit_in_order(key_at, group_at, cnt, thr, need, k, 0u, 0u, warp_tmp, row, a.err, &cta_gt, &cta_eq, true);
    cluster.sync();
    uint32_t gt_c = 0, eq_c = 0;
#pragma unroll
    for (int r = 0; r < kCl; ++r) {
        if (r < rank) {
            gt_c += *cluster.map_shared_rank(&cta_gt, r);
            eq_c += *cluster.map_shared_rank(&cta_eq, r);
        }
    }
    emit_in_order(key_at, group_at, cnt, thr, need, k, gt_c, eq_c, warp_tmp, row, a.err, &cta_gt, &cta_eq, false);
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
    const int slice = slice_len(gmax);
    const bool cached = slice <= kCacheKeys;
    const size_t cand_bytes = size_t(2) * kCandCap * 4;
    const size_t dyn = cand_bytes + (cached ? size_t(slice > 0 ? slice : 1) * 4 : 0);
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(select_emit_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(cand_bytes + size_t(kCacheKeys) * 4));
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(select_emit_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 int(cand_bytes));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const dim3 grid(unsigned(a.batch) * kCl);
    if (cached)
        select_emit_kernel<true><<<grid, kThreads, dyn, s>>>(a);
    else
        select_emit_kernel<false><<<grid, kThreads, dyn, s>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa
