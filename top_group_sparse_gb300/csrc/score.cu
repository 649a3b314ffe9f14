// score.cu -- stage 1: group scoring.
//
// "A sparse mask is not sparse attention" (AFN-016), Decision: score complete
// groups in bounded tiles; Why a sparse mask can still be dense: the indexer
// pools complete four-token groups of raw index keys and scores each as
// sum(ReLU(dot_h)).  The score of group g of query b is
//
//   p[j] = (((k[4g][j] + k[4g+1][j]) + k[4g+2][j]) + k[4g+3][j]) * 0.25
//   s    = sum over h = 0..H-1, left to right from +0, of ReLU(dot_h),
//   dot_h = fma chain over j = 0..D-1 from +0,  ReLU(x) = x > 0 ? x : +0,
//
// in binary32 round-to-nearest with the __f*_rn intrinsics, which the
// compiler never contracts or reorders: scores are bit-identical to any
// implementation of that order.  No tensor cores: the order is the contract.
//
// The stage is a stream over the raw keys (T * D * 4 bytes per query), so it
// is bound by HBM bandwidth.  Design: persistent CTAs (two per SM for the
// usual shapes) walk tiles -- TG groups of one query, one contiguous block --
// with a ring of shared-memory stages filled by one-dimensional bulk copies
// (cp.async.bulk + mbarrier complete_tx), ~192 KB in flight per SM.  The keys
// are read once, so their L2 lines are marked first to evict: the stream then
// neither pushes out the scores and quad maxima that selection reads next nor
// keeps dead lines around (measured: ~8% more read bandwidth).  Each
// tile is pooled cooperatively, 16 bytes per thread-item, into a swizzled
// double-buffered pooled tile (one barrier per tile); then thread (g, h) runs
// the D-long FMA chain of head h for group g with q_h in registers, and the H
// head results are summed in order after a warp shuffle gather.
//
// The same kernel scores from a pooled-key cache (the incremental form: the
// pooled key of every complete group kept in device memory, appended as
// groups complete): then a stage holds pooled rows, already in the swizzled
// tile layout (the cache is stored that way), the dots read the stage in
// place, and the stream is G * D * 4 bytes per query instead of T * D * 4.
// There a thread holds two heads of q and runs their chains for H/2 groups
// of the tile, so each 16-byte shared load feeds 8 FMAs.
// pool_groups_kernel fills that cache with the very
// pooling arithmetic of the raw path (pool4 below), so both forms give the
// same scores bit for bit -- the full-raw / incremental identity.
#include "pooling.cuh"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

template <int H, int D, bool kPooled>
struct ScoreCfg {
    // The pooled form moves 4x fewer bytes per group, so FMA latency, not
    // HBM, sets its pace: small CTAs (three per SM) whose threads hold two
    // heads of q (each 16-byte shared load feeds 8 FMAs) and run H
    // independent FMA chains per tile (H/2 groups x 2 heads).
    static constexpr int kThreads = kPooled ? 128 : 256;
    static constexpr int kHPT = kPooled ? 2 : 1;            // heads per thread
    static constexpr int kLPG = H / kHPT;                   // threads (lanes) per group
    static constexpr int kGPT = kPooled ? H / 2 : 1;        // groups per thread per tile
    static constexpr int kTG1 = kThreads / kLPG;            // groups per pass of the CTA
    static constexpr int kTG = kTG1 * kGPT;                 // groups per tile
    static constexpr int kGroupFloats = kPooled ? D : kGroup * D;  // stage floats per group
    static constexpr int kStageFloats = kTG * kGroupFloats;
    static constexpr int kStageBytes = kStageFloats * 4;
    // Raw: two CTAs per SM when a stage is small enough, so that one CTA's
    // barriers and FMA chains overlap the other's; ~96-192 KB of raw keys in
    // flight per SM either way.  Pooled: three CTAs of 64 KB of stages.
    static constexpr int kCtasPerSm = kPooled ? (kStageBytes <= 32768 ? 3 : 1) : (kStageBytes <= 32768 ? 2 : 1);
    static constexpr int kStageBudget = kCtasPerSm == 3 ? 65536 : (kCtasPerSm == 2 ? 98304 : 196608);
    static constexpr int kStagesRaw = kStageBudget / kStageBytes;
    static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
    // one pooled tile (swizzled), double buffered; the pooled form reads its
    // stage directly and needs none
    static constexpr int kPoolFloats = kPooled ? 0 : kTG * D;
    static constexpr size_t kSmem = size_t(kStages) * kStageBytes + 2 * size_t(kPoolFloats) * 4 + kStages * 8;
    static_assert(H % kHPT == 0 && kThreads % kLPG == 0 && 32 % (4 * kLPG) == 0, "a warp holds whole quads of groups");
    static_assert(kTG % 4 == 0, "tiles start on quad boundaries");
    static_assert(D % 32 == 0, "the pooled-tile swizzle needs D/4 to be a multiple of 8");
    static_assert(kSmem <= 232448, "shared memory per CTA");
};


// Per-query values a thread needs, reloaded only when the query changes.
struct QueryCache {
    int b = -1;
    int G = 0;
};

__device__ __forceinline__ int groups_of(const ScoreArgs &a, int b, QueryCache &qc)
{
    if (b != qc.b) {
        const int T = __ldg(a.visible + b);
        qc.b = b;
        qc.G = (T < 0 || T > a.max_visible) ? 0 : (T >> 2);
    }
    return qc.G;
}

struct TileRef {
    int b;      // query
    int g0;     // first group of the tile
    int n;      // valid groups in the tile
};

// Next tile t' >= t (below `end`) that holds at least one group.
template <int TG>
__device__ __forceinline__ int next_tile(const ScoreArgs &a, int t, int end, int tiles_per_q,
                                         QueryCache &qc, TileRef &ref)
{
    for (; t < end; ++t) {
        const int b = t / tiles_per_q;
        const int g0 = (t - b * tiles_per_q) * TG;
        const int G = groups_of(a, b, qc);
        if (g0 < G) {
            ref.b = b;
            ref.g0 = g0;
            ref.n = min(TG, G - g0);
            return t;
        }
    }
    return end;
}

// The tile range of a CTA of a cooperative raw-key launch (kCtas per SM on
// every SM): the share of this SM, by its weight, halved between its CTAs,
// which tell themselves apart by a counter.  Without complete weights (the
// first launch, another GPU size) the equal range passed in stays.  The
// shares cover the tiles exactly when a launch runs on the SMs whose times
// were recorded -- every SM of the GPU, for a process that has the whole
// device; a cooperative launch the runtime refuses as too large (part of the
// GPU is not this process's) falls back to equal shares.  Writes begin, end
// and the slot the CTA records its time in (-1: none).
template <int kCtas>
__device__ void balanced_range(ScoreBalance *bl, int total, int begin, int end, int *out)
{
    uint32_t smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    int slot = -1;
    if (smid < uint32_t(kBalSlots)) {
        const uint32_t magic = __ldcg(&bl->magic), nsm = __ldcg(&bl->nsm), wt = __ldcg(&bl->w_total);
        const uint32_t wb = __ldcg(&bl->w_before[smid]), ws = __ldcg(&bl->w[smid]);
        const uint32_t sub = atomicAdd(&bl->ctr[smid], 1u) % uint32_t(kCtas);
        slot = int(smid) * 2 + int(sub);
        if (magic == kBalMagic && nsm * kCtas == gridDim.x && ws > 0 && wt > 0 && wb + ws <= wt) {
            const uint64_t den = uint64_t(kCtas) * wt;
            const uint64_t u0 = uint64_t(kCtas) * wb + uint64_t(sub) * ws;
            end = int(min(uint64_t(total), (uint64_t(total) * (u0 + ws)) / den));
            begin = int(min(uint64_t(end), (uint64_t(total) * u0) / den));
        }
    }
    out[0] = begin;
    out[1] = end;
    out[2] = slot;
}

template <int H, int D, bool kPooled>
__global__ void __launch_bounds__(ScoreCfg<H, D, kPooled>::kThreads, ScoreCfg<H, D, kPooled>::kCtasPerSm)
score_groups_kernel(const ScoreArgs a, const int tiles_per_q)
{
    using C = ScoreCfg<H, D, kPooled>;
    constexpr int F4 = D / 4;
    extern __shared__ __align__(128) unsigned char smem[];
    float *stages = reinterpret_cast<float *>(smem);
    float *pooled = reinterpret_cast<float *>(smem + size_t(C::kStages) * C::kStageBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + size_t(C::kStages) * C::kStageBytes +
                                                  2 * size_t(C::kPoolFloats) * 4);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int hl = tid % C::kLPG;  // lane within the group: heads hl * kHPT .. + kHPT - 1
    const int gl = tid / C::kLPG;  // group within the tile
    // Each CTA walks one contiguous range of tiles: it meets at most a couple
    // of queries (few reloads of q) and streams its keys sequentially.
    const int total = a.batch * tiles_per_q;
    int t_begin = int((int64_t(total) * blockIdx.x) / gridDim.x);
    int t_end = int((int64_t(total) * (blockIdx.x + 1)) / gridDim.x);
    // a cooperative raw-key launch: the range comes from the per-SM weights
    constexpr bool kBal = !kPooled && C::kCtasPerSm <= 2;
    const bool bal = kBal && a.bal_coop != 0;
    __shared__ int s_bal[3];
    const uint64_t t_start = global_timer_ns();

    allow_successor_launch();  // selection CTAs fill SMs as this grid's CTAs retire
    // The pooled form may be launched while the kernel before it (the append
    // of new groups to the cache) finishes: wait for it before any input.
    if constexpr (kPooled) wait_for_predecessor();
    if (blockIdx.x == 0) {
        for (int b = tid; b < a.batch; b += blockDim.x) {
            const int T = __ldg(a.visible + b);
            if (T < 0 || T > a.max_visible) set_error(a.err, QSA_DEVERR_VISIBLE_RANGE);
        }
    }
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
        if (bal) balanced_range<C::kCtasPerSm>(a.bal, total, t_begin, t_end, s_bal);
    }
    __syncthreads();
    if (bal) {
        t_begin = s_bal[0];
        t_end = s_bal[1];
    }

    // Producer state lives in thread 0: the next tile to issue.
    int t_issue = t_begin;
    int n_issued = 0;
    QueryCache qc_issue;
    int64_t koff_b = -1, koff = 0;
    const uint64_t policy = l2_evict_first_policy();
    auto issue = [&](int stage) {
        TileRef r;
        t_issue = next_tile<C::kTG>(a, t_issue, t_end, tiles_per_q, qc_issue, r);
        if (t_issue >= t_end) return;
        if (r.b != koff_b) {
            koff = __ldg((kPooled ? a.pool_offset : a.key_offset) + r.b);
            koff_b = r.b;
        }
        const float *src = kPooled ? a.pooled + (koff + int64_t(r.g0)) * D
                                   : a.idx_keys + (koff + int64_t(r.g0) * kGroup) * D;
        const uint32_t bytes = uint32_t(r.n) * C::kGroupFloats * 4u;
        mbar_arrive_expect_tx(&full[stage], bytes);
        bulk_copy_g2s_hint(stages + size_t(stage) * C::kStageFloats, src, bytes, &full[stage], policy);
        ++t_issue;
        ++n_issued;
    };
    if (tid == 0 && !a.no_issue)
        for (int s = 0; s < C::kStages; ++s) issue(s);

    float qreg[C::kHPT][D];
    int cur_b = -1;
    QueryCache qc;
    int t_cons = t_begin;
    int it = 0;
    bool timed_out = false;

    while (true) {
        TileRef r;
        t_cons = next_tile<C::kTG>(a, t_cons, t_end, tiles_per_q, qc, r);
        if (t_cons >= t_end) break;
        const int s = it % C::kStages;
        const uint32_t parity = uint32_t(it / C::kStages) & 1u;
        float *pool = pooled + (it & 1) * C::kPoolFloats;

        if (r.b != cur_b) {
#pragma unroll
            for (int u = 0; u < C::kHPT; ++u) {
                const float4 *qp =
                    reinterpret_cast<const float4 *>(a.q_idx + (int64_t(r.b) * H + hl * C::kHPT + u) * D);
#pragma unroll
                for (int j4 = 0; j4 < F4; ++j4) {
                    const float4 v = __ldg(qp + j4);
                    qreg[u][4 * j4 + 0] = v.x;
                    qreg[u][4 * j4 + 1] = v.y;
                    qreg[u][4 * j4 + 2] = v.z;
                    qreg[u][4 * j4 + 3] = v.w;
                }
            }
            cur_b = r.b;
        }

        const bool ok = mbar_wait_bounded(&full[s], parity, a.wait_ns != 0 ? a.wait_ns : kWaitLimitNs);

        if constexpr (!kPooled) {
            // Pool, 16 bytes per item: item e is (group e / F4, chunk e % F4).
            const float4 *raw = reinterpret_cast<const float4 *>(stages + size_t(s) * C::kStageFloats);
            for (int e = tid; e < r.n * F4; e += C::kThreads) {
                const int g = e / F4;
                const int j4 = e - g * F4;
                const float4 *k = raw + g * (kGroup * F4) + j4;
                *reinterpret_cast<float4 *>(pool + pool_index<D>(g, j4)) = pool4(k[0], k[F4], k[2 * F4], k[3 * F4]);
            }
            // One barrier per tile: the pooled tile is ready and raw stage s is
            // consumed.  (The pooled tile is double buffered, so the next tile's
            // pooling cannot overwrite what slower threads still read.)
            if (__syncthreads_or(!ok)) {
                timed_out = true;
                break;
            }
            if (tid == 0 && !a.no_issue) issue(s);  // refill stage s with the tile kStages ahead
        }
        // (the pooled form reads its stage in place: one barrier per tile,
        // after the dots, settles a timed-out wait and frees the stage)

        // Dots: groups gl + kTG1 * i of the tile, i < kGPT, times this
        // thread's kHPT heads, each a D-long chain.
        const float *tile = kPooled ? stages + size_t(s) * C::kStageFloats : pool;
        // The kGPT x kHPT chains advance side by side (independent FMAs to
        // overlap); rows past the tile's end compute from stale shared memory
        // and are dropped below.
        float acc[C::kGPT][C::kHPT];
#pragma unroll
        for (int i = 0; i < C::kGPT; ++i)
#pragma unroll
            for (int u = 0; u < C::kHPT; ++u) acc[i][u] = 0.0f;
#pragma unroll
        for (int j4 = 0; j4 < F4; ++j4) {
            float4 pv[C::kGPT];
#pragma unroll
            for (int i = 0; i < C::kGPT; ++i)
                pv[i] = *reinterpret_cast<const float4 *>(tile + pool_index<D>(gl + C::kTG1 * i, j4));
#pragma unroll
            for (int i = 0; i < C::kGPT; ++i)
#pragma unroll
                for (int u = 0; u < C::kHPT; ++u) {
                    acc[i][u] = __fmaf_rn(qreg[u][4 * j4 + 0], pv[i].x, acc[i][u]);
                    acc[i][u] = __fmaf_rn(qreg[u][4 * j4 + 1], pv[i].y, acc[i][u]);
                    acc[i][u] = __fmaf_rn(qreg[u][4 * j4 + 2], pv[i].z, acc[i][u]);
                    acc[i][u] = __fmaf_rn(qreg[u][4 * j4 + 3], pv[i].w, acc[i][u]);
                }
        }
        float relu[C::kGPT][C::kHPT];
#pragma unroll
        for (int i = 0; i < C::kGPT; ++i)
#pragma unroll
            for (int u = 0; u < C::kHPT; ++u)
                relu[i][u] = (ok && gl + C::kTG1 * i < r.n && acc[i][u] > 0.0f) ? acc[i][u] : 0.0f;
        if constexpr (kPooled) {
            // the stage has been read by every thread: refill it
            if (__syncthreads_or(!ok)) {
                timed_out = true;
                break;
            }
            if (tid == 0 && !a.no_issue) issue(s);
        }
        const int base = lane & ~(C::kLPG - 1);
#pragma unroll
        for (int i = 0; i < C::kGPT; ++i) {
            const int g = gl + C::kTG1 * i;
            // Head sum, h = 0..H-1 in order, gathered from the kLPG lanes of the
            // group (head h is component h % kHPT of lane h / kHPT).
            float hv[H];
#pragma unroll
            for (int hh = 0; hh < H; ++hh)
                hv[hh] = __shfl_sync(0xffffffffu, relu[i][hh % C::kHPT], base + hh / C::kHPT);
            float sum = 0.0f;
#pragma unroll
            for (int hh = 0; hh < H; ++hh) sum = __fadd_rn(sum, hv[hh]);
            if (hl == 0 && g < r.n) a.scores[int64_t(r.b) * a.score_stride + r.g0 + g] = sum;
            // Selection hint: the largest key among groups 4j..4j+3 (the
            // kLPG-lane blocks of those four groups sit side by side in the warp).
            uint32_t qk = (g < r.n) ? order_key(sum) : 0u;
            qk = max(qk, __shfl_xor_sync(0xffffffffu, qk, C::kLPG));
            qk = max(qk, __shfl_xor_sync(0xffffffffu, qk, 2 * C::kLPG));
            if ((lane & (4 * C::kLPG - 1)) == 0 && g < r.n)
                a.qmax[int64_t(r.b) * a.qmax_stride + ((r.g0 + g) >> 2)] = qk;
        }

        ++t_cons;
        ++it;
    }

    // this CTA's time, for the next launch's weights (a launch whose waits ran
    // out measured nothing about the SM's speed)
    if (bal && tid == 0 && s_bal[2] >= 0 && !timed_out) {
        const uint64_t dt = global_timer_ns() - t_start;
        a.bal->el_ns[s_bal[2] >> 1][s_bal[2] & 1] = uint32_t(dt < 0xffffffffull ? dt : 0xffffffffull);
        a.bal->tiles[s_bal[2] >> 1][s_bal[2] & 1] = uint32_t(t_end - t_begin);
    }
    if (timed_out && tid == 0) {
        set_error(a.err, QSA_DEVERR_WAIT_TIMEOUT);
        // Let every copy still in flight land (bounded) before the CTA exits.
        for (int i = it; i < n_issued; ++i)
            (void)mbar_wait_bounded(&full[i % C::kStages], uint32_t(i / C::kStages) & 1u, kDrainLimitNs);
    }
}

template <int H, int D, bool kPooled>
cudaError_t launch_score_t(const ScoreArgs &a, int num_sms, cudaStream_t s)
{
    using C = ScoreCfg<H, D, kPooled>;
    const int gmax = a.max_visible / kGroup;
    const int tiles_per_q = (gmax + C::kTG - 1) / C::kTG;
    const long long total = (long long)a.batch * tiles_per_q;
    if (total == 0) return cudaSuccess;
    if (total > 0x7fffffffLL) return cudaErrorInvalidValue;
    static int resident[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (resident[dev] == 0) {
        cudaError_t e = cudaFuncSetAttribute(score_groups_kernel<H, D, kPooled>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kSmem));
        if (e != cudaSuccess) return e;
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, score_groups_kernel<H, D, kPooled>, C::kThreads, C::kSmem);
        if (e != cudaSuccess) return e;
        resident[dev] = per_sm > 0 ? per_sm : 1;
    }
    const long long slots = (long long)num_sms * resident[dev];
    const int grid = int(total < slots ? total : slots);
    ScoreArgs ab = a;
    ab.bal_coop = 0;
    if (!kPooled && C::kCtasPerSm <= 2 && a.bal != nullptr && grid == slots) {
        // every SM gets exactly its resident CTAs: a cooperative launch (all
        // CTAs resident at once), so ranges by SM cover the tiles exactly
        ab.bal_coop = 1;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(unsigned(grid));
        cfg.blockDim = dim3(C::kThreads);
        cfg.dynamicSmemBytes = C::kSmem;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        const cudaError_t e = cudaLaunchKernelEx(&cfg, score_groups_kernel<H, D, kPooled>, ab, tiles_per_q);
        if (e != cudaErrorCooperativeLaunchTooLarge) return e;
        // not every SM is ours (e.g. a partitioned GPU): equal shares, ordinary launch
        (void)cudaGetLastError();
        ab.bal_coop = 0;
    }
    if constexpr (kPooled)  // its launch overlaps the tail of the kernel before it
        return launch_kernel(score_groups_kernel<H, D, kPooled>, dim3(unsigned(grid)), dim3(C::kThreads), C::kSmem, s,
                             true, ab, tiles_per_q);
    score_groups_kernel<H, D, kPooled><<<grid, C::kThreads, C::kSmem, s>>>(ab, tiles_per_q);
    return cudaGetLastError();
}


// ---- the pooled-key cache ------------------------------------------------------

constexpr int kPoolThreads = 256;
constexpr int kPoolGroupsPerCta = 64;

// pooled[pool_offset[b] + g] = pool of raw rows key_offset[b] + 4g .. 4g+3,
// for g in [group_begin[b], group_end[b]).  One 16-byte chunk per thread-item;
// the row is stored in the pooled-tile layout (chunk j4 at j4 ^ (g & 7)), so a
// bulk copy of whole rows lands in shared memory ready for conflict-free reads.
template <int D>
__global__ void __launch_bounds__(kPoolThreads)
pool_groups_kernel(const PoolArgs a)
{
    constexpr int F4 = D / 4;
    allow_successor_launch();  // a scorer launched after this append may start its launch now
    const int b = blockIdx.y;
    const int g_begin = __ldg(a.group_begin + b), g_end = __ldg(a.group_end + b);
    if (g_begin < 0 || g_end < g_begin || g_end > a.g_max || g_end - g_begin > a.max_groups) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_error(a.err, QSA_DEVERR_VISIBLE_RANGE);
        return;
    }
    const int g_lo = g_begin + int(blockIdx.x) * kPoolGroupsPerCta;
    const int g_hi = min(g_end, g_lo + kPoolGroupsPerCta);
    if (g_lo >= g_hi) return;
    const float4 *keys = reinterpret_cast<const float4 *>(a.idx_keys + __ldg(a.key_offset + b) * D);
    float4 *out = reinterpret_cast<float4 *>(a.pooled + __ldg(a.pool_offset + b) * D);
    for (int e = threadIdx.x; e < (g_hi - g_lo) * F4; e += kPoolThreads) {
        const int g = g_lo + e / F4;
        const int j4 = e % F4;
        const float4 *k = keys + int64_t(g) * (kGroup * F4) + j4;
        out[int64_t(g) * F4 + (j4 ^ (g & 7))] = pool4(__ldg(k), __ldg(k + F4), __ldg(k + 2 * F4), __ldg(k + 3 * F4));
    }
}

}  // namespace

bool score_shape_supported(int idx_heads, int idx_dim)
{
    return (idx_heads == 4 || idx_heads == 8) && (idx_dim == 32 || idx_dim == 64);
}

cudaError_t launch_score(const ScoreArgs &a, int num_sms, cudaStream_t s)
{
    const bool pooled = a.pooled != nullptr;
    if (a.idx_heads == 8 && a.idx_dim == 64)
        return pooled ? launch_score_t<8, 64, true>(a, num_sms, s) : launch_score_t<8, 64, false>(a, num_sms, s);
    if (a.idx_heads == 4 && a.idx_dim == 32)
        return pooled ? launch_score_t<4, 32, true>(a, num_sms, s) : launch_score_t<4, 32, false>(a, num_sms, s);
    if (a.idx_heads == 8 && a.idx_dim == 32)
        return pooled ? launch_score_t<8, 32, true>(a, num_sms, s) : launch_score_t<8, 32, false>(a, num_sms, s);
    if (a.idx_heads == 4 && a.idx_dim == 64)
        return pooled ? launch_score_t<4, 64, true>(a, num_sms, s) : launch_score_t<4, 64, false>(a, num_sms, s);
    return cudaErrorInvalidValue;
}

cudaError_t launch_pool(const PoolArgs &a, cudaStream_t s)
{
    if (a.batch == 0 || a.max_groups == 0) return cudaSuccess;
    const dim3 grid(unsigned((a.max_groups + kPoolGroupsPerCta - 1) / kPoolGroupsPerCta), unsigned(a.batch));
    if (a.idx_dim == 64) pool_groups_kernel<64><<<grid, kPoolThreads, 0, s>>>(a);
    else if (a.idx_dim == 32) pool_groups_kernel<32><<<grid, kPoolThreads, 0, s>>>(a);
    else return cudaErrorInvalidValue;
    return cudaGetLastError();
}

}  // namespace qsa
