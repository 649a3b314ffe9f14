// score_shared.cu -- stage 1 for a batch of queries that read one shared key
// history (a chunked prefill: consecutive positions of one sequence).
//
// "A sparse mask is not sparse attention" (AFN-016), Why a sparse mask can
// still be dense: every query scores every complete group of its history,
// s = sum over h of ReLU(q_h . pooled key), the same binary32 order as the
// per-query scorer (pool: ((k0+k1)+k2)+k3 then x0.25; dot: an fma chain over
// j = 0..D-1 from +0; head sum h = 0..H-1 from +0), so the scores are those of
// independent single-query decodes bit for bit ("Top-k chooses the set; time
// chooses the order" (AFN-017): chunk = decode).
//
// Queries that share the history share its pooled keys, so a tile of keys is
// streamed and pooled once per CTA and then used by all of the CTA's queries:
// the stage turns from a byte stream into FFMA work.  A CTA takes the kQPC
// queries of one query block and one contiguous range of 32-group tiles; the
// query blocks get CTAs in proportion to their queries (the last block may be
// partial), so every CTA does about the same number of (query, tile) pairs.
//
// Lane layout: one lane per query.  A warp holds two heads of its 32
// queries over all D dims (2*D registers of q per lane), so every FMA chain
// j = 0..D-1 runs inside one lane and nothing is handed between lanes; each
// 16-byte pooled load is the same address for the whole warp (a broadcast)
// and feeds 8 FMAs per lane.  A lane runs 8 groups at once (16 independent
// chains).  Eight warps per SM: the shared-memory pipe, not the warp count,
// is the limit (12 warps at 168 registers measured slower).  The H/2 warps of a 32-query block each leave ReLU(dot) of their
// two heads in shared memory; after a barrier, a second pass (lane = group)
// sums the H values of each (query, group) in order h = 0..H-1 from +0 and
// stores the tile's scores and quad maxima with coalesced writes.
#include "pooling.cuh"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

template <int H, int D>
struct SharedCfg {
    static constexpr int kThreads = 256;
    static constexpr int kWarps = kThreads / 32;
    static constexpr int kHPW = 2;                     // heads held by a lane (the warp's head pair)
    static constexpr int kWarpsPerBlock = H / kHPW;    // warps of one 32-query block
    static constexpr int kBlocks = kWarps / kWarpsPerBlock;
    static constexpr int kQPC = 32 * kBlocks;          // queries per CTA
    static constexpr int kGI = 8;                      // groups a lane runs at once
    static constexpr int kTG = 32;                     // groups per tile
    static constexpr int kStageBytes = kTG * kGroup * D * 4;
    static constexpr int kStages = 98304 / kStageBytes;  // 96 KB of raw keys in flight per CTA
    static constexpr int kPoolFloats = kTG * D;        // pooled tile, plain rows (read by broadcast)
    static constexpr int kRStride = kTG + 1;           // rl[(h * kQPC + ql) * kRStride + g]: both passes conflict-free
    static constexpr int kRFloats = H * kQPC * kRStride;
    static constexpr size_t kSmem = size_t(kStages) * kStageBytes + size_t(kPoolFloats) * 4 +
                                    size_t(kRFloats) * 4 + size_t(kStages) * 8;
    static_assert(H % kHPW == 0 && kWarps % kWarpsPerBlock == 0, "whole head pairs, whole blocks");
    static_assert(kTG % kGI == 0 && kTG == 32, "a tile is one warp wide (second pass: lane = group)");
    static_assert(kSmem <= 227 * 1024, "shared memory per CTA");
};

// First CTA of query block i when n_ctas CTAs are dealt to the blocks in
// proportion to their queries.
template <int kQPC>
__host__ __device__ __forceinline__ int block_cta_start(int i, int n_ctas, int batch)
{
    const int64_t qi = min(int64_t(i) * kQPC, int64_t(batch));
    return int((int64_t(n_ctas) * qi) / batch);
}

template <int H, int D>
__global__ void __launch_bounds__(SharedCfg<H, D>::kThreads, 1)
score_shared_kernel(const ScoreArgs a, const int tiles_total)
{
    using C = SharedCfg<H, D>;
    constexpr int F4 = D / 4;
    extern __shared__ __align__(128) unsigned char smem[];
    float *stages = reinterpret_cast<float *>(smem);
    float *pooled = reinterpret_cast<float *>(smem + size_t(C::kStages) * C::kStageBytes);
    float *rl = pooled + C::kPoolFloats;  // ReLU(dot) of the current tile
    uint64_t *full = reinterpret_cast<uint64_t *>(rl + C::kRFloats);
    __shared__ int g_need;       // groups any query of this CTA needs
    __shared__ int s_G[C::kQPC];  // groups of each query of the CTA (0: none or flagged)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int blk = warp / C::kWarpsPerBlock, hp = warp % C::kWarpsPerBlock;
    // this CTA's query block qb (the last block whose first CTA is <= blockIdx.x) and range
    const int n_ctas = int(gridDim.x), qblocks = (a.batch + C::kQPC - 1) / C::kQPC;
    int qb = 0;
    for (int lo = 0, hi = qblocks - 1; lo <= hi;) {
        const int mid = (lo + hi) >> 1;
        if (block_cta_start<C::kQPC>(mid, n_ctas, a.batch) <= int(blockIdx.x)) {
            qb = mid;
            lo = mid + 1;
        } else {
            hi = mid - 1;
        }
    }
    const int r0 = block_cta_start<C::kQPC>(qb, n_ctas, a.batch);
    const int n_ranges = block_cta_start<C::kQPC>(qb + 1, n_ctas, a.batch) - r0;
    const int range = int(blockIdx.x) - r0;
    const int ql = blk * 32 + lane;                 // this lane's query within the CTA
    const int q0 = qb * C::kQPC;                    // the block's first query
    const int b = q0 + ql;
    const bool have_q = b < a.batch;
    const bool blk_live = q0 + blk * 32 < a.batch;  // (uniform per warp)

    allow_successor_launch();  // selection CTAs fill SMs as this grid's CTAs retire
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
        g_need = 0;
    }
    __syncthreads();
    // this lane's query: its groups, the shared history check, q for its two heads
    int G = 0;
    if (have_q) {
        const int T = __ldg(a.visible + b);
        if (T < 0 || T > a.max_visible) {
            if (range == 0 && hp == 0) set_error(a.err, QSA_DEVERR_VISIBLE_RANGE);
        } else {
            G = T >> 2;
        }
        if (__ldg(a.key_offset + b) != __ldg(a.key_offset)) {
            if (range == 0 && hp == 0) set_error(a.err, QSA_DEVERR_NOT_SHARED);
            G = 0;
        }
    }
    if (hp == 0) s_G[ql] = G;
    atomicMax(&g_need, G);
    float q[C::kHPW][D];
#pragma unroll
    for (int u = 0; u < C::kHPW; ++u) {
        const float4 *qp =
            reinterpret_cast<const float4 *>(a.q_idx + (int64_t(have_q ? b : 0) * H + C::kHPW * hp + u) * D);
#pragma unroll
        for (int i = 0; i < F4; ++i) {
            const float4 v = have_q ? __ldg(qp + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            q[u][4 * i + 0] = v.x;
            q[u][4 * i + 1] = v.y;
            q[u][4 * i + 2] = v.z;
            q[u][4 * i + 3] = v.w;
        }
    }
    __syncthreads();
    const int gmax = g_need;

    // tiles of this range that some query of the CTA needs
    const int t_begin = int((int64_t(tiles_total) * range) / n_ranges);
    int t_end = int((int64_t(tiles_total) * (range + 1)) / n_ranges);
    t_end = min(t_end, (gmax + C::kTG - 1) / C::kTG);
    const float *keys = a.idx_keys + __ldg(a.key_offset) * D;
    const uint64_t policy = l2_evict_first_policy();

    int t_issue = t_begin, n_issued = 0;
    auto issue = [&](int stage) {
        if (t_issue >= t_end) return;
        const int g0 = t_issue * C::kTG;
        const int n = min(C::kTG, gmax - g0);
        const uint32_t bytes = uint32_t(n) * uint32_t(kGroup * D) * 4u;
        mbar_arrive_expect_tx(&full[stage], bytes);
        bulk_copy_g2s_hint(stages + size_t(stage) * (C::kStageBytes / 4), keys + int64_t(g0) * kGroup * D, bytes,
                           &full[stage], policy);
        ++t_issue;
        ++n_issued;
    };
    if (tid == 0)
        for (int s = 0; s < C::kStages; ++s) issue(s);

    float *my_rl = rl + (C::kHPW * hp * C::kQPC + ql) * C::kRStride;  // head 2*hp, this query, group 0
    int it = 0;
    bool timed_out = false;
    for (int t = t_begin; t < t_end; ++t, ++it) {
        const int s = it % C::kStages;
        const uint32_t parity = uint32_t(it / C::kStages) & 1u;
        const int g0 = t * C::kTG;
        const int n = min(C::kTG, gmax - g0);
        const bool ok = mbar_wait_bounded(&full[s], parity, kWaitLimitNs);
        // pool the tile once, for every query of the CTA
        const float4 *raw = reinterpret_cast<const float4 *>(stages + size_t(s) * (C::kStageBytes / 4));
        for (int e = tid; e < n * F4; e += C::kThreads) {
            const int g = e / F4, j4 = e - g * F4;
            const float4 *k = raw + g * (kGroup * F4) + j4;
            *reinterpret_cast<float4 *>(pooled + g * D + 4 * j4) = pool4(k[0], k[F4], k[2 * F4], k[3 * F4]);
        }
        if (__syncthreads_or(!ok)) {  // (also: the previous tile's second pass is done with rl)
            timed_out = true;
            break;
        }
        if (tid == 0) issue(s);

        // first pass: dot products of this lane's query and two heads with
        // kGI groups at a time (groups past n read stale rows: never stored)
        for (int gb = 0; blk_live && gb < n; gb += C::kGI) {
            float acc[C::kGI][C::kHPW];
#pragma unroll
            for (int gi = 0; gi < C::kGI; ++gi)
#pragma unroll
                for (int u = 0; u < C::kHPW; ++u) acc[gi][u] = 0.0f;
            const float *prow = pooled + gb * D;
#pragma unroll
            for (int j4 = 0; j4 < F4; ++j4) {
                float4 p[C::kGI];
#pragma unroll
                for (int gi = 0; gi < C::kGI; ++gi) p[gi] = *reinterpret_cast<const float4 *>(prow + gi * D + 4 * j4);
#pragma unroll
                for (int gi = 0; gi < C::kGI; ++gi)
#pragma unroll
                    for (int u = 0; u < C::kHPW; ++u) {
                        acc[gi][u] = __fmaf_rn(q[u][4 * j4 + 0], p[gi].x, acc[gi][u]);
                        acc[gi][u] = __fmaf_rn(q[u][4 * j4 + 1], p[gi].y, acc[gi][u]);
                        acc[gi][u] = __fmaf_rn(q[u][4 * j4 + 2], p[gi].z, acc[gi][u]);
                        acc[gi][u] = __fmaf_rn(q[u][4 * j4 + 3], p[gi].w, acc[gi][u]);
                    }
            }
#pragma unroll
            for (int gi = 0; gi < C::kGI; ++gi)
#pragma unroll
                for (int u = 0; u < C::kHPW; ++u)
                    my_rl[u * C::kQPC * C::kRStride + gb + gi] = acc[gi][u] > 0.0f ? acc[gi][u] : 0.0f;
        }
        __syncthreads();

        // second pass: lane = group of the tile; the ordered head sum of each
        // of the CTA's queries, its score and its quad maximum
        const int gg = g0 + lane;
        for (int qq = warp; qq < C::kQPC; qq += C::kWarps) {
            const int bq = q0 + qq;
            if (bq >= a.batch) break;  // (uniform)
            const float *rq = rl + qq * C::kRStride + lane;
            float hs = 0.0f;
#pragma unroll
            for (int h = 0; h < H; ++h) hs = __fadd_rn(hs, rq[h * C::kQPC * C::kRStride]);
            const bool valid = lane < n && gg < s_G[qq];
            if (valid) a.scores[int64_t(bq) * a.score_stride + gg] = hs;
            uint32_t key = valid ? order_key(hs) : 0u;
            key = max(key, __shfl_xor_sync(0xffffffffu, key, 1));
            key = max(key, __shfl_xor_sync(0xffffffffu, key, 2));
            if (valid && (lane & 3) == 0) a.qmax[int64_t(bq) * a.qmax_stride + (gg >> 2)] = key;
        }
    }

    if (timed_out && tid == 0) {
        set_error(a.err, QSA_DEVERR_WAIT_TIMEOUT);
        for (int i = it; i < n_issued; ++i)
            (void)mbar_wait_bounded(&full[i % C::kStages], uint32_t(i / C::kStages) & 1u, kDrainLimitNs);
    }
}

template <int H, int D>
cudaError_t launch_shared_t(const ScoreArgs &a, int num_sms, cudaStream_t s)
{
    using C = SharedCfg<H, D>;
    const int tiles_total = (a.max_visible / kGroup + C::kTG - 1) / C::kTG;
    if (tiles_total == 0) return cudaSuccess;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(score_shared_kernel<H, D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             int(C::kSmem));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    // one CTA per SM, dealt to the query blocks in proportion to their queries
    // (a block gets at least one CTA: more blocks than SMs give one each)
    const int qblocks = (a.batch + C::kQPC - 1) / C::kQPC;
    const int n_ctas = max(qblocks, num_sms);
    score_shared_kernel<H, D><<<unsigned(n_ctas), C::kThreads, C::kSmem, s>>>(a, tiles_total);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_score_shared(const ScoreArgs &a, int num_sms, cudaStream_t s)
{
    if (a.batch == 0) return cudaSuccess;
    if (a.idx_heads == 8 && a.idx_dim == 64) return launch_shared_t<8, 64>(a, num_sms, s);
    if (a.idx_heads == 4 && a.idx_dim == 32) return launch_shared_t<4, 32>(a, num_sms, s);
    if (a.idx_heads == 8 && a.idx_dim == 32) return launch_shared_t<8, 32>(a, num_sms, s);
    if (a.idx_heads == 4 && a.idx_dim == 64) return launch_shared_t<4, 64>(a, num_sms, s);
    return cudaErrorInvalidValue;
}

}  // namespace qsa
