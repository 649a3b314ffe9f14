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
// the stage turns from a byte stream into FFMA work.  CTA (range r, query block
// qb) takes kQPC queries and one contiguous range of 32-group tiles.
//
// The FMA chains are cut into D/16 segments of 16 dims and run as a systolic
// pipeline across the lanes of a warp: lane (seg, slot) holds q for all H
// heads of one query restricted to dims 16*seg .. 16*seg+15 (16*H registers),
// applies each pooled value it loads to every head, and hands its H running
// sums to the lane of the next segment by a shuffle; at step t segment seg
// works on group t - seg of the tile, and the last segment's lane finishes
// the ordered head sum on its own.  The chain order over j is unchanged --
// the running sum just moves between lanes -- and one 16-byte shared-memory
// load feeds 4*H FMAs instead of 4.  (With H = 8 a CTA of 8 warps takes most
// of an SM's registers: one CTA per SM.)
#include "pooling.cuh"
#include "qsa_internal.cuh"

namespace qsa {
namespace {

template <int H, int D>
struct SharedCfg {
    static constexpr int kThreads = 256;
    static constexpr int kWarps = kThreads / 32;
    static constexpr int kSeg = D / 16;               // chain segments of 16 dims
    static constexpr int kSlots = 32 / kSeg;          // lanes per segment
    static constexpr int kHPS = H;                    // heads held by a lane: all of them
    static constexpr int kCtasPerSm = kHPS * 16 > 64 ? 1 : 2;  // q takes kHPS x 16 registers
    static constexpr int kSlotsPerQ = H / kHPS;       // lanes (per segment) of one query
    static constexpr int kQPW = kSlots / kSlotsPerQ;  // queries per warp
    static constexpr int kQPC = kQPW * kWarps;        // queries per CTA
    static constexpr int kTG = 32;                    // groups per tile
    static constexpr int kStageBytes = kTG * kGroup * D * 4;
    static constexpr int kStages = 98304 / kStageBytes;  // 96 KB of raw keys in flight per CTA
    static constexpr int kPoolFloats = kTG * D;
    static constexpr size_t kSmem =
        size_t(kStages) * kStageBytes + 2 * size_t(kPoolFloats) * 4 + size_t(kStages) * 8;
    static_assert(D % 16 == 0 && kSlotsPerQ == 1, "lane layout: one lane per (segment, query)");
    static_assert(kTG % 4 == 0, "tiles hold whole quads of groups");
};

template <int H, int D>
__global__ void __launch_bounds__(SharedCfg<H, D>::kThreads, SharedCfg<H, D>::kCtasPerSm)
score_shared_kernel(const ScoreArgs a, const int n_ranges, const int tiles_total)
{
    using C = SharedCfg<H, D>;
    constexpr int F4 = D / 4;
    extern __shared__ __align__(128) unsigned char smem[];
    float *stages = reinterpret_cast<float *>(smem);
    float *pooled = reinterpret_cast<float *>(smem + size_t(C::kStages) * C::kStageBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + size_t(C::kStages) * C::kStageBytes +
                                                  2 * size_t(C::kPoolFloats) * 4);
    __shared__ int g_need;  // groups any query of this CTA needs

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int seg = lane / C::kSlots, slot = lane % C::kSlots;
    const int qi = slot / C::kSlotsPerQ, hq = slot % C::kSlotsPerQ;
    const int b = int(blockIdx.y) * C::kQPC + warp * C::kQPW + qi;   // this lane's query
    const bool have_q = b < a.batch;

    allow_successor_launch();  // selection CTAs fill SMs as this grid's CTAs retire
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
        g_need = 0;
    }
    __syncthreads();
    // this lane's query: its groups, the shared history check, q for H heads x 16 dims
    int G = 0;
    if (have_q) {
        const int T = __ldg(a.visible + b);
        if (T < 0 || T > a.max_visible) {
            if (blockIdx.x == 0 && seg == 0 && hq == 0) set_error(a.err, QSA_DEVERR_VISIBLE_RANGE);
        } else {
            G = T >> 2;
        }
        if (__ldg(a.key_offset + b) != __ldg(a.key_offset)) {
            if (blockIdx.x == 0 && seg == 0 && hq == 0) set_error(a.err, QSA_DEVERR_NOT_SHARED);
            G = 0;
        }
    }
    atomicMax(&g_need, G);
    float q[C::kHPS][16];
#pragma unroll
    for (int u = 0; u < C::kHPS; ++u) {
        const float4 *qp = reinterpret_cast<const float4 *>(
            a.q_idx + (int64_t(have_q ? b : 0) * H + C::kHPS * hq + u) * D + 16 * seg);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
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
    const int t_begin = int((int64_t(tiles_total) * blockIdx.x) / n_ranges);
    int t_end = int((int64_t(tiles_total) * (blockIdx.x + 1)) / n_ranges);
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

    float acc[C::kHPS];
#pragma unroll
    for (int u = 0; u < C::kHPS; ++u) acc[u] = 0.0f;
    uint32_t qk = 0u;  // quad maximum under way (the writing lane)
    int it = 0;
    bool timed_out = false;
    for (int t = t_begin; t < t_end; ++t, ++it) {
        const int s = it % C::kStages;
        const uint32_t parity = uint32_t(it / C::kStages) & 1u;
        float *pool = pooled + (it & 1) * C::kPoolFloats;
        const int g0 = t * C::kTG;
        const int n = min(C::kTG, gmax - g0);
        const bool ok = mbar_wait_bounded(&full[s], parity, kWaitLimitNs);
        // pool the tile once, for every query of the CTA
        const float4 *raw = reinterpret_cast<const float4 *>(stages + size_t(s) * (C::kStageBytes / 4));
        for (int e = tid; e < n * F4; e += C::kThreads) {
            const int g = e / F4, j4 = e - g * F4;
            const float4 *k = raw + g * (kGroup * F4) + j4;
            *reinterpret_cast<float4 *>(pool + pool_index<D>(g, j4)) = pool4(k[0], k[F4], k[2 * F4], k[3 * F4]);
        }
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        if (tid == 0) issue(s);

        // systolic pass: at step st, segment seg works on group st - seg
        for (int st = 0; st < n + C::kSeg - 1; ++st) {
            float a4[C::kHPS];
#pragma unroll
            for (int u = 0; u < C::kHPS; ++u) {
                a4[u] = __shfl_up_sync(0xffffffffu, acc[u], C::kSlots);  // the previous segment's sums
                if (seg == 0) a4[u] = 0.0f;
            }
            const int g = st - seg;
            if (g >= 0 && g < n) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const float4 p = *reinterpret_cast<const float4 *>(pool + pool_index<D>(g, 4 * seg + i));
#pragma unroll
                    for (int u = 0; u < C::kHPS; ++u) {
                        a4[u] = __fmaf_rn(q[u][4 * i + 0], p.x, a4[u]);
                        a4[u] = __fmaf_rn(q[u][4 * i + 1], p.y, a4[u]);
                        a4[u] = __fmaf_rn(q[u][4 * i + 2], p.z, a4[u]);
                        a4[u] = __fmaf_rn(q[u][4 * i + 3], p.w, a4[u]);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < C::kHPS; ++u) acc[u] = a4[u];
            // last segment: ReLU per head, head sum in order h = 0..H-1 (the
            // lane holds every head of its query)
            float hs = 0.0f;
#pragma unroll
            for (int u = 0; u < C::kHPS; ++u) hs = __fadd_rn(hs, a4[u] > 0.0f ? a4[u] : 0.0f);
            const int gg = g0 + g;
            if (seg == C::kSeg - 1 && hq == C::kSlotsPerQ - 1 && g >= 0 && g < n && gg < G) {
                a.scores[int64_t(b) * a.score_stride + gg] = hs;
                const uint32_t key = order_key(hs);
                qk = (gg & 3) == 0 ? key : max(qk, key);
                if ((gg & 3) == 3 || gg == G - 1) a.qmax[int64_t(b) * a.qmax_stride + (gg >> 2)] = qk;
            }
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
    const int qblocks = (a.batch + C::kQPC - 1) / C::kQPC;
    if (qblocks > 65535) return cudaErrorInvalidValue;
    int ranges = (C::kCtasPerSm * num_sms) / qblocks;
    if (ranges < 1) ranges = 1;
    if (ranges > tiles_total) ranges = tiles_total;
    score_shared_kernel<H, D><<<dim3(unsigned(ranges), unsigned(qblocks)), C::kThreads, C::kSmem, s>>>(
        a, ranges, tiles_total);
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
