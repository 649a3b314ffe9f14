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
// is bound by HBM bandwidth.  Design: one persistent CTA per SM walks tiles
// (TG groups of one query, contiguous in memory) with a ring of kStages
// shared-memory buffers filled by one-dimensional bulk copies
// (cp.async.bulk + mbarrier complete_tx), so ~160 KB per SM is in flight.
// Each tile is pooled cooperatively into shared memory (coalesced, conflict
// free), then thread (g, h) runs the D-long FMA chain of head h for group g
// with q_h in registers, and the H head results are summed in order through
// warp shuffles.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

template <int H, int D>
struct ScoreCfg {
    static constexpr int kThreads = 256;
    static constexpr int kTG = kThreads / H;                // groups per tile
    static constexpr int kGroupFloats = kGroup * D;         // raw floats per group
    static constexpr int kStageFloats = kTG * kGroupFloats;
    static constexpr int kStageBytes = kStageFloats * 4;
    static constexpr int kStagesRaw = 163840 / kStageBytes;
    static constexpr int kStages = kStagesRaw < 2 ? 2 : (kStagesRaw > 8 ? 8 : kStagesRaw);
    static constexpr int kPoolStride = D + 4;               // floats; keeps float4 rows
                                                            // on distinct banks
    static constexpr size_t kPoolBytes = size_t(kTG) * kPoolStride * 4;
    static constexpr size_t kSmem = size_t(kStages) * kStageBytes + kPoolBytes + kStages * 8;
    static_assert(kThreads % H == 0 && 32 % H == 0, "heads must divide a warp");
    static_assert(D % 4 == 0, "index keys are read as float4");
};

struct TileRef {
    int b;      // query
    int g0;     // first group of the tile
    int n;      // valid groups in the tile (0 = nothing to do)
};

__device__ __forceinline__ int groups_of(const ScoreArgs &a, int b)
{
    const int T = __ldg(a.visible + b);
    return (T < 0 || T > a.max_visible) ? 0 : (T >> 2);
}

// Next tile t' >= t (stepping by `step`) that holds at least one group.
template <int TG>
__device__ __forceinline__ int next_tile(const ScoreArgs &a, int t, int step, int total,
                                         int tiles_per_q, TileRef &ref)
{
    for (; t < total; t += step) {
        const int b = t / tiles_per_q;
        const int g0 = (t - b * tiles_per_q) * TG;
        const int G = groups_of(a, b);
        if (g0 < G) {
            ref.b = b;
            ref.g0 = g0;
            ref.n = min(TG, G - g0);
            return t;
        }
    }
    return total;
}

template <int H, int D>
__global__ void __launch_bounds__(ScoreCfg<H, D>::kThreads, 1)
score_groups_kernel(const ScoreArgs a, const int tiles_per_q)
{
    using C = ScoreCfg<H, D>;
    extern __shared__ __align__(128) unsigned char smem[];
    float *stages = reinterpret_cast<float *>(smem);
    float *pooled = reinterpret_cast<float *>(smem + size_t(C::kStages) * C::kStageBytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + size_t(C::kStages) * C::kStageBytes +
                                                  C::kPoolBytes);

    const int tid = threadIdx.x;
    const int lane = tid & 31;
    const int h = tid % H;       // indexer head of this thread
    const int gl = tid / H;      // group within the tile
    const int total = a.batch * tiles_per_q;
    const int step = gridDim.x;

    if (blockIdx.x == 0) {
        for (int b = tid; b < a.batch; b += blockDim.x) {
            const int T = __ldg(a.visible + b);
            if (T < 0 || T > a.max_visible) set_error(a.err, QSA_DEVERR_VISIBLE_RANGE);
        }
    }
    if (tid == 0) {
        for (int s = 0; s < C::kStages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // Producer state lives in thread 0: the next tile to issue.
    int t_issue = blockIdx.x;
    int n_issued = 0;
    auto issue = [&](int stage) {
        TileRef r;
        t_issue = next_tile<C::kTG>(a, t_issue, step, total, tiles_per_q, r);
        if (t_issue >= total) return;
        const float *src = a.idx_keys + (__ldg(a.key_offset + r.b) + int64_t(r.g0) * kGroup) * D;
        const uint32_t bytes = uint32_t(r.n) * C::kGroupFloats * 4u;
        mbar_arrive_expect_tx(&full[stage], bytes);
        bulk_copy_g2s(stages + size_t(stage) * C::kStageFloats, src, bytes, &full[stage]);
        t_issue += step;
        ++n_issued;
    };
    if (tid == 0)
        for (int s = 0; s < C::kStages; ++s) issue(s);

    float qreg[D];
    int cur_b = -1;
    int t_cons = blockIdx.x;
    int it = 0;
    bool timed_out = false;

    while (true) {
        TileRef r;
        t_cons = next_tile<C::kTG>(a, t_cons, step, total, tiles_per_q, r);
        if (t_cons >= total) break;
        const int s = it % C::kStages;
        const uint32_t parity = uint32_t(it / C::kStages) & 1u;

        if (r.b != cur_b) {
            const float4 *qp = reinterpret_cast<const float4 *>(a.q_idx + (int64_t(r.b) * H + h) * D);
#pragma unroll
            for (int j4 = 0; j4 < D / 4; ++j4) {
                const float4 v = __ldg(qp + j4);
                qreg[4 * j4 + 0] = v.x;
                qreg[4 * j4 + 1] = v.y;
                qreg[4 * j4 + 2] = v.z;
                qreg[4 * j4 + 3] = v.w;
            }
            cur_b = r.b;
        }

        const bool ok = mbar_wait_bounded(&full[s], parity, kWaitLimitNs);

        // Pool: element e of the tile's pooled block is (group e / D, lane e % D).
        const float *raw = stages + size_t(s) * C::kStageFloats;
        for (int e = tid; e < r.n * D; e += C::kThreads) {
            const int g = e / D;
            const int j = e - g * D;
            const float *k = raw + g * C::kGroupFloats + j;
            float acc = k[0];
            acc = __fadd_rn(acc, k[D]);
            acc = __fadd_rn(acc, k[2 * D]);
            acc = __fadd_rn(acc, k[3 * D]);
            pooled[g * C::kPoolStride + j] = __fmul_rn(acc, 0.25f);
        }
        if (__syncthreads_or(!ok)) {
            timed_out = true;
            break;
        }
        // Stage s is free again: refill it with the tile kStages ahead.
        if (tid == 0) issue(s);

        float relu = 0.0f;
        if (gl < r.n) {
            const float *pg = pooled + gl * C::kPoolStride;
            float acc = 0.0f;
#pragma unroll
            for (int j4 = 0; j4 < D / 4; ++j4) {
                const float4 pv = *reinterpret_cast<const float4 *>(pg + 4 * j4);
                acc = __fmaf_rn(qreg[4 * j4 + 0], pv.x, acc);
                acc = __fmaf_rn(qreg[4 * j4 + 1], pv.y, acc);
                acc = __fmaf_rn(qreg[4 * j4 + 2], pv.z, acc);
                acc = __fmaf_rn(qreg[4 * j4 + 3], pv.w, acc);
            }
            relu = acc > 0.0f ? acc : 0.0f;
        }
        // Head sum, h = 0..H-1 in order, gathered from the H lanes of the group.
        const int base = lane & ~(H - 1);
        float sum = 0.0f;
#pragma unroll
        for (int hh = 0; hh < H; ++hh) sum = __fadd_rn(sum, __shfl_sync(0xffffffffu, relu, base + hh));
        if (h == 0 && gl < r.n) a.scores[int64_t(r.b) * a.score_stride + r.g0 + gl] = sum;

        __syncthreads();  // pooled block is rewritten by the next tile
        t_cons += step;
        ++it;
    }

    if (timed_out && tid == 0) {
        set_error(a.err, QSA_DEVERR_WAIT_TIMEOUT);
        // Let every copy still in flight land (bounded) before the CTA exits.
        for (int i = it; i < n_issued; ++i)
            (void)mbar_wait_bounded(&full[i % C::kStages], uint32_t(i / C::kStages) & 1u, kDrainLimitNs);
    }
}

template <int H, int D>
cudaError_t launch_score_t(const ScoreArgs &a, int num_sms, cudaStream_t s)
{
    using C = ScoreCfg<H, D>;
    const int gmax = a.max_visible / kGroup;
    const int tiles_per_q = (gmax + C::kTG - 1) / C::kTG;
    const long long total = (long long)a.batch * tiles_per_q;
    if (total == 0) return cudaSuccess;
    if (total > 0x7fffffffLL) return cudaErrorInvalidValue;
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(score_groups_kernel<H, D>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(C::kSmem));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const int grid = int(total < num_sms ? total : num_sms);
    score_groups_kernel<H, D><<<grid, C::kThreads, C::kSmem, s>>>(a, tiles_per_q);
    return cudaGetLastError();
}

}  // namespace

bool score_shape_supported(int idx_heads, int idx_dim)
{
    return (idx_heads == 4 || idx_heads == 8) && (idx_dim == 32 || idx_dim == 64);
}

cudaError_t launch_score(const ScoreArgs &a, int num_sms, cudaStream_t s)
{
    if (a.idx_heads == 8 && a.idx_dim == 64) return launch_score_t<8, 64>(a, num_sms, s);
    if (a.idx_heads == 4 && a.idx_dim == 32) return launch_score_t<4, 32>(a, num_sms, s);
    if (a.idx_heads == 8 && a.idx_dim == 32) return launch_score_t<8, 32>(a, num_sms, s);
    if (a.idx_heads == 4 && a.idx_dim == 64) return launch_score_t<4, 64>(a, num_sms, s);
    return cudaErrorInvalidValue;
}

}  // namespace qsa
