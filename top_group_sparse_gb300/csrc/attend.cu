// attend.cu -- stage 4: online softmax over the compact row.
//
// "Top-k chooses the set; time chooses the order" (AFN-017), Floating point
// makes order observable: a real online softmax is a sequence of rounded
// max / rescale / exp / denominator / accumulator updates, so one canonical
// visit order is needed -- the emitted, chronological one.  "A sparse mask is
// not sparse attention" (AFN-016), Decision: online softmax over at most
// 2,051 gathered rows.
//
// GPU order (fixed, documented, batch independent): the emitted row of query
// b is cut into chunks of kAttendChunk consecutive rows.  One CTA per (chunk,
// KV head, query) loads its rows of K and V from scratch into shared memory
// and, for each of the n_q/n_kv query heads sharing that KV head, computes the
// chunk's scaled scores, the chunk max m_c, p_i = exp(x_i - m_c),
// l_c = sum p_i (fixed tree), acc_c = sum_i p_i v_i (rows in order).  The
// last CTA of a (query, KV head) -- found with an atomic ticket, no waiting --
// merges the chunk partials in ascending chunk order:
//   M = max m_c,  L = sum l_c e^(m_c - M),  out = sum acc_c e^(m_c - M) / L.
// The split depends only on n_ids[b], so a query's output is bit-identical
// whatever else is in the batch; there are no floating-point atomics.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 256;
constexpr int kCH = kAttendChunk;

template <int D>
struct AttendSmem {
    static constexpr int kKStride = D + 4;   // float4 rows on distinct banks
    float q[kMaxGqa][D];
    float k[kCH][kKStride];
    float v[kCH][D];
    float p[kMaxGqa][kCH];
    float m[kMaxGqa];
    float l[kMaxGqa];
    int last;
};

template <int D>
__global__ void __launch_bounds__(kThreads, 2)
attend_kernel(const AttendArgs a)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    AttendSmem<D> &sm = *reinterpret_cast<AttendSmem<D> *>(smem_raw);

    const int c = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = a.q_heads / a.kv_heads;
    const int h0 = kvh * gq;

    const int n = __ldg(a.n_ids + b);
    if (n < 0 || n > a.row_cap) {
        // Bad row length: zero this query's heads of this KV head, flag it.
        if (c == 0) {
            for (int e = tid; e < gq * D; e += kThreads)
                a.out[(int64_t(b) * a.q_heads + h0) * D + e] = 0.0f;
            if (kvh == 0 && tid == 0) set_error(a.err, QSA_DEVERR_ROW_RANGE);
        }
        return;
    }
    const int nch = n > 0 ? (n + kCH - 1) / kCH : 1;
    if (c >= nch) return;
    const int r0 = c * kCH;
    const int rows = min(kCH, n - r0);  // 0 only for an empty row

    // ---- load q heads, K and V rows of this chunk ------------------------------
    constexpr int F4 = D / 4;
    {
        const float4 *qg = reinterpret_cast<const float4 *>(a.q + (int64_t(b) * a.q_heads + h0) * D);
        for (int e = tid; e < gq * F4; e += kThreads) {
            const int hh = e / F4, j4 = e - hh * F4;
            *reinterpret_cast<float4 *>(&sm.q[hh][4 * j4]) = __ldg(qg + e);
        }
        const int64_t row_stride4 = int64_t(a.kv_heads) * F4;  // float4 per scratch row
        const float4 *kg = reinterpret_cast<const float4 *>(a.k_scr) +
                           (int64_t(b) * a.row_cap + r0) * row_stride4 + int64_t(kvh) * F4;
        const float4 *vg = reinterpret_cast<const float4 *>(a.v_scr) +
                           (int64_t(b) * a.row_cap + r0) * row_stride4 + int64_t(kvh) * F4;
        for (int e = tid; e < rows * F4; e += kThreads) {
            const int i = e / F4, j4 = e - i * F4;
            const float4 kv = __ldcs(kg + i * row_stride4 + j4);
            const float4 vv = __ldcs(vg + i * row_stride4 + j4);
            *reinterpret_cast<float4 *>(&sm.k[i][4 * j4]) = kv;
            *reinterpret_cast<float4 *>(&sm.v[i][4 * j4]) = vv;
        }
    }
    __syncthreads();

    // ---- scaled scores x = scale * (q_h . k_i) -------------------------------
    for (int e = tid; e < gq * kCH; e += kThreads) {
        const int hh = e / kCH, i = e - hh * kCH;
        float x = -INFINITY;
        if (i < rows) {
            float dot = 0.0f;
#pragma unroll 8
            for (int j4 = 0; j4 < F4; ++j4) {
                const float4 kv = *reinterpret_cast<const float4 *>(&sm.k[i][4 * j4]);
                const float4 qv = *reinterpret_cast<const float4 *>(&sm.q[hh][4 * j4]);
                dot = fmaf(qv.x, kv.x, dot);
                dot = fmaf(qv.y, kv.y, dot);
                dot = fmaf(qv.z, kv.z, dot);
                dot = fmaf(qv.w, kv.w, dot);
            }
            x = a.scale * dot;
        }
        sm.p[hh][i] = x;
    }
    __syncthreads();

    // ---- chunk max, weights and denominator per head -------------------------
    for (int hh = warp; hh < gq; hh += kThreads / 32) {
        const float x0 = sm.p[hh][lane], x1 = sm.p[hh][lane + 32];
        float m = fmaxf(x0, x1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float p0 = 0.0f, p1 = 0.0f;
        if (m != -INFINITY) {
            p0 = expf(x0 - m);
            p1 = expf(x1 - m);
        }
        sm.p[hh][lane] = p0;
        sm.p[hh][lane + 32] = p1;
        float l = p0 + p1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            sm.m[hh] = m;
            sm.l[hh] = l;
        }
    }
    __syncthreads();

    // ---- acc_c = sum_i p_i v_i, rows in emitted order ------------------------
    const int64_t pbase = (int64_t(b) * a.q_heads + h0) * a.nchunk_max + c;  // head h0, chunk c
    for (int e = tid; e < gq * F4; e += kThreads) {
        const int hh = e / F4, j4 = e - hh * F4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int i = 0; i < rows; ++i) {
            const float p = sm.p[hh][i];
            const float4 v = *reinterpret_cast<const float4 *>(&sm.v[i][4 * j4]);
            acc.x = fmaf(p, v.x, acc.x);
            acc.y = fmaf(p, v.y, acc.y);
            acc.z = fmaf(p, v.z, acc.z);
            acc.w = fmaf(p, v.w, acc.w);
        }
        float4 *dst = reinterpret_cast<float4 *>(a.part_acc + (pbase + int64_t(hh) * a.nchunk_max) * D);
        dst[j4] = acc;
    }
    if (tid < gq) {
        a.part_m[pbase + int64_t(tid) * a.nchunk_max] = sm.m[tid];
        a.part_l[pbase + int64_t(tid) * a.nchunk_max] = sm.l[tid];
    }

    // ---- last CTA of this (query, KV head) merges, ascending chunk order -------
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        uint32_t *ticket = a.tickets + int64_t(b) * a.kv_heads + kvh;
        sm.last = atomicAdd(ticket, 1u) == uint32_t(nch - 1);
        if (sm.last) *ticket = 0u;  // leave the ticket clean for the next call
    }
    __syncthreads();
    if (!sm.last) return;
    __threadfence();

    for (int e = tid; e < gq * D; e += kThreads) {
        const int hh = e / D, j = e - hh * D;
        const int64_t hb = (int64_t(b) * a.q_heads + h0 + hh) * a.nchunk_max;
        float M = -INFINITY;
        for (int cc = 0; cc < nch; ++cc) M = fmaxf(M, __ldcg(a.part_m + hb + cc));
        float L = 0.0f, O = 0.0f;
        if (M != -INFINITY) {
            for (int cc = 0; cc < nch; ++cc) {
                const float w = expf(__ldcg(a.part_m + hb + cc) - M);
                L = fmaf(__ldcg(a.part_l + hb + cc), w, L);
                O = fmaf(__ldcg(a.part_acc + (hb + cc) * D + j), w, O);
            }
        }
        a.out[(int64_t(b) * a.q_heads + h0 + hh) * D + j] = L > 0.0f ? O / L : 0.0f;
    }
}

template <int D>
cudaError_t launch_attend_t(const AttendArgs &a, cudaStream_t s)
{
    const size_t smem = sizeof(AttendSmem<D>);
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(attend_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const dim3 grid(unsigned(a.nchunk_max), unsigned(a.kv_heads), unsigned(a.batch));
    attend_kernel<D><<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool attend_shape_supported(int head_dim, int q_heads, int kv_heads)
{
    if (head_dim != 64 && head_dim != 128) return false;
    if (kv_heads <= 0 || q_heads <= 0 || q_heads % kv_heads != 0) return false;
    return q_heads / kv_heads <= kMaxGqa;
}

cudaError_t launch_attend(const AttendArgs &a, cudaStream_t s)
{
    if (a.batch == 0) return cudaSuccess;
    if (a.head_dim == 128) return launch_attend_t<128>(a, s);
    if (a.head_dim == 64) return launch_attend_t<64>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace qsa
