// attend.cu -- stage 4 (online softmax over the compact row), alone or fused
// with stage 3 (slot resolution and compact gather).
//
// "Top-k chooses the set; time chooses the order" (AFN-017), Floating point
// makes order observable: a real online softmax is a sequence of rounded
// max / rescale / exp / denominator / accumulator updates, so one canonical
// visit order is needed -- the emitted, chronological one.  "A sparse mask is
// not sparse attention" (AFN-016), Decision: online softmax over at most
// 2,051 gathered rows; only the gather crosses from logical identity into the
// physical cache layout, and it copies exactly the selected rows into bounded
// scratch (Why compact gather comes before fusion).
//
// GPU order (fixed, documented, batch independent): the emitted row of query
// b is cut into chunks of kAttendChunk consecutive rows.  One CTA per (chunk,
// KV head, query) brings its K and V rows into shared memory with one
// bulk copy per row (cp.async.bulk, completion on an mbarrier) and, for the
// n_q/n_kv query heads sharing that KV head, computes the chunk's scaled
// scores, the chunk max m_c, p_i = exp(x_i - m_c), l_c = sum p_i (fixed
// tree) and acc_c = sum_i p_i v_i (rows in a fixed order).  The last CTA of a
// (query, KV head) -- found with an atomic ticket, nothing waits -- merges the
// chunk partials in ascending chunk order:
//   M = max m_c,  L = sum l_c e^(m_c - M),  out = sum acc_c e^(m_c - M) / L.
// The split depends only on n_ids[b], so a query's output is bit-identical
// whatever else is in the batch; there are no floating-point atomics.
//
// Row source: kFromCache = false reads the rows from the gathered scratch
// (qsa_attend); kFromCache = true resolves each ID through the slot map,
// copies the row from the K/V cache, and writes it to the scratch with a bulk
// store from shared memory while the attention math runs (qsa_gather_attend,
// qsa_decode) -- the gather's output is the same bytes either way.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 256;
constexpr int kCH = kAttendChunk;
constexpr int kMaxChunks = (4 * QSA_MAX_BUDGET + 3 + kAttendChunk - 1) / kAttendChunk;  // 33
constexpr int kQuarters = kThreads / kCH;                                              // 4

template <int D>
struct AttendSmem {
    static constexpr int kKStride = D + 4;       // float4 rows land on distinct banks
    static constexpr int kPartFloats = 4096;     // 16 KB of partial sums, reused
    float q[kMaxGqa][D];
    float k[kCH][kKStride];
    float v[kCH][D];
    float part[kPartFloats];                     // dot quarters, then P.V row splits
    float x[kMaxGqa][kCH];                       // scaled scores
    float pt[kCH][kMaxGqa];                      // weights, row-major (heads inner)
    float m[kMaxGqa];
    float l[kMaxGqa];
    float w[kMaxGqa][kMaxChunks];                // merge: m_c, then e^(m_c - M)
    float lc[kMaxGqa][kMaxChunks];               // merge: l_c
    float L[kMaxGqa];
    uint64_t bar;
    int last;
};

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void bulk_store_s2g(void *dst, const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

template <int D, bool kFromCache>
__global__ void __launch_bounds__(kThreads, 2)
attend_kernel(const AttendArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    AttendSmem<D> &sm = *reinterpret_cast<AttendSmem<D> *>(smem_raw);
    constexpr int F4 = D / 4;
    constexpr int kRowBytes = D * 4;

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

    if (tid == 0) {
        mbar_init(&sm.bar, kCH);  // one arrival per row thread
        fence_mbar_init();
    }
    __syncthreads();

    // ---- rows into shared memory: one bulk copy per K row and per V row ------
    const int64_t scr_row0 = (int64_t(b) * a.row_cap + r0) * a.kv_heads + kvh;  // scratch row r0, head kvh
    const int64_t scr_rs = a.kv_heads;                                          // rows apart, in D units
    if (tid < kCH) {
        const int i = tid;
        const float *ksrc = nullptr, *vsrc = nullptr;
        if (i < rows) {
            if (kFromCache) {
                const int id = __ldg(a.ids + int64_t(b) * a.row_cap + r0 + i);
                const int T = __ldg(a.visible + b);
                if (id >= 0 && id < T) {
                    const int64_t slot = __ldg(a.slot_map + __ldg(a.slot_offset + b) + id);
                    if (slot >= 0 && slot < a.num_slots) {
                        ksrc = a.k_cache + (slot * a.kv_heads + kvh) * D;
                        vsrc = a.v_cache + (slot * a.kv_heads + kvh) * D;
                    } else {
                        set_error(a.err, QSA_DEVERR_SLOT_RANGE);
                    }
                } else {
                    set_error(a.err, QSA_DEVERR_ROW_RANGE);
                }
            } else {
                ksrc = a.k_scr + (scr_row0 + i * scr_rs) * D;
                vsrc = a.v_scr + (scr_row0 + i * scr_rs) * D;
            }
        }
        if (ksrc != nullptr) {
            mbar_arrive_expect_tx(&sm.bar, 2u * kRowBytes);
            bulk_copy_g2s(&sm.k[i][0], ksrc, kRowBytes, &sm.bar);
            bulk_copy_g2s(&sm.v[i][0], vsrc, kRowBytes, &sm.bar);
        } else {
            if (i < rows) {  // unresolvable row: zeros, flagged above
                for (int j4 = 0; j4 < F4; ++j4) {
                    *reinterpret_cast<float4 *>(&sm.k[i][4 * j4]) = make_float4(0.f, 0.f, 0.f, 0.f);
                    *reinterpret_cast<float4 *>(&sm.v[i][4 * j4]) = make_float4(0.f, 0.f, 0.f, 0.f);
                }
                fence_proxy_async_smem();
            }
            mbar_arrive(&sm.bar);
        }
    }
    {
        const float4 *qg = reinterpret_cast<const float4 *>(a.q + (int64_t(b) * a.q_heads + h0) * D);
        for (int e = tid; e < gq * F4; e += kThreads) {
            const int hh = e / F4, j4 = e - hh * F4;
            *reinterpret_cast<float4 *>(&sm.q[hh][4 * j4]) = __ldg(qg + e);
        }
    }
    const bool landed = mbar_wait_bounded(&sm.bar, 0u, kWaitLimitNs);
    if (__syncthreads_or(!landed)) {
        if (tid == 0) {
            set_error(a.err, QSA_DEVERR_WAIT_TIMEOUT);
            (void)mbar_wait_bounded(&sm.bar, 0u, kDrainLimitNs);
        }
        return;
    }
    if (kFromCache && tid < rows) {
        // the gather's output: this KV head's slice of scratch row r0 + tid
        bulk_store_s2g(a.k_scr_out + (scr_row0 + tid * scr_rs) * D, &sm.k[tid][0], kRowBytes);
        bulk_store_s2g(a.v_scr_out + (scr_row0 + tid * scr_rs) * D, &sm.v[tid][0], kRowBytes);
        bulk_commit();
    }

    // ---- scaled scores: thread = (row, quarter of d); all heads per thread ------
    {
        const int i = tid % kCH;
        const int qd = tid / kCH;
        constexpr int Q4 = F4 / kQuarters;  // float4 per quarter
        float acc[kMaxGqa];
#pragma unroll
        for (int hh = 0; hh < kMaxGqa; ++hh) acc[hh] = 0.0f;
        if (i < rows) {
#pragma unroll
            for (int u = 0; u < Q4; ++u) {
                const int j4 = qd * Q4 + u;
                const float4 kv = *reinterpret_cast<const float4 *>(&sm.k[i][4 * j4]);
#pragma unroll
                for (int hh = 0; hh < kMaxGqa; ++hh) {
                    if (hh < gq) {
                        const float4 qv = *reinterpret_cast<const float4 *>(&sm.q[hh][4 * j4]);
                        acc[hh] = fmaf(qv.x, kv.x, acc[hh]);
                        acc[hh] = fmaf(qv.y, kv.y, acc[hh]);
                        acc[hh] = fmaf(qv.z, kv.z, acc[hh]);
                        acc[hh] = fmaf(qv.w, kv.w, acc[hh]);
                    }
                }
            }
        }
        // part[qd][hh][i]
#pragma unroll
        for (int hh = 0; hh < kMaxGqa; ++hh)
            if (hh < gq) sm.part[(qd * kMaxGqa + hh) * kCH + i] = acc[hh];
    }
    __syncthreads();
    for (int e = tid; e < gq * kCH; e += kThreads) {
        const int hh = e / kCH, i = e - hh * kCH;
        float x = -INFINITY;
        if (i < rows) {
            const float s0 = sm.part[(0 * kMaxGqa + hh) * kCH + i], s1 = sm.part[(1 * kMaxGqa + hh) * kCH + i];
            const float s2 = sm.part[(2 * kMaxGqa + hh) * kCH + i], s3 = sm.part[(3 * kMaxGqa + hh) * kCH + i];
            x = a.scale * ((s0 + s1) + (s2 + s3));
        }
        sm.x[hh][i] = x;
    }
    __syncthreads();

    // ---- chunk max, weights and denominator per head -------------------------
    for (int hh = warp; hh < gq; hh += kThreads / 32) {
        const float x0 = sm.x[hh][lane], x1 = sm.x[hh][lane + 32];
        float m = fmaxf(x0, x1);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        float p0 = 0.0f, p1 = 0.0f;
        if (m != -INFINITY) {
            p0 = expf(x0 - m);
            p1 = expf(x1 - m);
        }
        sm.pt[lane][hh] = p0;
        sm.pt[lane + 32][hh] = p1;
        float l = p0 + p1;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) {
            sm.m[hh] = m;
            sm.l[hh] = l;
        }
    }
    __syncthreads();

    // ---- acc_c = sum_i p_i v_i: thread = (d4, group of 4 heads, row split) --------
    {
        constexpr int kSlots = kThreads / F4;          // 8 (D=128) or 16 (D=64)
        const int hg_n = (gq + 3) / 4;                 // head groups
        const int rs_n = kSlots / hg_n;                // row splits
        const int d4 = tid % F4;
        const int slot = tid / F4;
        const int hg = slot % hg_n;
        const int rs = slot / hg_n;
        if (rs < rs_n) {
            const int rlen = (kCH + rs_n - 1) / rs_n;
            const int i0 = rs * rlen;
            const int i1 = min(rows, i0 + rlen);
            float4 acc[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int i = i0; i < i1; ++i) {
                const float4 vv = *reinterpret_cast<const float4 *>(&sm.v[i][4 * d4]);
                const float4 pp = *reinterpret_cast<const float4 *>(&sm.pt[i][4 * hg]);
                const float pw[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    acc[u].x = fmaf(pw[u], vv.x, acc[u].x);
                    acc[u].y = fmaf(pw[u], vv.y, acc[u].y);
                    acc[u].z = fmaf(pw[u], vv.z, acc[u].z);
                    acc[u].w = fmaf(pw[u], vv.w, acc[u].w);
                }
            }
            // part[rs][hh][d]: rs_n * gq * D <= 4096 floats for every supported shape
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int hh = 4 * hg + u;
                if (hh < gq) *reinterpret_cast<float4 *>(&sm.part[(rs * gq + hh) * D + 4 * d4]) = acc[u];
            }
        }
    }
    __syncthreads();
    const int64_t pbase = (int64_t(b) * a.q_heads + h0) * a.nchunk_max + c;  // head h0, chunk c
    {
        constexpr int kSlots = kThreads / F4;
        const int hg_n = (gq + 3) / 4;
        const int rs_n = kSlots / hg_n;
        for (int e = tid; e < gq * F4; e += kThreads) {
            const int hh = e / F4, j4 = e - hh * F4;
            float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int rs = 0; rs < rs_n; ++rs) {
                const float4 p = *reinterpret_cast<const float4 *>(&sm.part[(rs * gq + hh) * D + 4 * j4]);
                o.x += p.x;
                o.y += p.y;
                o.z += p.z;
                o.w += p.w;
            }
            float4 *dst = reinterpret_cast<float4 *>(a.part_acc + (pbase + int64_t(hh) * a.nchunk_max) * D);
            dst[j4] = o;
        }
    }
    if (tid < gq) {
        a.part_m[pbase + int64_t(tid) * a.nchunk_max] = sm.m[tid];
        a.part_l[pbase + int64_t(tid) * a.nchunk_max] = sm.l[tid];
    }
    if (kFromCache && tid < rows) bulk_wait_all();  // scratch rows written, shared memory free

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

    const int64_t hb0 = (int64_t(b) * a.q_heads + h0) * a.nchunk_max;
    // chunk maxima and denominators of every head, all loads in flight at once
    for (int e = tid; e < gq * nch; e += kThreads) {
        const int hh = e / nch, cc = e - hh * nch;
        sm.w[hh][cc] = __ldcg(a.part_m + hb0 + int64_t(hh) * a.nchunk_max + cc);
        sm.lc[hh][cc] = __ldcg(a.part_l + hb0 + int64_t(hh) * a.nchunk_max + cc);
    }
    __syncthreads();
    // per head: M = max_c m_c, weights e^(m_c - M), L = sum_c l_c w_c (ascending c)
    for (int hh = warp; hh < gq; hh += kThreads / 32) {
        float M = -INFINITY;
        for (int cc = lane; cc < nch; cc += 32) M = fmaxf(M, sm.w[hh][cc]);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
        __syncwarp();
        for (int cc = lane; cc < nch; cc += 32)
            sm.w[hh][cc] = M == -INFINITY ? 0.0f : expf(sm.w[hh][cc] - M);
        __syncwarp();
        if (lane == 0) {
            float L = 0.0f;
            for (int cc = 0; cc < nch; ++cc) L = fmaf(sm.lc[hh][cc], sm.w[hh][cc], L);
            sm.L[hh] = L;
        }
    }
    __syncthreads();
    // out = sum_c acc_c w_c / L, ascending c; independent loads unrolled
    for (int e = tid; e < gq * F4; e += kThreads) {
        const int hh = e / F4, j4 = e - hh * F4;
        const float4 *src =
            reinterpret_cast<const float4 *>(a.part_acc + (hb0 + int64_t(hh) * a.nchunk_max) * D) + j4;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
        int cc = 0;
        for (; cc + 4 <= nch; cc += 4) {
            float4 xv[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) xv[u] = __ldcg(src + int64_t(cc + u) * F4);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float wgt = sm.w[hh][cc + u];
                o.x = fmaf(xv[u].x, wgt, o.x);
                o.y = fmaf(xv[u].y, wgt, o.y);
                o.z = fmaf(xv[u].z, wgt, o.z);
                o.w = fmaf(xv[u].w, wgt, o.w);
            }
        }
        for (; cc < nch; ++cc) {
            const float4 xv = __ldcg(src + int64_t(cc) * F4);
            const float wgt = sm.w[hh][cc];
            o.x = fmaf(xv.x, wgt, o.x);
            o.y = fmaf(xv.y, wgt, o.y);
            o.z = fmaf(xv.z, wgt, o.z);
            o.w = fmaf(xv.w, wgt, o.w);
        }
        const float L = sm.L[hh];
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        if (L > 0.0f) r = make_float4(o.x / L, o.y / L, o.z / L, o.w / L);
        *reinterpret_cast<float4 *>(a.out + (int64_t(b) * a.q_heads + h0 + hh) * D + 4 * j4) = r;
    }
}

template <int D, bool kFromCache>
cudaError_t launch_attend_t(const AttendArgs &a, cudaStream_t s)
{
    const size_t smem = sizeof(AttendSmem<D>);
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(attend_kernel<D, kFromCache>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const dim3 grid(unsigned(a.nchunk_max), unsigned(a.kv_heads), unsigned(a.batch));
    attend_kernel<D, kFromCache><<<grid, kThreads, smem, s>>>(a);
    return cudaGetLastError();
}

static_assert(sizeof(AttendSmem<128>) <= 113 * 1024, "two CTAs per SM");

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
    const bool fused = a.k_cache != nullptr;
    if (a.head_dim == 128) return fused ? launch_attend_t<128, true>(a, s) : launch_attend_t<128, false>(a, s);
    if (a.head_dim == 64) return fused ? launch_attend_t<64, true>(a, s) : launch_attend_t<64, false>(a, s);
    return cudaErrorInvalidValue;
}

}  // namespace qsa
