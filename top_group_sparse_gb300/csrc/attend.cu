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
// GPU order (fixed, documented, batch independent).  The emitted row of
// query b is cut into sub-chunks of 64 consecutive rows, and the sub-chunks
// into kParts consecutive runs, one per CTA working on (query b, KV head); the
// split depends only on n_ids[b].  Each CTA walks its sub-chunks in row order
// with an online softmax for the n_q/n_kv query heads of that KV head: per
// sub-chunk, scaled scores x_i, the new running max m' = max(m, max x_i), the
// rescale e^(m - m') of the denominator l and of the accumulator, then
// l += sum_i e^(x_i - m') and acc += sum_i e^(x_i - m') v_i.  The last CTA of
// the (query, KV head) to finish -- an atomic ticket, nothing waits -- merges
// the kParts partials in order: M = max m_p, L = sum l_p e^(m_p - M),
// out = sum acc_p e^(m_p - M) / L.  No floating-point atomics; the bits of a
// query's output do not depend on the rest of the batch.
//
// Layout of a CTA: eight warps.  They resolve all of the CTA's rows once (every
// ID load, then every slot load) and stream the K/V sub-chunks through a
// two-stage ring in shared memory with 16-byte asynchronous copies (four
// threads per row, so each row read is one contiguous 512-byte run).  In the
// math a lane owns one 16-byte column of a row: the query heads' slices of
// that column live in registers, a warp forms R rows x GQ heads = 32 partial
// dot products at a time and a 31-shuffle reduce-scatter leaves each lane one
// finished score; for P.V each warp takes 8 rows of the sub-chunk for every head.
// Row source: kFromCache = false reads the gathered scratch (qsa_attend);
// kFromCache = true resolves each ID through the slot map, copies the row
// from the K/V cache, and the threads write their pieces of it to the scratch
// from shared memory (qsa_gather_attend, qsa_decode) -- the gather's output is
// the same bytes either way.
#include <cstddef>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kParts = kAttendParts;             // CTAs per (query, KV head)
constexpr int kSC = kAttendChunk;                // rows per sub-chunk
constexpr int kStages = 2;
constexpr int kThreads = 256;                    // 8 warps
constexpr int kMaxSub = (4 * QSA_MAX_BUDGET + 3 + kSC - 1) / kSC;   // 33 sub-chunks at most
constexpr int kMaxSubPerCta = (kMaxSub + kParts - 1) / kParts;     // 5
constexpr int kMaxRows = kMaxSubPerCta * kSC;                      // 320 rows per CTA at most

template <int D, int GQ>
struct AttendSmem {
    static constexpr int kKStride = D + 4;       // float4 rows land on distinct banks
    // every array read or written as float4 (or by 16-byte async copies)
    // starts on a 16-byte boundary whatever GQ and D are
    alignas(16) float q[GQ][D];
    alignas(16) float k[kStages][kSC][kKStride]; // also the end-of-run reduction area
    alignas(16) float v[kStages][kSC][D];
    alignas(16) float x[2][GQ][kSC];             // scaled scores, double buffered
    alignas(16) float pt[2][kSC][GQ < 4 ? 4 : GQ]; // weights, heads inner, double buffered
    alignas(16) float alpha[2][GQ < 4 ? 4 : GQ];   // rescale factors, double buffered
    int64_t off[kMaxRows];                       // element offset of each row in its source, -1: none
    float m_fin[GQ], l_fin[GQ];
    int last;
};

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// 32 partial values per lane, v[t], t = 0..31 -> lane L holds sum over lanes of v[L]
// (recursive halving: 31 shuffles).
__device__ __forceinline__ float reduce_scatter32(float (&v)[32], int lane)
{
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int j = 0; j < off; ++j) {
            const float give = upper ? v[j] : v[j + off];
            const float keep = upper ? v[j + off] : v[j];
            v[j] = keep + __shfl_xor_sync(0xffffffffu, give, off);
        }
    }
    return v[0];
}

template <int D, int GQ, bool kFromCache>
__global__ void __launch_bounds__(kThreads, 1)
attend_kernel(const AttendArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    using Sm = AttendSmem<D, GQ>;
    Sm &sm = *reinterpret_cast<Sm *>(smem_raw);
    constexpr int F4 = D / 4;
    constexpr int kGP = GQ < 4 ? 4 : GQ;
    constexpr int kPerRowThreads = 4;              // threads moving one row
    constexpr int kChunks = F4 / kPerRowThreads;   // 16-byte pieces per thread per row and matrix

    const int part = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = a.q_heads / a.kv_heads;  // <= GQ
    const int h0 = kvh * gq;

    // ---- independent of the previous kernel: the queries ---------------------------
    {
        const float4 *qg = reinterpret_cast<const float4 *>(a.q + (int64_t(b) * a.q_heads + h0) * D);
        for (int e = tid; e < GQ * F4; e += kThreads) {
            const int hh = e / F4, j4 = e - hh * F4;
            *reinterpret_cast<float4 *>(&sm.q[hh][4 * j4]) =
                hh < gq ? __ldg(qg + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    wait_for_predecessor();  // ids, n_ids (and the scratch) come from earlier kernels

    // n_ids and ids come from the previous kernel, which may still have been
    // running when this one started: L2-coherent loads, never the read-only path
    const int n = __ldcg(a.n_ids + b);
    if (n < 0 || n > a.row_cap) {
        if (part == 0) {
            for (int e = tid; e < gq * D; e += kThreads) a.out[(int64_t(b) * a.q_heads + h0) * D + e] = 0.0f;
            if (kvh == 0 && tid == 0) set_error(a.err, QSA_DEVERR_ROW_RANGE);
        }
        return;
    }
    const int nsub = (n + kSC - 1) / kSC;
    const int per = (nsub + kParts - 1) / kParts;
    const int s_begin = min(nsub, part * per);
    const int s_end = min(nsub, s_begin + per);
    const int my_sub = s_end - s_begin;
    const int64_t row_base = int64_t(b) * a.row_cap;          // scratch / ids row of query b
    const int64_t scr_rs = a.kv_heads;                        // scratch rows apart, in D units
    const int r_first = s_begin * kSC;
    const int r_last = min(n, s_end * kSC);
    const float *ksrc = kFromCache ? a.k_cache : a.k_scr;
    const float *vsrc = kFromCache ? a.v_cache : a.v_scr;

    // ---- resolve every row of this CTA once: all ID loads, then all slot loads ------
    {
        constexpr int kPer = (kMaxRows + kThreads - 1) / kThreads;  // 2
        int id[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int r = r_first + tid + u * kThreads;
            id[u] = (kFromCache && r < r_last) ? __ldcg(a.ids + row_base + r) : -1;
        }
        const int T = kFromCache ? __ldg(a.visible + b) : 0;
        const int32_t *smap = kFromCache ? a.slot_map + __ldg(a.slot_offset + b) : nullptr;
        int64_t slot[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int r = r_first + tid + u * kThreads;
            slot[u] = -1;
            if (kFromCache && r < r_last) {
                if (id[u] >= 0 && id[u] < T) slot[u] = __ldg(smap + id[u]);
                else set_error(a.err, QSA_DEVERR_ROW_RANGE);
            }
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int rl = tid + u * kThreads;  // row within this CTA's run
            if (rl < kMaxRows) {
                const int r = r_first + rl;
                int64_t o = -1;
                if (r < r_last) {
                    if (kFromCache) {
                        if (slot[u] >= 0 && slot[u] < a.num_slots) o = (slot[u] * a.kv_heads + kvh) * D;
                        else if (id[u] >= 0 && id[u] < T) set_error(a.err, QSA_DEVERR_SLOT_RANGE);
                    } else {
                        o = ((row_base + r) * scr_rs + kvh) * D;
                    }
                }
                sm.off[rl] = o;
            }
        }
    }
    __syncthreads();

    // rows of sub-chunk s into stage st: thread = (row i, quarter), 16-byte async copies
    const int mi = tid / kPerRowThreads;        // row moved by this thread
    const int mq = tid % kPerRowThreads;        // its quarter of the row
    auto issue = [&](int s) {
        const int st = s % kStages;
        const int r = (s_begin + s) * kSC + mi;
        const int64_t o = sm.off[s * kSC + mi];
        if (o >= 0) {
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                const int j4 = mq * kChunks + c;
                cp_async16(&sm.k[st][mi][4 * j4], ksrc + o + 4 * j4);
                cp_async16(&sm.v[st][mi][4 * j4], vsrc + o + 4 * j4);
            }
        } else if (r < n) {  // unresolvable row (flagged): zeros
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                const int j4 = mq * kChunks + c;
                *reinterpret_cast<float4 *>(&sm.k[st][mi][4 * j4]) = make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4 *>(&sm.v[st][mi][4 * j4]) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        cp_async_commit();
    };
    if (my_sub > 0) issue(0);

    // lane = 16-byte column d4 of a row (lanes >= F4 idle in the math)
    const bool col = lane < F4;
    float4 qreg[GQ];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh)
        qreg[hh] = col ? *reinterpret_cast<const float4 *>(&sm.q[hh][4 * lane]) : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 acc[GQ];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) acc[hh] = make_float4(0.f, 0.f, 0.f, 0.f);
    float m_run = -INFINITY, l_run = 0.0f;   // softmax state of this warp's head(s)
    float m_run2 = -INFINITY, l_run2 = 0.0f;
    constexpr int R = 32 / GQ;   // rows per group: R rows x GQ heads = 32 dot products
    constexpr int NG = kSC / R;  // groups per sub-chunk

    for (int s = 0; s < my_sub; ++s) {
        const int st = s % kStages;
        const int buf = s & 1;
        const int r0 = (s_begin + s) * kSC;
        const int rows = min(kSC, n - r0);
        if (s + 1 < my_sub) {
            issue(s + 1);        // the next sub-chunk streams in while this one is used
            cp_async_wait<1>();  // this thread's pieces of sub-chunk s have landed
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();         // ... and everyone else's

        if (kFromCache && mi < rows) {
            // the gather's output: this KV head's slice of scratch row r0 + mi
            float4 *kd = reinterpret_cast<float4 *>(a.k_scr_out + ((row_base + r0 + mi) * scr_rs + kvh) * D);
            float4 *vd = reinterpret_cast<float4 *>(a.v_scr_out + ((row_base + r0 + mi) * scr_rs + kvh) * D);
#pragma unroll
            for (int c = 0; c < kChunks; ++c) {
                const int j4 = mq * kChunks + c;
                kd[j4] = *reinterpret_cast<const float4 *>(&sm.k[st][mi][4 * j4]);
                vd[j4] = *reinterpret_cast<const float4 *>(&sm.v[st][mi][4 * j4]);
            }
        }

        // ---- scaled scores: a warp takes R rows at a time, lane = column ------------
        for (int g = warp; g < NG; g += kThreads / 32) {
            float v[32];
#pragma unroll
            for (int r = 0; r < R; ++r) {
                const float4 kv = col ? *reinterpret_cast<const float4 *>(&sm.k[st][g * R + r][4 * lane])
                                      : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int hh = 0; hh < GQ; ++hh) {
                    float d = qreg[hh].x * kv.x;
                    d = fmaf(qreg[hh].y, kv.y, d);
                    d = fmaf(qreg[hh].z, kv.z, d);
                    d = fmaf(qreg[hh].w, kv.w, d);
                    v[r * GQ + hh] = d;
                }
            }
            const float dot = reduce_scatter32(v, lane);  // lane L: row L / GQ, head L % GQ
            const int hh = lane % GQ;
            const int i = g * R + lane / GQ;
            sm.x[buf][hh][i] = (i < rows && hh < gq) ? a.scale * dot : -INFINITY;
        }
        __syncthreads();

        // ---- online softmax state, one warp per head (two for 16 heads) ---------------
#pragma unroll
        for (int rep = 0; rep < (GQ + 7) / 8; ++rep) {
            const int hh = warp + 8 * rep;
            if (hh < GQ) {
                const float x0 = sm.x[buf][hh][lane], x1 = sm.x[buf][hh][lane + 32];
                float mc = fmaxf(x0, x1);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
                float &mr = rep == 0 ? m_run : m_run2;
                float &lr = rep == 0 ? l_run : l_run2;
                const float m_new = fmaxf(mr, mc);
                float p0 = 0.0f, p1 = 0.0f, al = 0.0f;
                if (m_new != -INFINITY) {
                    p0 = expf(x0 - m_new);
                    p1 = expf(x1 - m_new);
                    al = mr == -INFINITY ? 0.0f : expf(mr - m_new);
                }
                sm.pt[buf][lane][hh] = p0;
                sm.pt[buf][lane + 32][hh] = p1;
                float ps = p0 + p1;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
                lr = fmaf(lr, al, ps);
                mr = m_new;
                if (lane == 0) sm.alpha[buf][hh] = al;
            }
        }
        __syncthreads();

        // ---- acc[h] = acc[h] * alpha_h + sum_i p_ih v_i over this warp's 8 rows --------
        if (col) {
#pragma unroll
            for (int hh = 0; hh < GQ; ++hh) {
                const float al = sm.alpha[buf][hh];
                acc[hh].x *= al;
                acc[hh].y *= al;
                acc[hh].z *= al;
                acc[hh].w *= al;
            }
            const int i0 = warp * (kSC / 8);
            const int i1 = min(rows, i0 + kSC / 8);
            for (int i = i0; i < i1; ++i) {
                const float4 vv = *reinterpret_cast<const float4 *>(&sm.v[st][i][4 * lane]);
#pragma unroll
                for (int h4 = 0; h4 < kGP / 4; ++h4) {
                    const float4 pp = *reinterpret_cast<const float4 *>(&sm.pt[buf][i][4 * h4]);
                    const float pw[4] = {pp.x, pp.y, pp.z, pp.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int hh = 4 * h4 + u;
                        if (hh < GQ) {
                            acc[hh].x = fmaf(pw[u], vv.x, acc[hh].x);
                            acc[hh].y = fmaf(pw[u], vv.y, acc[hh].y);
                            acc[hh].z = fmaf(pw[u], vv.z, acc[hh].z);
                            acc[hh].w = fmaf(pw[u], vv.w, acc[hh].w);
                        }
                    }
                }
            }
        }
        __syncthreads();  // stage st may be refilled by the next iteration's copies
    }

    // ---- this CTA's partial: acc summed over the 8 warps (fixed order) --------------
    float *red = &sm.k[0][0][0];  // [8 warps][GQ][D]; every copy has landed
    if (col) {
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh)
            *reinterpret_cast<float4 *>(&red[(warp * GQ + hh) * D + 4 * lane]) = acc[hh];
    }
    if (lane == 0) {
#pragma unroll
        for (int rep = 0; rep < (GQ + 7) / 8; ++rep) {
            const int hh = warp + 8 * rep;
            if (hh < GQ) {
                sm.m_fin[hh] = rep == 0 ? m_run : m_run2;
                sm.l_fin[hh] = rep == 0 ? l_run : l_run2;
            }
        }
    }
    __syncthreads();
    const int64_t pbase = (int64_t(b) * a.q_heads + h0) * a.nparts + part;  // head h0, part
    for (int e = tid; e < gq * F4; e += kThreads) {
        const int hh = e / F4, j4 = e - hh * F4;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < 8; ++w) {
            const float4 p = *reinterpret_cast<const float4 *>(&red[(w * GQ + hh) * D + 4 * j4]);
            o.x += p.x;
            o.y += p.y;
            o.z += p.z;
            o.w += p.w;
        }
        reinterpret_cast<float4 *>(a.part_acc + (pbase + int64_t(hh) * a.nparts) * D)[j4] = o;
    }
    if (tid < gq) {
        a.part_m[pbase + int64_t(tid) * a.nparts] = sm.m_fin[tid];
        a.part_l[pbase + int64_t(tid) * a.nparts] = sm.l_fin[tid];
    }

    // ---- the last CTA of this (query, KV head) merges the parts in order ----------
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        uint32_t *ticket = a.tickets + int64_t(b) * a.kv_heads + kvh;
        sm.last = atomicAdd(ticket, 1u) == uint32_t(kParts - 1);
        if (sm.last) *ticket = 0u;  // leave the ticket clean for the next call
    }
    __syncthreads();
    if (!sm.last) return;
    __threadfence();
    const int64_t hb0 = (int64_t(b) * a.q_heads + h0) * a.nparts;
    // part maxima and denominators first (one round of loads), then the accumulators
    float *wm = &sm.x[0][0][0];  // [GQ][kParts] weights, reused
    for (int e = tid; e < gq * kParts; e += kThreads) {
        const int hh = e / kParts, c = e - hh * kParts;
        wm[hh * kParts + c] = __ldcg(a.part_m + hb0 + int64_t(hh) * a.nparts + c);
    }
    __syncthreads();
    if (tid < gq) {
        float M = -INFINITY;
        for (int c = 0; c < kParts; ++c) M = fmaxf(M, wm[tid * kParts + c]);
        float L = 0.0f;
        for (int c = 0; c < kParts; ++c) {
            const float w = M == -INFINITY ? 0.0f : expf(wm[tid * kParts + c] - M);
            L = fmaf(__ldcg(a.part_l + hb0 + int64_t(tid) * a.nparts + c), w, L);
            wm[tid * kParts + c] = w;
        }
        sm.l_fin[tid] = L;
    }
    __syncthreads();
    for (int e = tid; e < gq * F4; e += kThreads) {
        const int hh = e / F4, j4 = e - hh * F4;
        const float4 *src = reinterpret_cast<const float4 *>(a.part_acc + (hb0 + int64_t(hh) * a.nparts) * D) + j4;
        float4 xv[kParts];
#pragma unroll
        for (int c = 0; c < kParts; ++c) xv[c] = __ldcg(src + int64_t(c) * F4);
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kParts; ++c) {
            const float w = wm[hh * kParts + c];
            o.x = fmaf(xv[c].x, w, o.x);
            o.y = fmaf(xv[c].y, w, o.y);
            o.z = fmaf(xv[c].z, w, o.z);
            o.w = fmaf(xv[c].w, w, o.w);
        }
        const float L = sm.l_fin[hh];
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        if (L > 0.0f) r = make_float4(o.x / L, o.y / L, o.z / L, o.w / L);
        *reinterpret_cast<float4 *>(a.out + (int64_t(b) * a.q_heads + h0 + hh) * D + 4 * j4) = r;
    }
}

template <int D, int GQ, bool kFromCache>
cudaError_t launch_attend_t(const AttendArgs &a, cudaStream_t s, bool pdl)
{
    const size_t smem = sizeof(AttendSmem<D, GQ>);
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(attend_kernel<D, GQ, kFromCache>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    const dim3 grid(kParts, unsigned(a.kv_heads), unsigned(a.batch));
    return launch_kernel(attend_kernel<D, GQ, kFromCache>, grid, dim3(kThreads), smem, s, pdl, a);
}

template <int D, bool kFromCache>
cudaError_t launch_attend_d(const AttendArgs &a, cudaStream_t s, bool pdl)
{
    const int gq = a.q_heads / a.kv_heads;
    if (gq <= 1) return launch_attend_t<D, 1, kFromCache>(a, s, pdl);
    if (gq <= 2) return launch_attend_t<D, 2, kFromCache>(a, s, pdl);
    if (gq <= 4) return launch_attend_t<D, 4, kFromCache>(a, s, pdl);
    if (gq <= 8) return launch_attend_t<D, 8, kFromCache>(a, s, pdl);
    return launch_attend_t<D, 16, kFromCache>(a, s, pdl);
}

static_assert(sizeof(AttendSmem<128, 16>) <= 227 * 1024, "shared memory per CTA");
static_assert(kThreads / 32 == 8, "the end-of-run reduction sums 8 warps; P.V takes 8 rows per warp");

template <int D, int GQ>
constexpr bool layout_ok()
{
    using S = AttendSmem<D, GQ>;
    return offsetof(S, q) % 16 == 0 && offsetof(S, k) % 16 == 0 && offsetof(S, v) % 16 == 0 &&
           offsetof(S, x) % 16 == 0 && offsetof(S, pt) % 16 == 0 && offsetof(S, alpha) % 16 == 0 &&
           offsetof(S, off) % 8 == 0 && (S::kKStride * 4) % 16 == 0 && sizeof(S::x) >= GQ * kParts * 4 &&
           sizeof(S::k) >= size_t(8) * GQ * D * 4;  // room for the end-of-run reduction
}
static_assert(layout_ok<64, 1>() && layout_ok<64, 2>() && layout_ok<64, 4>() && layout_ok<64, 8>() &&
                  layout_ok<64, 16>() && layout_ok<128, 1>() && layout_ok<128, 2>() && layout_ok<128, 4>() &&
                  layout_ok<128, 8>() && layout_ok<128, 16>(),
              "16-byte alignment of every float4 / bulk-copy array");

}  // namespace

bool attend_shape_supported(int head_dim, int q_heads, int kv_heads)
{
    if (head_dim != 64 && head_dim != 128) return false;
    if (kv_heads <= 0 || q_heads <= 0 || q_heads % kv_heads != 0) return false;
    return q_heads / kv_heads <= kMaxGqa;
}

cudaError_t launch_attend(const AttendArgs &a, cudaStream_t s, bool pdl)
{
    if (a.batch == 0) return cudaSuccess;
    const bool fused = a.k_cache != nullptr;
    if (a.head_dim == 128)
        return fused ? launch_attend_d<128, true>(a, s, pdl) : launch_attend_d<128, false>(a, s, pdl);
    if (a.head_dim == 64)
        return fused ? launch_attend_d<64, true>(a, s, pdl) : launch_attend_d<64, false>(a, s, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace qsa
