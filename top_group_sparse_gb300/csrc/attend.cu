// attend.cu -- stage 4 (online softmax over the compact row), alone or fused
// with stage 3 (slot resolution and compact gather).
//
// "Top-k chooses the set; time chooses the order" (AFN-017), Floating point
// makes order observable: a real online softmax is a sequence of rounded
// max / rescale / exp / denominator / accumulator updates, so one canonical
// visit order is needed -- the emitted, chronological one.  "A sparse mask is
// not sparse attention" (AFN-016), Decision: online softmax over at most
// 2,051 gathered rows; only the gather crosses from logical identity into the
// physical cache layout.
//
// GPU order (fixed, documented, batch independent).  The emitted row of
// query b is cut into runs of kRowsPerPart (128) consecutive rows, one CTA per
// (run, KV head, query b); the cut depends only on n_ids[b].  A run is cut
// into steps of 4 consecutive rows, and step j goes to warp j mod 8, which
// keeps its own online-softmax state for the GQ query heads of the KV head:
// per step, scaled scores x_i, the new running max m' = max(m, max x_i), the
// rescale e^(m - m') of the denominator l and of the accumulator, then
// l += sum_i e^(x_i - m') and acc += sum_i e^(x_i - m') v_i.  At the end of
// the run the eight warp states are merged in warp order (M = max m_w,
// L = sum l_w e^(m_w - M), acc = sum acc_w e^(m_w - M)), and the runs are
// merged in order the same way and divided by L (merge_runs): by the last CTA
// of the (query, KV head) to finish -- an atomic ticket, nothing waits -- when
// the grid fits on the GPU at once, else by a second small launch after the
// grid, so that no CTA holds its SM through the fence and the ticket.  With
// the state export (AttendArgs::m_out) the merge stores M, L and the undivided
// acc instead, so that separately attended slices of one row combine in row
// order.  No floating-point atomics; the bits of a query's output do not
// depend on the rest of the batch.
//
// Data movement: the CTA's threads resolve every row of its run at once
// (one row each: the ID load, then the slot-map load).  Each warp then
// streams only its own steps through its own three-slot ring in shared
// memory with 16-byte asynchronous copies, two steps ahead of its math, so no
// thread-block barrier and no cross-warp wait sits inside the loop.  Eight
// warps of short steps and two CTAs per SM (for GQ <= 8) keep sixteen warps
// on every SM: the loop is issue- and latency-bound, and each warp has only
// about four steps to run.
//
// Math of a step (4 rows x GQ heads).  Scores: lanes form HP = min(GQ, 4)
// head groups of DS = 32/HP lanes; a lane holds HPL = GQ/HP heads of the query
// in registers, restricted to its d-slice (16-byte columns ds, ds + DS, ...),
// forms 4 x HPL partial dot products, and a reduce-scatter over the DS lanes
// of its group leaves it NVO finished dots (one row, NVO consecutive heads).
// Weighted values: a lane owns one 16-byte column of V for all GQ heads.
//
// Row source: Src::kScratch reads the gathered scratch (qsa_attend);
// Src::kCache resolves each ID through the slot map and copies the row from
// the K/V cache straight into shared memory (qsa_decode: the compact row
// never exists in device memory); Src::kCacheStore does the same and also
// writes every row from shared memory to the scratch (qsa_gather_attend,
// the same bytes as qsa_gather).
#include <cstddef>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kRowsPerPart = kAttendRowsPerPart;  // 128
constexpr int kParts = kAttendParts;               // 17 runs at most (2,051 rows)
constexpr int kStepRows = 4;                       // rows per warp step
constexpr int kRing = 3;                           // steps in flight per warp (ring slots)
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;

// CTAs per SM the kernel is built for: the running state of GQ heads (an
// accumulator column and the query slice per head) fits 128 registers a
// thread up to GQ = 8.
template <int GQ>
constexpr int attend_ctas_per_sm() { return GQ <= 8 ? 2 : 1; }

enum class Src { kScratch, kCache, kCacheStore };

template <int D, int GQ>
struct AttendSmem {
    // every array read or written as float4 (or by 16-byte async copies)
    // starts on a 16-byte boundary whatever GQ and D are
    alignas(128) float k[kWarps][kRing][kStepRows][D];  // k and v: also the end-of-run reduction area
    alignas(128) float v[kWarps][kRing][kStepRows][D];
    alignas(16) float q[GQ][D];
    alignas(16) float pt[kWarps][kStepRows][GQ < 4 ? 4 : GQ];  // weights of a warp's step, [row][head]
    alignas(16) float alpha[kWarps][GQ < 4 ? 4 : GQ];          // rescale factors of a warp's step
    alignas(16) float wm[kWarps][GQ];       // warp states at the end of the run
    alignas(16) float wl[kWarps][GQ];
    alignas(16) float ww[kWarps][GQ];       // their merge weights
    alignas(16) float pw[GQ][kParts];       // merge weights of the runs (last CTA)
    int64_t off[kRowsPerPart];              // element offset of each row of the run; -1 none, -2 bad
    float l_fin[GQ];
    int last;
};

__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gmem_src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(gmem_src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Reduce-scatter over the DS = 2*O lanes of an xor group (offsets O, O/2, .., 1):
// N values per lane in, max(1, N/DS) values per lane out (v[0..]).  While more
// than one value is left, each level halves them (the lane with bit O set keeps
// the upper half); after that it is a plain butterfly sum.
template <int N, int O>
__device__ __forceinline__ void reduce_scatter(float (&v)[32], int lane)
{
    if constexpr (O >= 1) {
        if constexpr (N > 1) {
            const bool upper = (lane & O) != 0;
#pragma unroll
            for (int j = 0; j < N / 2; ++j) {
                const float give = upper ? v[j] : v[j + N / 2];
                const float keep = upper ? v[j + N / 2] : v[j];
                v[j] = keep + __shfl_xor_sync(0xffffffffu, give, O);
            }
            reduce_scatter<N / 2, O / 2>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
            reduce_scatter<1, O / 2>(v, lane);
        }
    }
}

// The runs of (query b, KV head kvh) merged in run order from their states in
// the workspace: M = max m_c, w_c = e^(m_c - M), L = sum_c l_c w_c,
// out = (sum_c acc_c w_c) / L, c = 0..used-1 in order (0 for L = 0); with the
// state export, out = sum_c acc_c w_c, m_out = M, l_out = L.  Every thread of
// the CTA (kNT of them) calls it.
template <int D, int GQ, int kNT>
__device__ __forceinline__ void merge_runs(const AttendArgs &a, int b, int kvh, int used, float (&pw)[GQ][kParts],
                                           float *l_fin)
{
    constexpr int F4 = D / 4;
    const int tid = threadIdx.x;
    const int gq = a.q_heads / a.kv_heads;
    const int h0 = kvh * gq;
    const int64_t hb0 = (int64_t(b) * a.q_heads + h0) * a.nparts;
    // every load first (one round trip), then the weights, then the sums
    const int e0 = tid;  // one (head, column) element per thread when gq * F4 <= kNT
    const int hh0 = e0 / F4, jj0 = e0 - hh0 * F4;
    float4 xv[kParts];
    if (e0 < gq * F4) {
        const float4 *src = reinterpret_cast<const float4 *>(a.part_acc + (hb0 + int64_t(hh0) * a.nparts) * D) + jj0;
#pragma unroll
        for (int c = 0; c < kParts; ++c)
            xv[c] = c < used ? __ldcg(src + int64_t(c) * F4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (tid < gq) {
        const int64_t hb = hb0 + int64_t(tid) * a.nparts;
        float pm[kParts], pl[kParts];
#pragma unroll
        for (int c = 0; c < kParts; ++c) {
            pm[c] = c < used ? __ldcg(a.part_m + hb + c) : -INFINITY;
            pl[c] = c < used ? __ldcg(a.part_l + hb + c) : 0.0f;
        }
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kParts; ++c) M = fmaxf(M, pm[c]);
        float L = 0.0f;
#pragma unroll
        for (int c = 0; c < kParts; ++c) {
            const float w = (c >= used || M == -INFINITY) ? 0.0f : expf(pm[c] - M);
            if (c < used) L = fmaf(pl[c], w, L);
            pw[tid][c] = w;
        }
        l_fin[tid] = L;
        if (a.m_out != nullptr) {
            a.m_out[int64_t(b) * a.q_heads + h0 + tid] = M;
            a.l_out[int64_t(b) * a.q_heads + h0 + tid] = L;
        }
    }
    __syncthreads();
    for (int e = tid; e < gq * F4; e += kNT) {
        const int hh = e / F4, j4 = e - hh * F4;
        if (e != e0) {  // more elements than threads: load this one now
            const float4 *src = reinterpret_cast<const float4 *>(a.part_acc + (hb0 + int64_t(hh) * a.nparts) * D) + j4;
#pragma unroll
            for (int c = 0; c < kParts; ++c)
                xv[c] = c < used ? __ldcg(src + int64_t(c) * F4) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kParts; ++c) {
            if (c < used) {
                const float w = pw[hh][c];
                o.x = fmaf(xv[c].x, w, o.x);
                o.y = fmaf(xv[c].y, w, o.y);
                o.z = fmaf(xv[c].z, w, o.z);
                o.w = fmaf(xv[c].w, w, o.w);
            }
        }
        const float L = l_fin[hh];
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        if (a.m_out != nullptr) r = o;
        else if (L > 0.0f) r = make_float4(o.x / L, o.y / L, o.z / L, o.w / L);
        *reinterpret_cast<float4 *>(a.out + (int64_t(b) * a.q_heads + h0 + hh) * D + 4 * j4) = r;
    }
}

constexpr int kMergeThreads = 256;

// qsa_merge_states: the states of n_parts consecutive slices of each row
// (m, l [n_parts, bh]; acc [n_parts, bh, D]) merged in slice order with the
// arithmetic of merge_runs -- M = max m_r, w_r = e^(m_r - M), L and acc
// summed by fmaf in slice order, then acc / L -- so that one slice of a whole
// row gives qsa_decode's output bit for bit.  One thread per (query-head,
// 16-byte column).
__global__ void __launch_bounds__(kMergeThreads)
merge_states_kernel(const float *m, const float *l, const float *acc, float *out, int n_parts, int bh, int f4)
{
    const int64_t e = int64_t(blockIdx.x) * kMergeThreads + threadIdx.x;
    if (e >= int64_t(bh) * f4) return;
    const int hb = int(e / f4), j4 = int(e - int64_t(hb) * f4);
    float M = -INFINITY;
    for (int r = 0; r < n_parts; ++r) M = fmaxf(M, __ldg(m + int64_t(r) * bh + hb));
    float L = 0.0f;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r = 0; r < n_parts; ++r) {
        const float w = M == -INFINITY ? 0.0f : expf(__ldg(m + int64_t(r) * bh + hb) - M);
        L = fmaf(__ldg(l + int64_t(r) * bh + hb), w, L);
        const float4 x = __ldg(reinterpret_cast<const float4 *>(acc) + (int64_t(r) * bh + hb) * f4 + j4);
        o.x = fmaf(x.x, w, o.x);
        o.y = fmaf(x.y, w, o.y);
        o.z = fmaf(x.z, w, o.z);
        o.w = fmaf(x.w, w, o.w);
    }
    float4 res = make_float4(0.f, 0.f, 0.f, 0.f);
    if (L > 0.0f) res = make_float4(o.x / L, o.y / L, o.z / L, o.w / L);
    reinterpret_cast<float4 *>(out)[e] = res;
}

// The second launch of a deferred merge: one CTA per (KV head, query).
template <int D, int GQ>
__global__ void __launch_bounds__(kMergeThreads) attend_merge_kernel(const AttendArgs a)
{
    __shared__ float pw[GQ][kParts];
    __shared__ float l_fin[GQ];
    const int kvh = blockIdx.x, b = blockIdx.y;
    wait_for_predecessor();  // the run states come from the attention launch
    const int n = __ldcg(a.n_ids + b);
    if (n < 0 || n > a.row_cap) return;  // the attention zeroed this output and flagged it
    const int used = max(1, (n + kRowsPerPart - 1) / kRowsPerPart);
    merge_runs<D, GQ, kMergeThreads>(a, b, kvh, used, pw, l_fin);
}

template <int D, int GQ, Src kSrc>
__global__ void __launch_bounds__(kThreads, attend_ctas_per_sm<GQ>())
attend_kernel(const AttendArgs a)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    using Sm = AttendSmem<D, GQ>;
    Sm &sm = *reinterpret_cast<Sm *>(smem_raw);
    constexpr int F4 = D / 4;                    // 16-byte columns of a row
    constexpr int kGP = GQ < 4 ? 4 : GQ;         // padded head count of pt / alpha
    constexpr bool kFromCache = kSrc != Src::kScratch;
    constexpr bool kStore = kSrc == Src::kCacheStore;
    // score layout: HP head groups x DS lanes; a lane holds HPL heads x NF columns
    constexpr int HP = GQ < 4 ? GQ : 4;
    constexpr int HPL = GQ / HP;
    constexpr int DS = 32 / HP;
    constexpr int NF = (F4 + DS - 1) / DS;
    constexpr int NV = kStepRows * HPL;          // partial dots per lane before the reduce
    // after the reduce-scatter a lane holds NVO finished dots, entries
    // (ds / RSH) * NVO + j of the [row][head] list (RSH lanes hold each copy):
    // one row, heads u0 .. u0 + NVO - 1; lanes ROFF apart hold the next row
    constexpr int NVO = NV >= DS ? NV / DS : 1;
    constexpr int RSH = NV >= DS ? 1 : DS / NV;
    constexpr int ROFF = (HPL / NVO) * RSH;
    static_assert(NV <= 32 && HPL % NVO == 0 && ROFF * kStepRows == DS, "one row per lane after the reduce");

    const int part = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int gq = a.q_heads / a.kv_heads;  // <= GQ
    const int h0 = kvh * gq;

    // ---- independent of the previous kernel: queries and the history -------------
    {
        const float4 *qg = reinterpret_cast<const float4 *>(a.q + (int64_t(b) * a.q_heads + h0) * D);
        for (int e = tid; e < GQ * F4; e += kThreads) {
            const int hh = e / F4, j4 = e - hh * F4;
            *reinterpret_cast<float4 *>(&sm.q[hh][4 * j4]) =
                hh < gq ? __ldg(qg + e) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    const int T = kFromCache ? __ldg(a.visible + b) : 0;
    const int64_t smap_off = kFromCache ? __ldg(a.slot_offset + b) : 0;
    wait_for_predecessor();  // ids and n_ids (or the scratch) come from earlier kernels

    // n_ids and ids come from the previous kernel, which may still have been
    // running when this one started: L2-coherent loads, never the read-only path.
    // The ID of this thread's row is loaded with n (one round trip) and used
    // only if the row exists.
    const int64_t row_base = int64_t(b) * a.row_cap;   // ids / scratch row of query b
    const int r0 = part * kRowsPerPart;
    const int my_r = r0 + tid;
    int id = 0;
    if (kFromCache && tid < kRowsPerPart && my_r < a.row_cap) id = __ldcg(a.ids + row_base + my_r);
    const int n = __ldcg(a.n_ids + b);
    if (a.ids_out != nullptr && kvh == 0) {  // the caller's copy of the rows and the count
        if (tid < kRowsPerPart && my_r < n && my_r < a.row_cap) a.ids_out[row_base + my_r] = id;
        if (part == 0 && tid == 0) a.n_ids_out[b] = n;
    }
    if (n < 0 || n > a.row_cap) {
        if (part == 0) {
            for (int e = tid; e < gq * D; e += kThreads) a.out[(int64_t(b) * a.q_heads + h0) * D + e] = 0.0f;
            if (a.m_out != nullptr && tid < gq) {  // the empty state
                a.m_out[int64_t(b) * a.q_heads + h0 + tid] = -INFINITY;
                a.l_out[int64_t(b) * a.q_heads + h0 + tid] = 0.0f;
            }
            if (kvh == 0 && tid == 0) set_error(a.err, QSA_DEVERR_ROW_RANGE);
        }
        return;
    }
    const int used = max(1, (n + kRowsPerPart - 1) / kRowsPerPart);  // runs of this query
    if (part >= used) return;
    const int r_end = min(n, r0 + kRowsPerPart);
    const int64_t rs = a.kv_heads;                                   // scratch rows apart, in D units

    // ---- resolve the run: thread t takes row r0 + t ---------------------------------
    {
        int64_t o = -1;
        if (tid < kRowsPerPart && my_r < r_end) {
            if constexpr (kFromCache) {
                if (id >= 0 && id < T) {
                    const int slot = __ldg(a.slot_map + smap_off + id);
                    if (slot >= 0 && slot < a.num_slots) {
                        o = (int64_t(slot) * a.kv_heads + kvh) * D;
                    } else {
                        o = -2;
                        set_error(a.err, QSA_DEVERR_SLOT_RANGE);
                    }
                } else {
                    o = -2;
                    set_error(a.err, QSA_DEVERR_ROW_RANGE);
                }
            } else {
                o = ((row_base + my_r) * rs + kvh) * D;
            }
        }
        if (tid < kRowsPerPart) sm.off[tid] = o;
    }
    __syncthreads();

    // ---- this warp's steps: j = warp, warp + kWarps, ... ----------------------------
    const int nsteps = (r_end - r0 + kStepRows - 1) / kStepRows;
    const int my_steps = nsteps > warp ? (nsteps - warp + kWarps - 1) / kWarps : 0;
    const float *ksrc = kFromCache ? a.k_cache : a.k_scr;
    const float *vsrc = kFromCache ? a.v_cache : a.v_scr;
    auto issue = [&](int k) {  // the warp's k-th step into ring slot k % kRing
        const int j = warp + kWarps * k;
        const int sl = k % kRing;
#pragma unroll
        for (int e = lane; e < kStepRows * F4; e += 32) {
            const int r = e / F4, c = e - r * F4;
            const int rl = j * kStepRows + r;  // row within the run
            const int64_t o = r0 + rl < r_end ? sm.off[rl] : -1;
            if (o >= 0) {
                cp_async16(&sm.k[warp][sl][r][4 * c], ksrc + o + 4 * c);
                cp_async16(&sm.v[warp][sl][r][4 * c], vsrc + o + 4 * c);
            } else if (o == -2) {  // unresolvable row (flagged): zeros
                *reinterpret_cast<float4 *>(&sm.k[warp][sl][r][4 * c]) = make_float4(0.f, 0.f, 0.f, 0.f);
                *reinterpret_cast<float4 *>(&sm.v[warp][sl][r][4 * c]) = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    };
#pragma unroll
    for (int k = 0; k < kRing - 1; ++k) {
        if (k < my_steps) issue(k);
        cp_async_commit();
    }

    // score-layout coordinates of this lane
    const int hg = lane / DS, ds = lane % DS;
    const int i0 = (ds / RSH) * NVO;             // first [row][head] entry this lane ends with
    const int r_lane = i0 / HPL;                 // its row
    const int h_lane = hg * HPL + i0 % HPL;      // its first head (NVO consecutive heads)
    float4 qreg[HPL][NF];
#pragma unroll
    for (int u = 0; u < HPL; ++u)
#pragma unroll
        for (int i = 0; i < NF; ++i) {
            const int c = ds + DS * i;
            qreg[u][i] = c < F4 ? *reinterpret_cast<const float4 *>(&sm.q[hg * HPL + u][4 * c])
                                : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    const bool col = lane < F4;  // value layout: lane = 16-byte column (lanes >= F4 idle)
    float4 acc[GQ];
#pragma unroll
    for (int hh = 0; hh < GQ; ++hh) acc[hh] = make_float4(0.f, 0.f, 0.f, 0.f);
    float m_run[NVO], l_run[NVO];  // states of heads h_lane + j over this warp's rows
#pragma unroll
    for (int j = 0; j < NVO; ++j) {
        m_run[j] = -INFINITY;
        l_run[j] = 0.0f;
    }

    for (int k = 0; k < my_steps; ++k) {
        if (k + kRing - 1 < my_steps) issue(k + kRing - 1);  // into the slot step k-1 used
        cp_async_commit();
        cp_async_wait<kRing - 1>();  // this lane's copies of step k have landed
        __syncwarp();                // ... and the whole warp's
        const int sl = k % kRing;
        const int j = warp + kWarps * k;
        const int rows = min(kStepRows, r_end - (r0 + j * kStepRows));

        if constexpr (kStore) {
            // the gather's output: the step's rows, from shared memory to the scratch
            for (int e = lane; e < rows * F4; e += 32) {
                const int r = e / F4, c = e - r * F4;
                const int64_t dst = ((row_base + r0 + j * kStepRows + r) * rs + kvh) * D + 4 * c;
                *reinterpret_cast<float4 *>(a.k_scr_out + dst) = *reinterpret_cast<const float4 *>(&sm.k[warp][sl][r][4 * c]);
                *reinterpret_cast<float4 *>(a.v_scr_out + dst) = *reinterpret_cast<const float4 *>(&sm.v[warp][sl][r][4 * c]);
            }
        }

        // ---- 4 rows x HPL heads of partial dots over this lane's columns --------------
        float v[32];
#pragma unroll
        for (int r = 0; r < kStepRows; ++r) {
#pragma unroll
            for (int i = 0; i < NF; ++i) {
                const int c = ds + DS * i;
                const float4 kv = c < F4 ? *reinterpret_cast<const float4 *>(&sm.k[warp][sl][r][4 * c])
                                         : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int u = 0; u < HPL; ++u) {
                    float d = i == 0 ? qreg[u][i].x * kv.x : fmaf(qreg[u][i].x, kv.x, v[r * HPL + u]);
                    d = fmaf(qreg[u][i].y, kv.y, d);
                    d = fmaf(qreg[u][i].z, kv.z, d);
                    d = fmaf(qreg[u][i].w, kv.w, d);
                    v[r * HPL + u] = d;
                }
            }
        }
        reduce_scatter<NV, DS / 2>(v, lane);  // v[j]: row r_lane, head h_lane + j

        // ---- online softmax step of this lane's heads over the 4 rows ------------------
        float al[NVO];
        bool unit = true;  // every rescale factor is 1 (nothing to rescale)
#pragma unroll
        for (int j = 0; j < NVO; ++j) {
            const bool ok = r_lane < rows && h_lane + j < gq;
            const float x = ok ? a.scale * v[j] : -INFINITY;
            float mc = x;
#pragma unroll
            for (int o = ROFF; o < DS; o <<= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
            const float m_new = fmaxf(m_run[j], mc);
            float p = 0.0f, alpha = 0.0f;
            if (m_new != -INFINITY) {
                p = expf(x - m_new);
                alpha = m_run[j] == -INFINITY ? 0.0f : expf(m_run[j] - m_new);
            }
            float ps = p;
#pragma unroll
            for (int o = ROFF; o < DS; o <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
            l_run[j] = fmaf(l_run[j], alpha, ps);
            m_run[j] = m_new;
            al[j] = alpha;
            unit = unit && (alpha == 1.0f || m_new == -INFINITY);
            if (ds % RSH == 0) sm.pt[warp][r_lane][h_lane + j] = p;
        }
        if (r_lane == 0 && ds % RSH == 0) {
#pragma unroll
            for (int j = 0; j < NVO; ++j) sm.alpha[warp][h_lane + j] = al[j];
        }
        const bool rescale = !__all_sync(0xffffffffu, unit);
        __syncwarp();

        // ---- acc[h] = acc[h] * alpha_h + sum_r p_rh v_r ---------------------------------
        if (col) {
            if (rescale) {  // (multiplying by 1 would change nothing)
#pragma unroll
                for (int h4 = 0; h4 < kGP / 4; ++h4) {
                    const float4 al4 = *reinterpret_cast<const float4 *>(&sm.alpha[warp][4 * h4]);
                    const float alw[4] = {al4.x, al4.y, al4.z, al4.w};
#pragma unroll
                    for (int w4 = 0; w4 < 4; ++w4) {
                        const int hh = 4 * h4 + w4;
                        if (hh < GQ) {
                            acc[hh].x *= alw[w4];
                            acc[hh].y *= alw[w4];
                            acc[hh].z *= alw[w4];
                            acc[hh].w *= alw[w4];
                        }
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < kStepRows; ++r) {
                if (r < rows) {
                    const float4 vv = *reinterpret_cast<const float4 *>(&sm.v[warp][sl][r][4 * lane]);
                    float pw[kGP];
#pragma unroll
                    for (int h4 = 0; h4 < kGP / 4; ++h4) {
                        const float4 pp = *reinterpret_cast<const float4 *>(&sm.pt[warp][r][4 * h4]);
                        pw[4 * h4 + 0] = pp.x;
                        pw[4 * h4 + 1] = pp.y;
                        pw[4 * h4 + 2] = pp.z;
                        pw[4 * h4 + 3] = pp.w;
                    }
#pragma unroll
                    for (int hh = 0; hh < GQ; ++hh) {
                        acc[hh].x = fmaf(pw[hh], vv.x, acc[hh].x);
                        acc[hh].y = fmaf(pw[hh], vv.y, acc[hh].y);
                        acc[hh].z = fmaf(pw[hh], vv.z, acc[hh].z);
                        acc[hh].w = fmaf(pw[hh], vv.w, acc[hh].w);
                    }
                }
            }
        }
        __syncwarp();  // the slot, pt and alpha are rewritten by later steps
    }
    cp_async_wait<0>();

    // ---- this CTA's partial: the warp states merged in warp order --------------------
    __syncthreads();  // every warp is done with its ring: it becomes the reduction area
    float *red = &sm.k[0][0][0][0];  // [kWarps][GQ][D], over k and then v
    if (col) {
#pragma unroll
        for (int hh = 0; hh < GQ; ++hh)
            *reinterpret_cast<float4 *>(&red[(warp * GQ + hh) * D + 4 * lane]) = acc[hh];
    }
    if (r_lane == 0 && ds % RSH == 0) {
#pragma unroll
        for (int j = 0; j < NVO; ++j) {
            sm.wm[warp][h_lane + j] = m_run[j];
            sm.wl[warp][h_lane + j] = l_run[j];
        }
    }
    __syncthreads();
    const int64_t pbase = (int64_t(b) * a.q_heads + h0) * a.nparts + part;  // head h0, this run
    if (tid < gq) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm.wm[w][tid]);
        float L = 0.0f;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float wt = M == -INFINITY ? 0.0f : expf(sm.wm[w][tid] - M);
            sm.ww[w][tid] = wt;
            L = fmaf(sm.wl[w][tid], wt, L);
        }
        a.part_m[pbase + int64_t(tid) * a.nparts] = M;
        a.part_l[pbase + int64_t(tid) * a.nparts] = L;
    }
    __syncthreads();
    for (int e = tid; e < gq * F4; e += kThreads) {
        const int hh = e / F4, j4 = e - hh * F4;
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kWarps; ++w) {
            const float4 p = *reinterpret_cast<const float4 *>(&red[(w * GQ + hh) * D + 4 * j4]);
            const float wt = sm.ww[w][hh];
            o.x = fmaf(p.x, wt, o.x);
            o.y = fmaf(p.y, wt, o.y);
            o.z = fmaf(p.z, wt, o.z);
            o.w = fmaf(p.w, wt, o.w);
        }
        reinterpret_cast<float4 *>(a.part_acc + (pbase + int64_t(hh) * a.nparts) * D)[j4] = o;
    }

    // ---- the runs merged in order: by a second launch, or by the last CTA ---------
    if (a.defer_merge) return;  // the kernel's end publishes the state to the merge launch
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        uint32_t *ticket = a.tickets + int64_t(b) * a.kv_heads + kvh;
        sm.last = atomicAdd(ticket, 1u) == uint32_t(used - 1);
        if (sm.last) *ticket = 0u;  // leave the ticket clean for the next call
    }
    __syncthreads();
    if (!sm.last) return;
    __threadfence();
    merge_runs<D, GQ, kThreads>(a, b, kvh, used, sm.pw, sm.l_fin);
}

template <int D, int GQ, Src kSrc>
cudaError_t launch_attend_t(const AttendArgs &a, cudaStream_t s, bool pdl)
{
    const size_t smem = sizeof(AttendSmem<D, GQ>);
    static bool attr_done[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(attend_kernel<D, GQ, kSrc>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    static long long resident[64] = {};  // CTAs of this kernel the GPU holds at once
    if (resident[dev] == 0) {
        int n = 0, per_sm = 0;
        cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, attend_kernel<D, GQ, kSrc>, kThreads, smem);
        if (e != cudaSuccess) return e;
        resident[dev] = (long long)(n > 0 ? n : 1) * (per_sm > 0 ? per_sm : 1);
    }
    const dim3 grid(kParts, unsigned(a.kv_heads), unsigned(a.batch));
    // In a grid of more than one wave every CTA would hold its SM through the
    // merge's fence and ticket, so the runs' states are merged by a second
    // launch instead (same arithmetic, same bits).
    AttendArgs ad = a;
    ad.defer_merge = (long long)kParts * a.kv_heads * a.batch > resident[dev] ? 1 : 0;
    cudaError_t e = launch_kernel(attend_kernel<D, GQ, kSrc>, grid, dim3(kThreads), smem, s, pdl, ad);
    if (e != cudaSuccess || !ad.defer_merge) return e;
    return launch_kernel(attend_merge_kernel<D, GQ>, dim3(unsigned(a.kv_heads), unsigned(a.batch)),
                         dim3(kMergeThreads), 0, s, true, ad);
}

template <int D, Src kSrc>
cudaError_t launch_attend_d(const AttendArgs &a, cudaStream_t s, bool pdl)
{
    const int gq = a.q_heads / a.kv_heads;
    if (gq <= 1) return launch_attend_t<D, 1, kSrc>(a, s, pdl);
    if (gq <= 2) return launch_attend_t<D, 2, kSrc>(a, s, pdl);
    if (gq <= 4) return launch_attend_t<D, 4, kSrc>(a, s, pdl);
    if (gq <= 8) return launch_attend_t<D, 8, kSrc>(a, s, pdl);
    return launch_attend_t<D, 16, kSrc>(a, s, pdl);
}

template <int D>
cudaError_t launch_attend_src(const AttendArgs &a, cudaStream_t s, bool pdl)
{
    if (a.k_cache == nullptr) return launch_attend_d<D, Src::kScratch>(a, s, pdl);
    if (a.k_scr_out == nullptr) return launch_attend_d<D, Src::kCache>(a, s, pdl);
    return launch_attend_d<D, Src::kCacheStore>(a, s, pdl);
}

static_assert(sizeof(AttendSmem<128, 16>) <= 227 * 1024, "shared memory per CTA");
static_assert(2 * (sizeof(AttendSmem<128, 8>) + 1024) <= 228 * 1024, "two CTAs per SM up to GQ = 8");
static_assert(kRowsPerPart <= kThreads, "one thread per row of the run resolves it");
static_assert(kParts * kRowsPerPart >= kGroup * QSA_MAX_BUDGET + kGroup - 1, "runs cover the longest row");
static_assert(kRowsPerPart % kStepRows == 0, "runs are whole steps");

template <int D, int GQ>
constexpr bool layout_ok()
{
    using S = AttendSmem<D, GQ>;
    return offsetof(S, k) % 16 == 0 && offsetof(S, v) % 16 == 0 && offsetof(S, q) % 16 == 0 &&
           offsetof(S, pt) % 16 == 0 && offsetof(S, alpha) % 16 == 0 && offsetof(S, off) % 8 == 0 &&
           (D * 4) % 16 == 0 && offsetof(S, v) == offsetof(S, k) + sizeof(S::k) &&
           sizeof(S::k) + sizeof(S::v) >= size_t(kWarps) * GQ * D * 4;  // room for the reduction
}
static_assert(layout_ok<64, 1>() && layout_ok<64, 2>() && layout_ok<64, 4>() && layout_ok<64, 8>() &&
                  layout_ok<64, 16>() && layout_ok<128, 1>() && layout_ok<128, 2>() && layout_ok<128, 4>() &&
                  layout_ok<128, 8>() && layout_ok<128, 16>(),
              "16-byte alignment of every float4 / async-copy array");

}  // namespace

bool attend_shape_supported(int head_dim, int q_heads, int kv_heads)
{
    if (head_dim != 64 && head_dim != 128) return false;
    if (kv_heads <= 0 || q_heads <= 0 || q_heads % kv_heads != 0) return false;
    return q_heads / kv_heads <= kMaxGqa;
}

cudaError_t launch_merge_states(const float *m, const float *l, const float *acc, float *out, int n_parts,
                                int bh, int head_dim, cudaStream_t s)
{
    const int f4 = head_dim / 4;
    const long long n = (long long)bh * f4;
    if (n == 0) return cudaSuccess;
    const unsigned grid = unsigned((n + kMergeThreads - 1) / kMergeThreads);
    merge_states_kernel<<<grid, kMergeThreads, 0, s>>>(m, l, acc, out, n_parts, bh, f4);
    return cudaGetLastError();
}

cudaError_t launch_attend(const AttendArgs &a, cudaStream_t s, bool pdl)
{
    if (a.batch == 0) return cudaSuccess;
    if (a.head_dim == 128) return launch_attend_src<128>(a, s, pdl);
    if (a.head_dim == 64) return launch_attend_src<64>(a, s, pdl);
    return cudaErrorInvalidValue;
}

}  // namespace qsa
