// gather.cu -- stage 3: slot resolution and compact K/V gather.
//
// "A sparse mask is not sparse attention" (AFN-016), Decision: the selected
// logical IDs are resolved through the shared slot map at one boundary --
// the only place where logical identity meets the physical cache layout --
// and only the selected K/V rows are copied into bounded contiguous scratch
// (Why compact gather comes before fusion).
//
// Row i of query b: s = slot_map[slot_offset[b] + ids[b][i]];
//   k_scr[b][i] = k_cache[s], v_scr[b][i] = v_cache[s]  (n_kv * d floats each).
// A pure copy, bound by HBM: each thread moves independent 16-byte pieces of
// K and V (several in flight per thread), consecutive threads take consecutive
// pieces of a row, so every row read and every scratch write is coalesced.
// An ID outside [0, T_b) or a slot outside [0, num_slots) zero-fills the row
// and sets a bit of the error word; nothing outside the buffers is read.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kThreads = 256;
constexpr int kPerThread = 4;  // 16-byte pieces of K (and of V) per thread

__global__ void __launch_bounds__(kThreads)
gather_kernel(const GatherArgs a)
{
    const int b = blockIdx.y;
    const int n = __ldcg(a.n_ids + b);
    const int T = __ldg(a.visible + b);
    if (n < 0 || n > a.row_cap) {
        if (blockIdx.x == 0 && threadIdx.x == 0) set_error(a.err, QSA_DEVERR_ROW_RANGE);
        return;
    }
    const int f4 = a.row_floats >> 2;  // 16-byte pieces per row
    const int64_t first = int64_t(blockIdx.x) * kThreads * kPerThread + threadIdx.x;
    const int64_t limit = int64_t(n) * f4;
    if (int64_t(blockIdx.x) * kThreads * kPerThread >= limit) return;

    const int32_t *ids = a.ids + int64_t(b) * a.row_cap;
    const int32_t *smap = a.slot_map + __ldg(a.slot_offset + b);
    const float4 *kc = reinterpret_cast<const float4 *>(a.k_cache);
    const float4 *vc = reinterpret_cast<const float4 *>(a.v_cache);
    float4 *ks = reinterpret_cast<float4 *>(a.k_scr) + int64_t(b) * a.row_cap * f4;
    float4 *vs = reinterpret_cast<float4 *>(a.v_scr) + int64_t(b) * a.row_cap * f4;

    float4 kv[kPerThread], vv[kPerThread];
    int64_t dst[kPerThread];
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
        const int64_t e = first + int64_t(u) * kThreads;
        dst[u] = -1;
        if (e >= limit) continue;
        const int i = int(e / f4);
        const int p = int(e - int64_t(i) * f4);
        const int id = __ldcg(ids + i);
        const bool id_ok = id >= 0 && id < T;
        const int64_t slot = id_ok ? int64_t(__ldg(smap + id)) : -1;
        dst[u] = e;
        if (slot < 0 || slot >= a.num_slots) {
            set_error(a.err, id_ok ? QSA_DEVERR_SLOT_RANGE : QSA_DEVERR_ROW_RANGE);
            kv[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            vv[u] = kv[u];
            continue;
        }
        kv[u] = __ldg(kc + slot * f4 + p);
        vv[u] = __ldg(vc + slot * f4 + p);
    }
#pragma unroll
    for (int u = 0; u < kPerThread; ++u) {
        if (dst[u] < 0) continue;
        ks[dst[u]] = kv[u];
        vs[dst[u]] = vv[u];
    }
}

}  // namespace

cudaError_t launch_gather(const GatherArgs &a, cudaStream_t s)
{
    if (a.batch == 0) return cudaSuccess;
    const int64_t pieces = int64_t(a.row_cap) * (a.row_floats >> 2);
    const int64_t per_block = int64_t(kThreads) * kPerThread;
    const dim3 grid(unsigned((pieces + per_block - 1) / per_block), unsigned(a.batch));
    gather_kernel<<<grid, kThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace qsa
