// pooling.cuh -- the group pooling arithmetic and the pooled-tile layout,
// shared by every scorer of libqsa so that all of them pool bit for bit alike.
//
// "A sparse mask is not sparse attention" (AFN-016), Why a sparse mask can
// still be dense: the indexer pools each complete four-token group of raw
// index keys.  The pooled key is the mean in binary32 with one fixed order.
#pragma once

#include <cuda_runtime.h>

namespace qsa {

// p = (((k0 + k1) + k2) + k3) * 0.25 in binary32, round to nearest, per lane.
__device__ __forceinline__ float4 pool4(float4 k0, float4 k1, float4 k2, float4 k3)
{
    float4 p;
    p.x = __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(k0.x, k1.x), k2.x), k3.x), 0.25f);
    p.y = __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(k0.y, k1.y), k2.y), k3.y), 0.25f);
    p.z = __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(k0.z, k1.z), k2.z), k3.z), 0.25f);
    p.w = __fmul_rn(__fadd_rn(__fadd_rn(__fadd_rn(k0.w, k1.w), k2.w), k3.w), 0.25f);
    return p;
}

// Pooled tile layout in shared memory: group g's 16-byte chunk j4 sits at
// chunk (j4 ^ (g & 7)) of row g, so up to 8 groups read at the same chunk hit
// distinct banks.
template <int D>
__device__ __forceinline__ int pool_index(int g, int j4)
{
    return g * D + ((j4 ^ (g & 7)) << 2);
}

}  // namespace qsa
