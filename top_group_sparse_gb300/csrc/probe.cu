// probe.cu -- the binary32 FFMA rate of this GPU, measured in the process
// that measures the path, as the denominator of an FFMA-bound roofline.
//
// Each thread runs kChains independent chains a = fma(a, x, y); x and y are
// kernel arguments, so nothing folds, and x < 1 keeps every chain finite and
// away from subnormals.  kChains independent chains per thread and
// kProbeThreads * blocks_per_sm threads per SM cover the FMA latency.
#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr int kProbeThreads = 256;
constexpr int kChains = 8;
constexpr int kUnroll = 16;

__global__ void __launch_bounds__(kProbeThreads) ffma_probe_kernel(float *sink, int iters, float x, float y)
{
    float a[kChains];
#pragma unroll
    for (int c = 0; c < kChains; ++c) a[c] = float(threadIdx.x & 7) + float(c);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
#pragma unroll
            for (int c = 0; c < kChains; ++c) a[c] = __fmaf_rn(a[c], x, y);
        }
    }
    float s = 0.0f;
#pragma unroll
    for (int c = 0; c < kChains; ++c) s += a[c];
    if (s == 12345.0f) sink[blockIdx.x] = s;  // keeps the chains live; never true for x, y below
}

}  // namespace
}  // namespace qsa

using namespace qsa;

extern "C" qsa_status qsa_probe_ffma(int32_t blocks_per_sm, int32_t iters, float *sink, int64_t *fma_count,
                                     void *stream)
{
    if (blocks_per_sm <= 0 || blocks_per_sm > 8 || iters <= 0 || !sink || !fma_count) return QSA_ERR_INVALID_ARG;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
        return QSA_ERR_CUDA;
    const int grid = sms * blocks_per_sm;
    *fma_count = int64_t(grid) * kProbeThreads * int64_t(iters) * kUnroll * kChains;
    ffma_probe_kernel<<<grid, kProbeThreads, 0, static_cast<cudaStream_t>(stream)>>>(sink, iters, 0.9999999f,
                                                                                     1.0e-3f);
    return cudaGetLastError() == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}
