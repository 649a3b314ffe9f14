// noalloc.cu -- the attention stage without a caller-provided workspace.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: a
// plugin loaded into a host runtime that owns every byte of device memory
// and forbids allocations by third-party code, or a latency-critical loop
// that must not allocate once it is running.  For them,
// qsa_attend_noalloc runs the same attention kernel as qsa_attend, but its
// scratch (error word, merge tickets, chunk partials) lives in one
// file-scope device array of a fixed size, loaded with the library.  The
// caller still owns and passes every input and output.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so the first call on each device, with that
// device current, asks the runtime for the array's device address with
// cudaGetSymbolAddress and keeps it.  That first call should therefore come
// before any stream capture.  The kept address is valid for as long as the
// device's context lives: after a cudaDeviceReset the device code may load at
// another address, so the call is not for use after a reset.  All calls
// share the array: the counters that must start at zero are cleared on the
// stream at every call, and calls that overlap on the GPU race with each
// other.
#include <cuda_runtime.h>

#include <mutex>

#include "qsa_internal.cuh"

namespace qsa {
namespace {

constexpr size_t kStaticScratchBytes = QSA_ATTEND_NOALLOC_SCRATCH_BYTES;  // held by every device until exit

static __device__ __align__(256) unsigned char g_attend_scratch[kStaticScratchBytes];

struct StaticLayout {
    size_t off_err, off_tickets, off_part_m, off_part_l, off_part_acc, header_bytes, total;
};

StaticLayout static_layout(const qsa_dims *d, int32_t nparts_per_head)
{
    StaticLayout L{};
    const size_t B = size_t(d->batch);
    const size_t nparts = B * size_t(d->q_heads) * size_t(nparts_per_head);
    size_t off = 0;
    L.off_err = off;
    off += kWsAlign;
    L.off_tickets = off;
    off = align_up(off + B * size_t(d->kv_heads) * 4, kWsAlign);
    L.header_bytes = off;
    L.off_part_m = off;
    off = align_up(off + nparts * 4, kWsAlign);
    L.off_part_l = off;
    off = align_up(off + nparts * 4, kWsAlign);
    L.off_part_acc = off;
    off = align_up(off + nparts * size_t(d->head_dim) * 4, kWsAlign);
    L.total = off;
    return L;
}

std::mutex g_setup_mu;
void *g_scratch_addr[64] = {};

// Device address of the static scratch on the current device (set up once).
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_setup_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attend_scratch);
        if (e != cudaSuccess) return e;
        if (p == nullptr) return cudaErrorInvalidSymbol;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace
}  // namespace qsa

using namespace qsa;

extern "C" qsa_status qsa_attend_noalloc(const qsa_dims *dims, const float *q, const float *k_scr,
                                         const float *v_scr, const int32_t *n_ids, float *out,
                                         void *stream)
{
    if (!dims_valid(dims)) return QSA_ERR_INVALID_ARG;
    if (!attend_shape_supported(dims->head_dim, dims->q_heads, dims->kv_heads))
        return QSA_ERR_UNSUPPORTED_SHAPE;
    if (!q || !k_scr || !v_scr || !n_ids || !out) return QSA_ERR_INVALID_ARG;
    const uintptr_t a16 = reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k_scr) |
                          reinterpret_cast<uintptr_t>(v_scr);
    if ((a16 & 15u) != 0 || (reinterpret_cast<uintptr_t>(n_ids) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(out) & 15u) != 0)
        return QSA_ERR_INVALID_ARG;
    const Layout W = make_layout(dims);  // row capacity and chunk count, as qsa_attend
    const StaticLayout L = static_layout(dims, W.nparts);
    if (L.total > kStaticScratchBytes) return QSA_ERR_WORKSPACE_TOO_SMALL;  // beyond the fixed maximum
    if (dims->batch == 0) return QSA_OK;

    void *base = nullptr;
    if (scratch_address(&base) != cudaSuccess) return QSA_ERR_CUDA;
    unsigned char *s = static_cast<unsigned char *>(base);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // The previous call's error word and tickets may linger: clear them.
    if (cudaMemsetAsync(s, 0, L.header_bytes, st) != cudaSuccess) return QSA_ERR_CUDA;
    AttendArgs a{q, k_scr, v_scr, n_ids, out,
                 reinterpret_cast<float *>(s + L.off_part_m), reinterpret_cast<float *>(s + L.off_part_l),
                 reinterpret_cast<float *>(s + L.off_part_acc), reinterpret_cast<uint32_t *>(s + L.off_tickets),
                 W.row_cap, W.nparts, dims->batch, dims->q_heads, dims->kv_heads, dims->head_dim,
                 dims->scale, reinterpret_cast<uint32_t *>(s + L.off_err)};
    return launch_attend(a, st) == cudaSuccess ? QSA_OK : QSA_ERR_CUDA;
}
