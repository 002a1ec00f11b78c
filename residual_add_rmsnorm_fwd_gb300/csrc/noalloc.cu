// noalloc.cu -- rmsnorm_bwd_noalloc: the backward for callers that cannot
// allocate device memory.
//
// rmsnorm_bwd needs a scratch buffer for the per-CTA dweight partials, and
// expects the caller to allocate it.  Some callers cannot: a serving engine
// that reserves all device memory at start-up and forbids allocation on the
// request path, a plugin interface that hands an operator only its input and
// output buffers, or code on a latency-critical path where a cudaMalloc
// (which may synchronise the device) is not acceptable.  This entry point
// takes the scratch from a fixed array that lives in the library's own
// device memory instead, so the call allocates nothing.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (kNoAllocScratchBytes) until the process exits.  Host code
// cannot use the array's name as a device address, so the first call on each
// device looks the address up with cudaGetSymbolAddress (that device being
// current) and caches it; that first call should therefore come before any
// stream capture.  All calls share the array and it keeps the last call's
// contents; the backward kernels overwrite every partial they later read, so
// nothing needs clearing between calls, but two calls whose kernels overlap
// on the GPU (different streams, no ordering between them) race on it.
#include <mutex>

#include "../../include/rmsnorm.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;   // 16 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's copy of the scratch array (looked up once).
// A device other than an sm_103 one is refused first, with the status the
// other entry points give, before its copy of the array is looked up.
int scratch_for_current_device(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return RMSN_ERR_UNSUPPORTED;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return RMSN_ERR_CUDA;
    if (major != 10 || minor != 3) return RMSN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) return RMSN_ERR_CUDA;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return RMSN_OK;
}

}  // namespace

extern "C" __attribute__((visibility("default"))) int rmsnorm_bwd_noalloc(
    const void *dy, const void *x, const void *weight, const float *rrms, void *dx, float *dweight,
    int64_t row_stride, int64_t M, int64_t H, int dtype, int has_weight, void *stream) {
    void *scratch = nullptr;
    if (has_weight && dweight != nullptr && M > 0) {
        const int st = scratch_for_current_device(&scratch);
        if (st != RMSN_OK) return st;
    }
    // Same validation, kernels and launch as rmsnorm_bwd; a problem whose
    // partials do not fit the array fails there with RMSN_ERR_WORKSPACE.
    return rmsnorm_bwd(dy, x, weight, rrms, dx, dweight, scratch, scratch ? kNoAllocScratchBytes : 0, row_stride, M,
                       H, dtype, has_weight, stream);
}
