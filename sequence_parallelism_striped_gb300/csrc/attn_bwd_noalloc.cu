// attn_bwd_noalloc.cu -- striped_attn_bwd for callers that cannot allocate.
//
// striped_attn_bwd needs a device workspace (the fp32 dQ accumulator and the
// per-row Delta values) that the caller allocates.  Some callers cannot do
// that: a host application that owns every byte of device memory through its
// own allocator or a fixed memory budget and has no way to hand the library
// an extra buffer, or a training loop that must not call cudaMalloc on its
// hot path because the call can synchronise the device and can fail under
// memory pressure.  For them this file keeps the workspace in a fixed
// file-scope device array, so striped_attn_bwd_noalloc allocates nothing.
//
// The array (kNoAllocScratchBytes) exists on every GPU that loads the
// library, for as long as the library stays loaded.  All calls on a device
// share it, so calls that overlap on that GPU (different streams, or host
// threads racing on one device) corrupt each other's results.  It keeps
// whatever the previous call left; the backward's first kernel rewrites
// every statistic it later reads and zeroes the dQ accumulator itself.
#include <mutex>

#include "internal.h"

namespace striped {

// 48 MiB: enough for B*H*S rows with D = 128 up to about 96,000 rows (e.g.
// the short-sequence workload B=1, H=8, S=8192), and for fp32 heads of any D.
constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the scratch array on the current device, looked up once
// per device with that device current (the host-side symbol is only a
// stand-in, never a device address).  The address belongs to the device's
// context: after cudaDeviceReset() it would be stale, and the library is
// not to be used on a reset device again (see striped.h).  Returns a
// status code.
static int noalloc_scratch(void **out) {
    static std::mutex mu;
    static void *cache[256] = {nullptr};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev < 0 || dev >= 256) return STRIPED_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess) return cuda_status(e);
        cache[dev] = ptr;
    }
    *out = cache[dev];
    return STRIPED_OK;
}

}  // namespace striped

extern "C" int striped_attn_bwd_noalloc(const void *q, const void *k, const void *v, const void *o,
                                        const float *lse, const void *dO, void *dq, void *dk, void *dv,
                                        int64_t B, int64_t H, int64_t S, int64_t D, int N, int layout,
                                        int dtype, float scale, int64_t *tile_stats, void *stream) {
    using namespace striped;
    const size_t need = striped_workspace_size(B, H, S, D, N, dtype);
    if (need > kNoAllocScratchBytes) return STRIPED_ERR_WORKSPACE;  // problem too large for the array
    void *scratch = nullptr;
    const int st = noalloc_scratch(&scratch);
    if (st != STRIPED_OK) return st;
    return striped_attn_bwd(q, k, v, o, lse, dO, dq, dk, dv, scratch, kNoAllocScratchBytes, B, H, S, D, N,
                            layout, dtype, scale, tile_stats, stream);
}
