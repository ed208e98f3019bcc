// rkv_noalloc.cu -- rkv_compress for callers that cannot hand the library a
// workspace allocation.
//
// Some callers have device pointers for their inputs and outputs but no way to
// obtain more device memory at the point of the call: code that runs while a CUDA
// graph is being captured (where cudaMalloc is not allowed), runtimes whose memory
// is owned by an arena or allocator the caller cannot reach, and serving loops that
// must not allocate after start-up.  For them the write path's scratch lives in a
// fixed array in the library's own device image, sized once at load time.
#include "rkv_internal.cuh"

namespace rkv {

// The scratch of rkv_compress_noalloc.  Every GPU that loads the library holds
// these bytes until the process exits.
constexpr size_t kNoAllocScratchBytes = (size_t)64 << 20;   // 64 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array, looked up once per device with that device current
// (thread-safe).  In host code the name g_noalloc_scratch is only a host-side
// stand-in, not a device address: only the looked-up address may reach a kernel.
static PerDevice<void *> g_scratch;

static cudaError_t scratch_address(void *&ptr)
{
    return per_device(g_scratch, ptr, [](void *&p) {
        p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e == cudaSuccess && p == nullptr) e = cudaErrorInvalidSymbol;
        return e;
    });
}

}  // namespace rkv

using namespace rkv;

extern "C" rkv_status rkv_compress_noalloc(const rkv_params *p, const void *kv,
                                           const rkv_ref_pool *pool, const void *W1t,
                                           const void *W2t, const void *W3t,
                                           const rkv_cache *cache, float *z_out,
                                           int32_t *dev_status, void *stream)
{
    size_t need = 0;
    rkv_status st = rkv_query_sizes(p, nullptr, nullptr, &need);
    if (st != RKV_OK) return st;
    if (need > kNoAllocScratchBytes) return RKV_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (scratch_address(scratch) != cudaSuccess || !scratch) return RKV_ERR_CUDA;
    return rkv_compress(p, kv, pool, W1t, W2t, W3t, cache, scratch, kNoAllocScratchBytes, z_out,
                        dev_status, stream);
}
