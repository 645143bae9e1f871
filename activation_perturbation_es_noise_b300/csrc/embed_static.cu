// embed_static.cu -- the embedding scatter-add for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they need the embedding gradient: code running inside an allocator-free
// region of a host framework, a plugin whose host process owns every device
// allocation, or a hook that runs while the caller's memory pool is locked.
// dust_embed_scatter needs a caller-provided workspace; this entry point runs
// the same kernels on a fixed scratch area that lives in the library itself.
//
// The scratch is a file-scope __device__ array of kEmbedStaticScratchBytes
// (32 MiB; enough for 16384 tokens x 1536 channels over 4096 rows).  Every GPU
// that loads the library holds it until the process exits.  Its device address
// is looked up once per device and context (cudaGetSymbolAddress, with that
// device current) by the first call made there, so that first call should
// come before any stream capture; a call that finds a different context on
// the device (the primary context was reset and recreated) looks the address
// up again, since the module may then sit elsewhere.  Every call shares the
// one array, and the embedding pipeline clears the parts it needs zeroed on
// each call; two calls that overlap on the GPU (different streams, no
// ordering between them) race on it.
#include <mutex>

#include "dust_common.cuh"
#include "internal.h"

namespace dust {
namespace {

constexpr size_t kEmbedStaticScratchBytes = size_t(32) << 20;  // 32 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) uint8_t g_embed_scratch[kEmbedStaticScratchBytes];

void* g_scratch_addr[kMaxDevices];
void* g_scratch_ctx[kMaxDevices];  // the context the address was looked up in
std::mutex g_scratch_mutex;

// The driver's cuCtxGetCurrent, reached through the runtime (the library links
// no driver library of its own).
using CtxGetCurrentFn = int (*)(void**);
CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static bool tried = false;
    if (!tried) {
        tried = true;
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
        else
            (void)cudaGetLastError();
    }
    return fn;
}

// Device address of the scratch on the current device.  In host code the name
// g_embed_scratch is only a host-side handle, never a device address.
dust_status scratch_address(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return DUST_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return DUST_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    const CtxGetCurrentFn cur = ctx_get_current();
    if (!cur) return DUST_ERR_CUDA;
    void* ctx = nullptr;
    if (cur(&ctx) != 0) return DUST_ERR_CUDA;
    if (g_scratch_addr[dev] == nullptr || ctx == nullptr || g_scratch_ctx[dev] != ctx) {
        // (the lookup makes the device's primary context current if this
        // thread has none yet; the context is read again after it)
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_embed_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();
            return DUST_ERR_CUDA;
        }
        if (cur(&ctx) != 0 || ctx == nullptr) return DUST_ERR_CUDA;
        g_scratch_addr[dev] = p;
        g_scratch_ctx[dev] = ctx;
    }
    *out = g_scratch_addr[dev];
    return DUST_OK;
}

}  // namespace
}  // namespace dust

using namespace dust;

extern "C" dust_status dust_embed_scatter_static(const float* g_hat, const int32_t* ids,
                                                 int64_t T, int64_t d, int64_t V, float* G_E,
                                                 int32_t* perm_out, void* stream) {
    const size_t need = dust_embed_workspace(T, d, V);
    if (need == 0) return DUST_ERR_INVALID_ARG;
    if (need > kEmbedStaticScratchBytes) return DUST_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    const dust_status st = scratch_address(&scratch);
    if (st != DUST_OK) return st;
    return dust_embed_scatter(g_hat, ids, T, d, V, G_E, perm_out, scratch,
                              kEmbedStaticScratchBytes, stream);
}
