// noalloc.cu — attn_bwd_noalloc: the backward pass with its scratch held in a
// buffer that lives inside this library instead of a caller-supplied workspace.
//
// Who needs it: callers that cannot allocate device memory where they run the
// backward — for example a plugin inside a host framework that owns every
// device allocation and hands its plugins no allocator, or latency-critical
// code that must not call cudaMalloc (or any routine that allocates) on its hot
// path.  They pass inputs and outputs only; the library supplies the scratch.
//
// The scratch is one file-scope __device__ array of kNoAllocScratchBytes
// (32 MiB).  Every GPU that loads this library holds that memory until the
// process exits.  In host code the array's name is only a host-side stand-in,
// so its device address is looked up with cudaGetSymbolAddress, once per
// device, on the first call made on that device (with that device current);
// make that first call before any stream capture.  The address is kept per
// device together with the context it was looked up in, and looked up again
// when the device's current context has changed (after a device reset).  All
// calls share the one array: the backward clears what must start at zero (the
// dQ accumulator) on every call, but two calls that overlap on the GPU race on
// the array.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"

namespace gbattn {
namespace {

constexpr size_t kNoAllocScratchBytes = size_t(32) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};

// The CUDA driver API's cuCtxGetCurrent, reached through the runtime (no -lcuda).
CUresult current_context(CUcontext* ctx) {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(ptr);
    });
    return fn != nullptr ? fn(ctx) : CUDA_ERROR_NOT_FOUND;
}

// Device address of the scratch array on the current device, looked up once
// per (device, context).
attn_status scratch_on_current_device(void** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    // The runtime makes the device's primary context current on the first
    // runtime call, so look the address up first and read the context after.
    void* ptr = g_scratch_addr[dev];
    CUcontext ctx = nullptr;
    if (ptr != nullptr && (current_context(&ctx) != CUDA_SUCCESS || ctx != g_scratch_ctx[dev]))
        ptr = nullptr;
    if (ptr == nullptr) {
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return ATTN_ERR_CUDA;
        if (current_context(&ctx) != CUDA_SUCCESS) return ATTN_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
        g_scratch_ctx[dev] = ctx;
    }
    *out = ptr;
    return ATTN_OK;
}

}  // namespace
}  // namespace gbattn

extern "C" attn_status attn_bwd_noalloc(const void* Q, const void* K, const void* V,
                                        const void* O, const void* dO, const float* LSE,
                                        void* dQ, void* dK, void* dV, int B, int H, int N,
                                        int Nk, int d, attn_dtype dtype, float scale, int causal,
                                        int window,
                                        const int32_t* key_lens, float dropout_p, uint64_t seed,
                                        int* dev_status, void* stream) {
    // attn_bwd's own argument errors come first, before any CUDA call; only
    // then does a shape too large for the scratch give ATTN_ERR_WORKSPACE.
    const attn_status bad = gbattn::check_bwd_args(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, Nk,
                                                   d, dtype, scale, dropout_p);
    if (bad != ATTN_OK) return bad;
    const size_t need = attn_bwd_workspace_size(B, H, N, d);
    if (need == 0 || need > gbattn::kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE;
    void* scratch = nullptr;
    const attn_status st = gbattn::scratch_on_current_device(&scratch);
    if (st != ATTN_OK) return st;
    return attn_bwd(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, Nk, d, dtype, scale, causal, window,
                    key_lens, dropout_p, seed, scratch, gbattn::kNoAllocScratchBytes, dev_status,
                    stream);
}
