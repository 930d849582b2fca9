// selftest.cu — a device self-test of the bounded waits every kernel relies on
// for failure detection: a warp waits on an mbarrier that nobody (or, for the
// control case, one thread) arrives on.  No copy, tensor-memory allocation or
// MMA is involved, so the expired wait leaves nothing in flight.
#include "internal.h"
#include "ptx.cuh"

namespace gbattn {
namespace {

__global__ void __launch_bounds__(32) wait_selftest_kernel(int* dev_status, int arrive) {
    __shared__ uint64_t bar;
    __shared__ volatile int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncwarp();
    if (arrive && threadIdx.x == 0) mbar_arrive(&bar);
    __syncwarp();
    const bool ok = mbar_wait_warp(&bar, 0, &abort_flag);
    if (threadIdx.x == 0 && dev_status != nullptr)
        atomicCAS(dev_status, 0, ok ? 0 : static_cast<int>(ATTN_ERR_DEVICE_TIMEOUT));
}

}  // namespace
}  // namespace gbattn

extern "C" attn_status attn_selftest_wait(int* dev_status, int arrive, void* stream) {
    if (dev_status == nullptr) return ATTN_ERR_INVALID_ARG;
    gbattn::wait_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev_status,
                                                                                 arrive);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
