// selftest.cu — device self-tests of the failure detection every kernel relies
// on, run without a fault:
//  * attn_selftest_wait: a warp waits on an mbarrier that nobody (or, for the
//    control case, one thread) arrives on.  No copy, tensor-memory allocation
//    or MMA is involved, so the expired wait leaves nothing in flight.
//  * attn_selftest_fwd_withheld: the fused forward kernel itself, with its
//    producer withholding one K tile (the copy is never issued, so nothing
//    ever completes that tile's barrier) and a short wait limit, so that a
//    wait expires while other copies and MMAs are in flight and the kernel's
//    own abort path (drain its copies and MMAs, free tensor memory, report
//    ATTN_ERR_DEVICE_TIMEOUT) runs on the GPU.
#include "attn_fwd_kernel.cuh"

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

extern "C" attn_status attn_selftest_fwd_withheld(const void* Q, const void* K, const void* V,
                                                  void* O, float* LSE, int B, int H, int N,
                                                  int Nk, int withhold_block, int wait_ms,
                                                  int* dev_status, void* stream) {
    using namespace gbattn;
    if (!Q || !K || !V || !O || !LSE || dev_status == nullptr) return ATTN_ERR_INVALID_ARG;
    if (B < 1 || H < 1 || N < 1 || Nk < 1 || wait_ms < 1 || wait_ms > 2000)
        return ATTN_ERR_INVALID_ARG;
    if (static_cast<long long>(B) * H * (N > Nk ? N : Nk) * 128 >= (1LL << 31))
        return ATTN_ERR_UNSUPPORTED;
    for (const void* ptr : {Q, K, V, static_cast<const void*>(O), static_cast<const void*>(LSE)})
        if ((reinterpret_cast<uintptr_t>(ptr) & 15u) != 0) return ATTN_ERR_MISALIGNED;
    CUtensorMap tq, tk, tv;
    if (!make_tmap_bhnd(&tq, Q, ATTN_DTYPE_BF16, B * H, N, 128) ||
        !make_tmap_bhnd(&tk, K, ATTN_DTYPE_BF16, B * H, Nk, 128) ||
        !make_tmap_bhnd(&tv, V, ATTN_DTYPE_BF16, B * H, Nk, 128))
        return ATTN_ERR_CUDA;
    FwdParams p{};
    p.V = V;
    p.O = O;
    p.LSE = LSE;
    p.key_lens = nullptr;
    p.dev_status = dev_status;
    p.B = B;
    p.H = H;
    p.N = N;
    p.Nk = Nk;
    p.scale_log2 = 0.08838834764831845f * 1.4426950408889634f;   // scale 1/sqrt(128)
    p.out_scale = 1.0f;
    p.lq = SeqLayout{nullptr, H, N, 0};
    p.lk = SeqLayout{nullptr, H, Nk, 0};
    p.withhold_block = withhold_block;
    p.wait_ns = static_cast<unsigned long long>(wait_ms) * 1000000ull;
    const cudaError_t e = launch_fwd_t<128, false, false, false, false, false, false, false, 2, true>(
        tq, tk, tv, p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}
