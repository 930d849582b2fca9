// attn_fwd.cu — forward launch for dense [B, H, N, d] tensors (the kernel is
// in attn_fwd_kernel.cuh); packed sequences go to attn_fwd_packed.cu, whose
// instantiations compile in parallel with these.
#include "attn_fwd_kernel.cuh"

namespace gbattn {

cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int d, attn_dtype dtype, bool causal, bool dropout,
                       int tiles, cudaStream_t stream) {
    if (p.lq.cu != nullptr)
        return launch_fwd_packed(tq, tk, tv, p, d, dtype, causal, dropout, tiles, stream);
    if (tiles == 1 && d <= 128 && (dtype == ATTN_DTYPE_BF16 || dtype == ATTN_DTYPE_FP16))
        return launch_fwd_1tile(tq, tk, tv, p, d, dtype, causal, dropout, stream);
    switch (dtype) {
        case ATTN_DTYPE_FP32:
            if (d == 64) return dispatch_mask<64, true, false, false, false>(tq, tk, tv, p, causal, dropout, stream);
            return cudaErrorInvalidValue;
        case ATTN_DTYPE_BF16:
            if (d == 64) return dispatch_mask<64, false, false, false, false>(tq, tk, tv, p, causal, dropout, stream);
            if (d == 128) return dispatch_mask<128, false, false, false, false>(tq, tk, tv, p, causal, dropout, stream);
            if (d == 256) return dispatch_mask<256, false, false, false, false>(tq, tk, tv, p, causal, dropout, stream);
            return cudaErrorInvalidValue;
        case ATTN_DTYPE_FP16:
            if (d == 64) return dispatch_mask<64, false, true, false, false>(tq, tk, tv, p, causal, dropout, stream);
            if (d == 128) return dispatch_mask<128, false, true, false, false>(tq, tk, tv, p, causal, dropout, stream);
            if (d == 256) return dispatch_mask<256, false, true, false, false>(tq, tk, tv, p, causal, dropout, stream);
            return cudaErrorInvalidValue;
        case ATTN_DTYPE_FP8_E4M3:   // output in bf16
            if (d == 128) return dispatch_mask<128, false, false, true, false>(tq, tk, tv, p, causal, dropout, stream);
            return cudaErrorInvalidValue;
    }
    return cudaErrorInvalidValue;
}

}  // namespace gbattn
