// attn_fwd_packed.cu — forward launch for packed variable-length sequences
// ([T, H, d] tensors located by cumulative offsets); 16-bit and e4m3 inputs.
#include "attn_fwd_kernel.cuh"

namespace gbattn {

cudaError_t launch_fwd_packed(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const FwdParams& p, int d, attn_dtype dtype, bool causal,
                              bool dropout, int tiles, cudaStream_t stream) {
    if (tiles == 1 && d <= 128 && (dtype == ATTN_DTYPE_BF16 || dtype == ATTN_DTYPE_FP16))
        return launch_fwd_packed_1tile(tq, tk, tv, p, d, dtype, causal, dropout, stream);
    switch (dtype) {
        case ATTN_DTYPE_BF16:
            if (d == 64) return dispatch_mask<64, false, false, false, true>(tq, tk, tv, p, causal, dropout, stream);
            if (d == 128) return dispatch_mask<128, false, false, false, true>(tq, tk, tv, p, causal, dropout, stream);
            if (d == 256) return dispatch_mask<256, false, false, false, true>(tq, tk, tv, p, causal, dropout, stream);
            return cudaErrorInvalidValue;
        case ATTN_DTYPE_FP16:
            if (d == 64) return dispatch_mask<64, false, true, false, true>(tq, tk, tv, p, causal, dropout, stream);
            if (d == 128) return dispatch_mask<128, false, true, false, true>(tq, tk, tv, p, causal, dropout, stream);
            if (d == 256) return dispatch_mask<256, false, true, false, true>(tq, tk, tv, p, causal, dropout, stream);
            return cudaErrorInvalidValue;
        case ATTN_DTYPE_FP8_E4M3:   // output in bf16
            if (d == 128) return dispatch_mask<128, false, false, true, true>(tq, tk, tv, p, causal, dropout, stream);
            return cudaErrorInvalidValue;
        default:
            return cudaErrorInvalidValue;
    }
}

}  // namespace gbattn
