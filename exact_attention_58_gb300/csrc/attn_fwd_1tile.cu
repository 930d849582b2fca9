// attn_fwd_1tile.cu — forward launches with one 128-row query tile per CTA
// (two CTAs per SM) for bf16 and fp16 inputs with d in {64, 128}: dense
// tensors and packed sequences.  Compiled apart from the two-tile
// instantiations so that the two compile in parallel.
#include "attn_fwd_kernel.cuh"

namespace gbattn {

cudaError_t launch_fwd_1tile(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdParams& p, int d, attn_dtype dtype, bool causal, bool dropout,
                             cudaStream_t stream) {
    const bool f16 = dtype == ATTN_DTYPE_FP16;
    if (d == 64)
        return f16 ? dispatch_mask<64, false, true, false, false, 1>(tq, tk, tv, p, causal, dropout, stream)
                   : dispatch_mask<64, false, false, false, false, 1>(tq, tk, tv, p, causal, dropout, stream);
    if (d == 128)
        return f16 ? dispatch_mask<128, false, true, false, false, 1>(tq, tk, tv, p, causal, dropout, stream)
                   : dispatch_mask<128, false, false, false, false, 1>(tq, tk, tv, p, causal, dropout, stream);
    return cudaErrorInvalidValue;
}

cudaError_t launch_fwd_packed_1tile(const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const FwdParams& p, int d,
                                    attn_dtype dtype, bool causal, bool dropout,
                                    cudaStream_t stream) {
    const bool f16 = dtype == ATTN_DTYPE_FP16;
    if (d == 64)
        return f16 ? dispatch_mask<64, false, true, false, true, 1>(tq, tk, tv, p, causal, dropout, stream)
                   : dispatch_mask<64, false, false, false, true, 1>(tq, tk, tv, p, causal, dropout, stream);
    if (d == 128)
        return f16 ? dispatch_mask<128, false, true, false, true, 1>(tq, tk, tv, p, causal, dropout, stream)
                   : dispatch_mask<128, false, false, false, true, 1>(tq, tk, tv, p, causal, dropout, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gbattn
