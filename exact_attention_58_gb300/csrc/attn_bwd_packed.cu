// attn_bwd_packed.cu — backward main-kernel launch for packed
// variable-length sequences ([T, H, d] tensors located by cumulative
// offsets); compiled apart from the dense instantiations.
#include "attn_bwd_kernel.cuh"

namespace gbattn {

cudaError_t launch_bwd_main_packed(const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const CUtensorMap& tdo,
                                   const CUtensorMap& tdk, const CUtensorMap& tdv,
                                   const BwdParams& p, int d, bool f16, bool causal, bool dropout,
                                   cudaStream_t stream) {
    if (d == 64)
        return f16 ? dispatch_bwd<64, true, true>(tq, tk, tv, tdo, tdk, tdv, p, causal, dropout, stream)
                   : dispatch_bwd<64, false, true>(tq, tk, tv, tdo, tdk, tdv, p, causal, dropout, stream);
    if (d == 128)
        return f16 ? dispatch_bwd<128, true, true>(tq, tk, tv, tdo, tdk, tdv, p, causal, dropout, stream)
                   : dispatch_bwd<128, false, true>(tq, tk, tv, tdo, tdk, tdv, p, causal, dropout, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gbattn
