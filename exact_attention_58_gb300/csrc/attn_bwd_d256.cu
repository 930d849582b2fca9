// attn_bwd_d256.cu — backward main-kernel launches for head dim 256 (bf16,
// fp16; dense tensors and packed sequences).  The kernel is in
// attn_bwd_d256.cuh.
#include "attn_bwd_d256.cuh"

namespace gbattn {

cudaError_t launch_bwd_main_d256(const CUtensorMap& tq64, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo64,
                                 const CUtensorMap& tdk, const CUtensorMap& tdv,
                                 const BwdParams& p, bool f16, bool causal, bool dropout,
                                 cudaStream_t stream) {
    if (p.lq.cu != nullptr)
        return f16 ? dispatch_bwd_d256<true, true>(tq64, tk, tv, tdo64, tdk, tdv, p, causal, dropout, stream)
                   : dispatch_bwd_d256<false, true>(tq64, tk, tv, tdo64, tdk, tdv, p, causal, dropout, stream);
    return f16 ? dispatch_bwd_d256<true, false>(tq64, tk, tv, tdo64, tdk, tdv, p, causal, dropout, stream)
               : dispatch_bwd_d256<false, false>(tq64, tk, tv, tdo64, tdk, tdv, p, causal, dropout, stream);
}

}  // namespace gbattn
