// internal.h — declarations shared by the C ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

#include "gbattn.h"

namespace gbattn {

// Rows per query / key tile (the MMA's M) and per forward CTA (two tiles).
constexpr int kTileRows = 128;
constexpr int kFwdRowsPerCta = 2 * kTileRows;

struct FwdParams {
    const void* V;            // read directly (not through TMA) on the fp32 path
    void* O;
    float* LSE;
    const int32_t* key_lens;
    int* dev_status;
    int B, H, N;              // N: query rows
    int Nk;                   // keys (N_k != N: cross-attention)
    int nqb;                  // query blocks of kFwdRowsPerCta rows
    float scale_log2;         // scale * log2(e)
    float out_scale;          // 1 / (1 - dropout_p)
    uint32_t drop_threshold;  // floor(p * 2^32), clamped
    uint32_t seed_lo, seed_hi;
    int window;               // > 0: sliding window of this many keys
};

struct BwdParams {
    void* dK;
    void* dV;
    const int32_t* key_lens;
    int* dev_status;
    float* dq_acc;            // [B*H][Npad][d] fp32
    const float* lse2;        // [B*H][Npad] LSE * log2(e); +inf marks "no contribution"
    const float* Drow;        // [B*H][Npad] dO . O
    int B, H, N, Npad;        // N: query rows, Npad: N rounded up to 128
    int Nk;                   // keys
    int nkb;                  // key blocks of kTileRows rows
    float scale_log2;
    float scale;              // applied to dK
    float drop_scale;         // 1 / (1 - dropout_p)
    uint32_t drop_threshold;
    uint32_t seed_lo, seed_hi;
    int window;               // > 0: sliding window of this many keys
};

// Tensor map over a contiguous [B*H][N][d] array, 128-row boxes of 128 bytes
// along d, 128-byte swizzle.  Returns false if the driver rejected it.
bool make_tmap_bhnd(CUtensorMap* map, const void* ptr, attn_dtype dtype, int BH, int N, int d);

// Forward launch (validated arguments only).
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int d, attn_dtype dtype, bool causal, bool dropout,
                       cudaStream_t stream);

// Backward launches (validated arguments only).
// f16: the 16-bit tensors are IEEE half (else bf16).
cudaError_t launch_bwd_pre(const void* O, const void* dO, const float* LSE, float* lse2,
                           float* Drow, float* dq_acc, int BH, int N, int Npad, int d, bool f16,
                           cudaStream_t stream);
// tdk / tdv: maps over the dK / dV outputs, written with TMA stores.
cudaError_t launch_bwd_main(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const BwdParams& p, int d, bool f16, bool causal, bool dropout,
                            cudaStream_t stream);
cudaError_t launch_bwd_dq_convert(void* dQ, const float* dq_acc, int BH, int N, int Npad, int d,
                                  bool f16, float scale, cudaStream_t stream);

}  // namespace gbattn
