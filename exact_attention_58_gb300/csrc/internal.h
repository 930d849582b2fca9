// internal.h — declarations shared by the C ABI layer and the kernel files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <utility>

#include "gbattn.h"

namespace gbattn {

// Rows per query / key tile (the MMA's M).
constexpr int kTileRows = 128;

// Where the rows of a sequence live.  Dense (cu == nullptr): activations
// [B, H, N, d] and per-row values (LSE) [B, H, N].  Packed sequences
// (cu != nullptr): the B sequences are concatenated along the token axis,
// activations [T, H, d] and per-row values [H, T]; sequence b holds tokens
// [cu[b], cu[b+1]), at most N of them.
struct SeqLayout {
    const int32_t* cu;        // B + 1 cumulative token offsets (device), or nullptr
    int H;
    int N;                    // dense: rows per head; packed: longest sequence allowed
    int total;                // packed: T tokens (unused when dense)
};

struct FwdParams {
    const void* V;            // read directly (not through TMA) on the fp32 path
    void* O;
    float* LSE;
    const int32_t* key_lens;
    int* dev_status;
    int B, H, N;              // N: query rows
    int Nk;                   // keys (N_k != N: cross-attention)
    int nqb;                  // query blocks of one forward CTA (set by the launch)
    float scale_log2;         // scale * log2(e)
    float out_scale;          // 1 / (1 - dropout_p)
    uint32_t drop_threshold;  // floor(p * 2^16), clamped to 2^16 - 1
    uint32_t seed_lo, seed_hi;
    int window;               // > 0: sliding window of this many keys
    SeqLayout lq, lk;         // query / key row placement (N, Nk are their N)
    // Read only by the self-test instantiation of the forward (see
    // attn_selftest_fwd_withheld): the key block whose K tile the producer
    // withholds, and the wait limit that replaces the default.
    int withhold_block;
    unsigned long long wait_ns;
};

struct BwdParams {
    void* dK;
    void* dV;
    const int32_t* key_lens;
    int* dev_status;
    float* dq_acc;            // [B*H][Npad][d] fp32
    const float* lse2;        // [B*H][Npad] -LSE * log2(e); -inf marks "no contribution"
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
    SeqLayout lq, lk;         // query / key row placement (N, Nk are their N)
};

// Dynamic shared memory above 48 KB has to be enabled for a kernel in each
// device's context before its first launch there.  `done` (one per kernel)
// remembers the devices already set up; the attribute call is idempotent, so
// two threads that race on the first launch both succeed.  Devices past the
// 64 bits of the mask set the attribute on every launch.
template <typename Kernel>
cudaError_t enable_smem_per_device(Kernel kern, int bytes, std::atomic<unsigned long long>& done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? (1ull << dev) : 0ull;
    if (bit != 0 && (done.load(std::memory_order_acquire) & bit) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit != 0) done.fetch_or(bit, std::memory_order_release);
    return e;
}

// Launch on `stream` with programmatic stream serialization, so that the
// kernel's CTAs may start (and run up to their grid_dep_wait()) while the
// kernel before it finishes.
template <typename... KArgs, typename... Args>
cudaError_t launch_overlapped(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                              cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// Tensor map over a contiguous [B*H][N][d] array, boxes of `rows` rows (128
// unless given) and 128 bytes along d, 128-byte swizzle.  Returns false if the
// driver rejected it.
bool make_tmap_bhnd(CUtensorMap* map, const void* ptr, attn_dtype dtype, int BH, int N, int d,
                    int rows = kTileRows);
// Tensor map over a contiguous [T][H][d] array (packed sequences) with the
// same boxes: `rows` consecutive tokens of one head, 128 bytes along d.
bool make_tmap_thd(CUtensorMap* map, const void* ptr, attn_dtype dtype, int T, int H, int d,
                   int rows = kTileRows);

// Every check attn_bwd makes before it looks at the workspace: NULL pointers,
// shape, key count, scale, dropout probability and 16-byte alignment, in that
// order, with attn_bwd's status codes.
attn_status check_bwd_args(const void* Q, const void* K, const void* V, const void* O,
                           const void* dO, const float* LSE, const void* dQ, const void* dK,
                           const void* dV, int B, int H, int N, int Nk, int d, attn_dtype dtype,
                           float scale, float dropout_p);

// Query tiles of 128 rows per forward CTA: 2 (the tiles share every K/V
// block; one CTA per SM) or 1 (two CTAs per SM).  Head dim 256, fp32 and e4m3
// inputs always take their one layout (1, 2 and 2 tiles).  For bf16 and fp16
// with d <= 128 the environment variable GBATTN_FWD_TILES ("1" or "2", read
// at each call) decides; without it, 1 for d = 64 with N <= 2048 query rows
// (the longest sequence when packed), else 2.
int fwd_tiles(int d, attn_dtype dtype, int N);

// Forward launch (validated arguments only) with `tiles` query tiles per CTA.
cudaError_t launch_fwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                       const FwdParams& p, int d, attn_dtype dtype, bool causal, bool dropout,
                       int tiles, cudaStream_t stream);

// The same for packed sequences (p.lq.cu != nullptr; bf16, fp16 or e4m3).
cudaError_t launch_fwd_packed(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const FwdParams& p, int d, attn_dtype dtype, bool causal,
                              bool dropout, int tiles, cudaStream_t stream);

// One query tile per CTA, bf16 or fp16 with d in {64, 128}: dense and packed.
cudaError_t launch_fwd_1tile(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                             const FwdParams& p, int d, attn_dtype dtype, bool causal, bool dropout,
                             cudaStream_t stream);
cudaError_t launch_fwd_packed_1tile(const CUtensorMap& tq, const CUtensorMap& tk,
                                    const CUtensorMap& tv, const FwdParams& p, int d,
                                    attn_dtype dtype, bool causal, bool dropout,
                                    cudaStream_t stream);

// Backward launches (validated arguments only).
// f16: the 16-bit tensors are IEEE half (else bf16).
// lq: placement of the query rows (O, dO, LSE); the workspace is
// [B*H][Npad] rows whatever the placement.
cudaError_t launch_bwd_pre(const void* O, const void* dO, const float* LSE, float* lse2,
                           float* Drow, float* dq_acc, int BH, const SeqLayout& lq, int Npad,
                           int d, bool f16, cudaStream_t stream);
// tdk / tdv: maps over the dK / dV outputs, written with TMA stores.
cudaError_t launch_bwd_main(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const BwdParams& p, int d, bool f16, bool causal, bool dropout,
                            cudaStream_t stream);
// The main launch for packed sequences (p.lq.cu != nullptr).
cudaError_t launch_bwd_main_packed(const CUtensorMap& tq, const CUtensorMap& tk,
                                   const CUtensorMap& tv, const CUtensorMap& tdo,
                                   const CUtensorMap& tdk, const CUtensorMap& tdv,
                                   const BwdParams& p, int d, bool f16, bool causal, bool dropout,
                                   cudaStream_t stream);
// The main launch at head dim 256 (dense or packed by p.lq.cu): Q and dO maps
// with 64-row boxes, the others with 128-row boxes.
cudaError_t launch_bwd_main_d256(const CUtensorMap& tq64, const CUtensorMap& tk,
                                 const CUtensorMap& tv, const CUtensorMap& tdo64,
                                 const CUtensorMap& tdk, const CUtensorMap& tdv,
                                 const BwdParams& p, bool f16, bool causal, bool dropout,
                                 cudaStream_t stream);
cudaError_t launch_bwd_dq_convert(void* dQ, const float* dq_acc, int BH, const SeqLayout& lq,
                                  int Npad, int d, bool f16, float scale, cudaStream_t stream);

}  // namespace gbattn
