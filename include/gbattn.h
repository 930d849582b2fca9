/*
 * gbattn.h — C ABI of the fused exact-attention library (libgbattn.so).
 *
 * The library computes exact scaled-dot-product attention
 *
 *     O = dropout(softmax(scale * Q K^T + mask)) V
 *
 * on one GPU (sm_103a) as a single tiled kernel that never writes the N x N
 * score or probability matrix to device memory, and the matching backward
 * pass that recomputes the probabilities tile by tile from Q, K and the
 * stored log-sum-exp.  The operation is the attention chain of
 * anthology-of-the-sota practice SOTA-114 ("The general form of the practice
 * above it": matmul, scale, mask, softmax, dropout, matmul fused into one
 * kernel) computed with the online-softmax tiling of "Why FlashAttention Is a
 * Kernel Story" (section "Tiling: fitting the work inside SRAM"); the
 * backward's recomputation is the one that page describes under "When it falls
 * down" (backward-pass complexity).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  Layout     Q, O, dO, dQ are contiguous [B, H, N, d] arrays and K, V, dK,
 *             dV contiguous [B, H, Nk, d] arrays, d innermost (row-major), one
 *             element type for all of them (O is bf16 for e4m3 inputs).  N is the number of query rows and
 *             Nk the number of keys (Nk = N for self-attention).  LSE is a
 *             contiguous float [B, H, N] array.  key_lens is an int32 [B]
 *             array.  Every pointer is a DEVICE pointer.
 *  Alignment  Every tensor pointer must be 16-byte aligned
 *             (ATTN_ERR_MISALIGNED otherwise).
 *  Types      ATTN_DTYPE_BF16: bf16 storage, bf16 x bf16 products with fp32
 *             accumulation.  ATTN_DTYPE_FP16: the same with IEEE half
 *             storage and f16 x f16 products (P and dS are rounded to f16).
 *             ATTN_DTYPE_FP32: fp32 storage, TF32 products with fp32
 *             accumulation (forward only, d = 64).
 *             ATTN_DTYPE_FP8_E4M3: Q, K, V stored as e4m3 (OCP FP8, one byte,
 *             no infinities), e4m3 x e4m3 products with fp32 accumulation; P
 *             is rounded to e4m3 (nearest even) for the P V product while l
 *             and LSE use the unrounded P; O is written as bf16.  Forward
 *             only, d = 128.  Per-tensor scales of quantised inputs are the
 *             caller's: fold s_q * s_k into `scale` and multiply O by s_v.
 *  Shapes     d in {64, 128} (and 256 for the bf16 and fp16 forward);
 *             B, H, N, Nk >= 1; B*H*N*d and B*H*Nk*d
 *             < 2^31 elements per tensor.  Anything else returns ATTN_ERR_UNSUPPORTED or
 *             ATTN_ERR_INVALID_ARG: the library never falls back to another
 *             implementation.
 *  Mask       query i stands at key position p = i + Nk - N: with N != Nk the
 *             queries are the last N positions of the key sequence (p = i
 *             for self-attention).  Key j of sequence b is attended by query i
 *             iff j < key_lens[b] (all Nk keys when key_lens is NULL), when
 *             causal != 0, j <= p, and, when window > 0 (sliding-window
 *             attention), p - j < window and, unless causal, j - p < window;
 *             window <= 0 means no window.  Key blocks outside the mask are
 *             skipped, not computed and masked.  A query row with no valid key
 *             gets O = 0 and LSE = -inf (and zero gradients).  key_lens values
 *             outside [0, Nk] are clamped on the device and reported as
 *             ATTN_ERR_INVALID_ARG through dev_status.
 *  Scale      scale must be finite and > 0 (1/sqrt(d) is the usual choice).
 *  Dropout    0 <= dropout_p < 1.  Kept probabilities are multiplied by
 *             1/(1 - dropout_p); the softmax denominator and LSE use the
 *             undropped probabilities.  The keep bit of score (i, j) of head
 *             (b, h) comes from one 16-bit draw of Philox4x32-10 (Salmon et
 *             al., SC'11) at counter (i, j>>3, h, b) under key (lo32(seed),
 *             hi32(seed)): output word (j>>1)&3, its low half for even j and
 *             its high half for odd j.  The score is dropped iff that draw <
 *             floor(dropout_p * 2^16), so dropout_p acts rounded down to a
 *             multiple of 2^-16.
 *             attn_bwd must get the same dropout_p, seed, causal and key_lens
 *             as the attn_fwd whose O and LSE it is given.
 *  Ownership  The caller owns every buffer, including the workspace.  The
 *             library never allocates, frees or synchronises.
 *  Streams    stream is a cudaStream_t (NULL = the legacy default stream).
 *             Work is enqueued asynchronously; outputs are valid once the
 *             stream has reached the work.  Kernels are launched with
 *             programmatic stream serialization: a kernel's blocks may be
 *             resident before the work ahead of it in the stream has
 *             finished, but no kernel touches a buffer before every earlier
 *             piece of work that may use it has finished (griddepcontrol
 *             .wait); the three backward stages overlap one another's
 *             start-up.
 *  Errors     Argument errors are returned before anything is enqueued, with
 *             the outputs untouched.  A failed launch returns ATTN_ERR_CUDA.
 *             Errors detected on the device (a bounded wait that expired, an
 *             out-of-range key length) are written to *dev_status (a device
 *             int, 0 = OK) when dev_status is not NULL; the kernel then exits
 *             cleanly and leaves the affected outputs unspecified.
 *  Tuning     The forward runs two 128-row query tiles per CTA (one CTA per
 *             SM) or, for bf16 and fp16 with d <= 128, one tile per CTA (two
 *             CTAs per SM): one tile by default for d = 64 with N <= 2048,
 *             else two; the environment variable GBATTN_FWD_TILES ("1" or
 *             "2", read at each call) overrides the choice.  The result does
 *             not depend on it.
 *  Threads    Every entry point is thread-safe.
 *  Devices    One process may drive several GPUs: every call runs on the
 *             device current in the calling thread (cudaSetDevice), whose
 *             context gets its own one-time kernel set-up on first use, and
 *             all pointers of a call must be memory of that device.  The library must not outlive a reset of
 *             a device it has used (cudaDeviceReset): what it set up in the
 *             old context is not redone in the new one.
 */
#ifndef GBATTN_H
#define GBATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,    /* NULL pointer, bad size, scale, dropout_p or key length */
    ATTN_ERR_UNSUPPORTED = 2,    /* d, dtype or pass not built (never a silent fallback) */
    ATTN_ERR_MISALIGNED = 3,     /* a tensor pointer is not 16-byte aligned */
    ATTN_ERR_WORKSPACE = 4,      /* workspace NULL or smaller than attn_bwd_workspace_size */
    ATTN_ERR_CUDA = 5,           /* a CUDA runtime or driver call failed */
    ATTN_ERR_DEVICE_TIMEOUT = 6  /* (dev_status only) a bounded device-side wait expired */
} attn_status;

typedef enum {
    ATTN_DTYPE_BF16 = 0,
    ATTN_DTYPE_FP32 = 1,
    ATTN_DTYPE_FP16 = 2,
    ATTN_DTYPE_FP8_E4M3 = 3
} attn_dtype;

/*
 * Forward pass.
 *   Q         in   [B, H, N, d]
 *   K, V      in   [B, H, Nk, d]
 *   O         out  [B, H, N, d]  (same dtype as Q; bf16 for e4m3 Q, K, V)
 *   LSE       out  [B, H, N] float: natural log of the sum over valid keys of
 *                  exp(scale * q_i . k_j) (-inf for a row with no valid key)
 * One kernel launch.  Supported: bf16 and fp16 with d in {64, 128, 256}; fp32
 * (TF32 products) with d = 64; e4m3 with d = 128.
 */
attn_status attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE,
                     int B, int H, int N, int Nk, int d, attn_dtype dtype, float scale,
                     int causal, int window, const int32_t* key_lens, float dropout_p,
                     uint64_t seed, int* dev_status, void* stream);

/*
 * Bytes of device workspace attn_bwd needs: per head, the row terms
 * D_i = dO_i . O_i and the log-sum-exp in base 2 (two floats per row) and an
 * fp32 accumulator for dQ, with N (query rows) rounded up to a multiple of
 * 128.  It does not depend on Nk.  Returns 0 for arguments attn_bwd would
 * reject.
 */
size_t attn_bwd_workspace_size(int B, int H, int N, int d);

/*
 * Backward pass: given the forward's inputs, its O and LSE and the incoming
 * gradient dO, writes dQ ([B, H, N, d]) and dK, dV ([B, H, Nk, d]), in the
 * dtype of Q.  bf16 or fp16, d in {64, 128}.  workspace must hold
 * attn_bwd_workspace_size(B, H, N, d) bytes (16-byte aligned); its contents
 * on entry do not matter.  Enqueues
 * three launches: attn_bwd_preprocess, attn_bwd_main, attn_bwd_dq_convert.
 */
attn_status attn_bwd(const void* Q, const void* K, const void* V, const void* O,
                     const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                     int B, int H, int N, int Nk, int d, attn_dtype dtype, float scale,
                     int causal, int window, const int32_t* key_lens, float dropout_p,
                     uint64_t seed, void* workspace, size_t workspace_bytes, int* dev_status,
                     void* stream);

/*
 * The three stages of attn_bwd, exported so that a caller can enqueue (and
 * time) them one by one.  Same arguments and rules as attn_bwd; calling the
 * three in this order on one stream with one workspace is exactly attn_bwd.
 *   preprocess: D_i = dO_i . O_i and -LSE_i * log2(e) into the workspace;
 *               clears the dQ accumulator.
 *   main:       recomputes P tile by tile; writes dK, dV; accumulates dQ
 *               (unscaled) into the workspace.
 *   dq_convert: dQ = scale * accumulator, rounded to the output dtype.
 */
attn_status attn_bwd_preprocess(const void* O, const void* dO, const float* LSE,
                                int B, int H, int N, int d, attn_dtype dtype,
                                void* workspace, size_t workspace_bytes, void* stream);
attn_status attn_bwd_main(const void* Q, const void* K, const void* V, const void* dO,
                          void* dK, void* dV, int B, int H, int N, int Nk, int d,
                          attn_dtype dtype, float scale, int causal, int window,
                          const int32_t* key_lens, float dropout_p, uint64_t seed,
                          void* workspace, size_t workspace_bytes, int* dev_status, void* stream);
attn_status attn_bwd_dq_convert(void* dQ, int B, int H, int N, int d, attn_dtype dtype,
                                float scale, const void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * attn_bwd without a workspace argument, for callers that cannot allocate
 * device memory where they run the backward (a plugin inside a framework that
 * owns every device allocation and gives it no allocator, or latency-critical
 * code that must not call cudaMalloc).  The pages have no counterpart: this is
 * a deployment convenience, not part of the method.
 *   Scratch   a 32 MiB buffer inside the library (a file-scope __device__
 *             array), held by every GPU that loads the library until exit.
 *             Shapes whose attn_bwd_workspace_size exceeds 32 MiB are
 *             rejected with ATTN_ERR_WORKSPACE before anything is enqueued.
 *   Set-up    the first call on a device looks up the buffer's device address
 *             (cudaGetSymbolAddress) with that device current; make that first
 *             call before any stream capture.  The address is looked up again
 *             if the device's context has changed since (a device reset).
 *   Sharing   every call uses the same buffer; each call clears what must
 *             start at zero, but calls that overlap on the GPU race on it.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * Otherwise identical to attn_bwd (same arguments minus the workspace, same
 * results, same errors).  attn_bwd's argument errors are checked first; a
 * shape that passes them but needs more scratch than 32 MiB then returns
 * ATTN_ERR_WORKSPACE.
 */
attn_status attn_bwd_noalloc(const void* Q, const void* K, const void* V, const void* O,
                             const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                             int B, int H, int N, int Nk, int d, attn_dtype dtype, float scale,
                             int causal, int window, const int32_t* key_lens, float dropout_p,
                             uint64_t seed, int* dev_status, void* stream);

/*
 * Packed variable-length sequences (the layout of batches without padding):
 * the B sequences of a batch are concatenated along the token axis.
 *   Q, O, dO, dQ   [total_q, H, d]     K, V, dK, dV   [total_k, H, d]
 *   LSE            float [H, total_q]
 *   cu_seqlens_q   int32 [B + 1], DEVICE, 4-byte aligned: sequence b holds
 *                  query tokens [cu_seqlens_q[b], cu_seqlens_q[b+1]);
 *                  cu_seqlens_q[0] = 0 and cu_seqlens_q[B] = total_q.
 *   cu_seqlens_k   the same for the keys (may equal cu_seqlens_q).
 *   max_seqlen_q   an upper bound on every query length (sets the grid and
 *                  the workspace); max_seqlen_k the same for the keys.
 * Each sequence is attended on its own, with the mask of the dense entry
 * points applied to its lengths N_b = cu_q[b+1] - cu_q[b] and
 * Nk_b = cu_k[b+1] - cu_k[b] (queries are the last N_b key positions; no
 * key_lens).  The dropout counter is (i, j>>3, h, b) with i, j counted within
 * sequence b.  bf16 or fp16 only.  Offsets that leave [0, total], decrease,
 * or give a sequence longer than its max_seqlen are clamped on the device
 * (no access leaves the tensors) and reported as ATTN_ERR_INVALID_ARG through
 * dev_status.  attn_bwd_varlen's workspace holds
 * attn_bwd_workspace_size(B, H, max_seqlen_q, d) bytes.  Otherwise the
 * conventions above hold; one launch for the forward, three for the backward.
 */
attn_status attn_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int B, int H, int total_q, int total_k, int max_seqlen_q,
                            int max_seqlen_k, int d, attn_dtype dtype, float scale, int causal,
                            int window, float dropout_p, uint64_t seed, int* dev_status,
                            void* stream);
attn_status attn_bwd_varlen(const void* Q, const void* K, const void* V, const void* O,
                            const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int B, int H, int total_q, int total_k, int max_seqlen_q,
                            int max_seqlen_k, int d, attn_dtype dtype, float scale, int causal,
                            int window, float dropout_p, uint64_t seed, void* workspace,
                            size_t workspace_bytes, int* dev_status, void* stream);

/*
 * Device self-test of the failure detection the kernels rely on: one warp
 * waits on an mbarrier with the same bounded wait (about 2 s of
 * %globaltimer) that every kernel uses.  arrive != 0: one thread arrives
 * first, the wait succeeds and *dev_status is left as it is.  arrive == 0:
 * nothing arrives, the wait expires and ATTN_ERR_DEVICE_TIMEOUT is written to
 * *dev_status (a device int, 0 on entry).  Nothing else is in flight, so the
 * expiry leaves the context usable.  Not part of the attention path.
 */
attn_status attn_selftest_wait(int* dev_status, int arrive, void* stream);

/*
 * Device self-test of the fused forward kernel's own abort path.  It runs the
 * bf16, d = 128, non-causal forward (the kernel of attn_fwd, in a test
 * instantiation that only this entry point launches) on Q [B, H, N, 128] and
 * K, V [B, H, Nk, 128], with two changes: the producer never issues the copy
 * of the K tile of key block withhold_block (a tile withheld, not a fault:
 * nothing ever completes that tile's barrier), and every wait gives up after
 * wait_ms milliseconds (1 to 2000) instead of about 2 s.  A CTA that walks
 * that key block then has copies and MMAs in flight when its wait expires: it
 * drains them, frees its tensor memory, writes ATTN_ERR_DEVICE_TIMEOUT to
 * *dev_status (required, a device int, 0 on entry) and returns; O and LSE of
 * such CTAs are unspecified.  withhold_block < 0 withholds nothing and gives
 * the ordinary result.  Not part of the attention path.
 */
attn_status attn_selftest_fwd_withheld(const void* Q, const void* K, const void* V, void* O,
                                       float* LSE, int B, int H, int N, int Nk,
                                       int withhold_block, int wait_ms, int* dev_status,
                                       void* stream);

/* Static, NUL-terminated description of a status code. */
const char* attn_status_string(attn_status status);

/* Library version: major * 10000 + minor * 100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* GBATTN_H */
