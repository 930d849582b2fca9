// api.cu — the C ABI declared in include/gbattn.h: argument validation,
// TMA tensor-map encoding and kernel dispatch.  Nothing here allocates,
// frees or synchronises; every launch goes on the caller's stream.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "internal.h"

namespace gbattn {
namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int npad_of(int N) { return ((N + kTileRows - 1) / kTileRows) * kTileRows; }

// Checks shared by every entry point that takes a shape.
attn_status check_shape(int B, int H, int N, int d, attn_dtype dtype, bool backward) {
    if (B < 1 || H < 1 || N < 1) return ATTN_ERR_INVALID_ARG;
    if (dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_FP32 && dtype != ATTN_DTYPE_FP16 &&
        dtype != ATTN_DTYPE_FP8_E4M3)
        return ATTN_ERR_INVALID_ARG;
    if (d != 64 && d != 128 && d != 256) return ATTN_ERR_UNSUPPORTED;
    if (d == 256 && dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_FP16)
        return ATTN_ERR_UNSUPPORTED;   // head dim 256: 16-bit types
    if (dtype == ATTN_DTYPE_FP32 && (backward || d != 64)) return ATTN_ERR_UNSUPPORTED;
    if (dtype == ATTN_DTYPE_FP8_E4M3 && (backward || d != 128)) return ATTN_ERR_UNSUPPORTED;
    const long long elems = static_cast<long long>(B) * H * npad_of(N) * d;
    if (elems >= (1LL << 31)) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

// Key length of cross-attention: K and V (and dK, dV) hold Nk rows a head.
attn_status check_keys(int B, int H, int Nk, int d) {
    if (Nk < 1) return ATTN_ERR_INVALID_ARG;
    const long long elems = static_cast<long long>(B) * H * npad_of(Nk) * d;
    if (elems >= (1LL << 31)) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

attn_status check_math(float scale, float dropout_p) {
    if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
    if (!(dropout_p >= 0.f && dropout_p < 1.f)) return ATTN_ERR_INVALID_ARG;
    return ATTN_OK;
}

// Threshold on a 16-bit dropout draw: floor(p * 2^16), clamped to 2^16 - 1.
uint32_t drop_threshold(float p) {
    if (!(p > 0.f)) return 0u;
    const double t = std::floor(static_cast<double>(p) * 65536.0);
    return t >= 65535.0 ? 0xFFFFu : static_cast<uint32_t>(t);
}

struct Workspace {
    float* lse2;
    float* Drow;
    float* dq_acc;
};

size_t workspace_bytes_of(int B, int H, int N, int d) {
    const size_t rows = static_cast<size_t>(B) * H * npad_of(N);
    return rows * (2 + static_cast<size_t>(d)) * sizeof(float);
}

Workspace carve(void* ws, int B, int H, int N) {
    const size_t rows = static_cast<size_t>(B) * H * npad_of(N);
    float* base = static_cast<float*>(ws);
    return Workspace{base, base + rows, base + 2 * rows};
}

attn_status check_workspace(const void* ws, size_t bytes, int B, int H, int N, int d) {
    if (ws == nullptr || bytes < workspace_bytes_of(B, H, N, d)) return ATTN_ERR_WORKSPACE;
    if (!aligned16(ws)) return ATTN_ERR_MISALIGNED;
    return ATTN_OK;
}

attn_status from_cuda(cudaError_t e) { return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA; }

}  // namespace

namespace {

cuuint64_t elem_bytes(attn_dtype dtype) {
    return dtype == ATTN_DTYPE_FP32 ? 4 : (dtype == ATTN_DTYPE_FP8_E4M3 ? 1 : 2);
}

bool encode_3d(CUtensorMap* map, const void* ptr, attn_dtype dtype, const cuuint64_t dims[3],
               const cuuint64_t strides[2], const cuuint32_t box[3]) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = encode_fn();
    if (enc == nullptr) return false;
    const cuuint32_t estr[3] = {1, 1, 1};
    CUtensorMapDataType ty = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
    if (dtype == ATTN_DTYPE_FP32) ty = CU_TENSOR_MAP_DATA_TYPE_FLOAT32;
    if (dtype == ATTN_DTYPE_FP16) ty = CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (dtype == ATTN_DTYPE_FP8_E4M3) ty = CU_TENSOR_MAP_DATA_TYPE_UINT8;   // bytes moved as they are
    const CUresult r = enc(map, ty, 3, const_cast<void*>(ptr), dims, strides, box, estr,
                           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

}  // namespace

int fwd_tiles(int d, attn_dtype dtype, int N) {
    if (d > 128) return 1;
    if (dtype != ATTN_DTYPE_BF16 && dtype != ATTN_DTYPE_FP16) return 2;
    const char* env = std::getenv("GBATTN_FWD_TILES");
    if (env != nullptr && (env[0] == '1' || env[0] == '2') && env[1] == '\0') return env[0] - '0';
    // Measured on GB300: at d = 64 with short sequences (N = 512, 1024) one
    // tile per CTA is as fast or faster (more, shorter CTAs balance better and
    // two CTAs per SM overlap one's start-up with the other's work); with
    // long sequences or d = 128 two tiles sharing each K/V block win.
    return (d == 64 && N <= 2048) ? 1 : 2;
}

bool make_tmap_bhnd(CUtensorMap* map, const void* ptr, attn_dtype dtype, int BH, int N, int d,
                    int rows) {
    const cuuint64_t es = elem_bytes(dtype);
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                static_cast<cuuint64_t>(BH)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * es,
                                   static_cast<cuuint64_t>(N) * d * es};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(rows), 1};
    return encode_3d(map, ptr, dtype, dims, strides, box);
}

bool make_tmap_thd(CUtensorMap* map, const void* ptr, attn_dtype dtype, int T, int H, int d,
                   int rows) {
    const cuuint64_t es = elem_bytes(dtype);
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(H),
                                static_cast<cuuint64_t>(T)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * es,
                                   static_cast<cuuint64_t>(H) * d * es};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / es), 1, static_cast<cuuint32_t>(rows)};
    return encode_3d(map, ptr, dtype, dims, strides, box);
}

namespace {

// Map over one activation tensor: [B*H][N][d] when dense, [T][H][d] when
// packed; boxes of `rows` rows.
bool make_tmap(CUtensorMap* map, const void* ptr, attn_dtype dtype, int B, const SeqLayout& l,
               int d, int rows = kTileRows) {
    return l.cu ? make_tmap_thd(map, ptr, dtype, l.total, l.H, d, rows)
                : make_tmap_bhnd(map, ptr, dtype, B * l.H, l.N, d, rows);
}

// Checks of the packed-sequence entry points, on top of those of the dense
// ones with N = max_seqlen_q and Nk = max_seqlen_k.
attn_status check_varlen(const int32_t* cu_q, const int32_t* cu_k, int B, int H, int total_q,
                         int total_k, int max_q, int max_k, int d, attn_dtype dtype,
                         bool backward) {
    if (cu_q == nullptr || cu_k == nullptr) return ATTN_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(cu_q) & 3u) || (reinterpret_cast<uintptr_t>(cu_k) & 3u))
        return ATTN_ERR_MISALIGNED;
    if (total_q < 1 || total_k < 1 || max_q < 1 || max_k < 1) return ATTN_ERR_INVALID_ARG;
    attn_status st = check_shape(B, H, max_q, d, dtype, backward);
    if (st != ATTN_OK) return st;
    if ((st = check_keys(B, H, max_k, d)) != ATTN_OK) return st;
    if (dtype == ATTN_DTYPE_FP32) return ATTN_ERR_UNSUPPORTED;   // packed: 16- and 8-bit types
    if (static_cast<long long>(total_q) * H * d >= (1LL << 31) ||
        static_cast<long long>(total_k) * H * d >= (1LL << 31))
        return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

// The forward for validated shapes.
attn_status fwd_impl(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                     const SeqLayout& lq, const SeqLayout& lk, int d, attn_dtype dtype,
                     float scale, int causal, int window, const int32_t* key_lens,
                     float dropout_p, uint64_t seed, int* dev_status, void* stream) {
    attn_status st = check_math(scale, dropout_p);
    if (st != ATTN_OK) return st;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(LSE))
        return ATTN_ERR_MISALIGNED;
    CUtensorMap tq, tk, tv;
    if (!make_tmap(&tq, Q, dtype, B, lq, d) || !make_tmap(&tk, K, dtype, B, lk, d) ||
        !make_tmap(&tv, V, dtype, B, lk, d))
        return ATTN_ERR_CUDA;
    FwdParams p{};
    p.V = V;
    p.O = O;
    p.LSE = LSE;
    p.key_lens = key_lens;
    p.dev_status = dev_status;
    p.B = B;
    p.H = lq.H;
    p.N = lq.N;
    p.Nk = lk.N;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.out_scale = 1.0f / (1.0f - dropout_p);
    p.drop_threshold = drop_threshold(dropout_p);
    p.seed_lo = static_cast<uint32_t>(seed & 0xFFFFFFFFu);
    p.seed_hi = static_cast<uint32_t>(seed >> 32);
    p.window = window > 0 ? window : 0;
    p.lq = lq;
    p.lk = lk;
    return from_cuda(launch_fwd(tq, tk, tv, p, d, dtype, causal != 0, dropout_p > 0.f,
                                fwd_tiles(d, dtype, lq.N), static_cast<cudaStream_t>(stream)));
}

attn_status pre_impl(const void* O, const void* dO, const float* LSE, int B, const SeqLayout& lq,
                     int d, attn_dtype dtype, void* workspace, void* stream) {
    if (!aligned16(O) || !aligned16(dO) || !aligned16(LSE)) return ATTN_ERR_MISALIGNED;
    const Workspace w = carve(workspace, B, lq.H, lq.N);
    return from_cuda(launch_bwd_pre(O, dO, LSE, w.lse2, w.Drow, w.dq_acc, B * lq.H, lq,
                                    npad_of(lq.N), d, dtype == ATTN_DTYPE_FP16,
                                    static_cast<cudaStream_t>(stream)));
}

attn_status main_impl(const void* Q, const void* K, const void* V, const void* dO, void* dK,
                      void* dV, int B, const SeqLayout& lq, const SeqLayout& lk, int d,
                      attn_dtype dtype, float scale, int causal, int window,
                      const int32_t* key_lens, float dropout_p, uint64_t seed, void* workspace,
                      int* dev_status, void* stream) {
    attn_status st = check_math(scale, dropout_p);
    if (st != ATTN_OK) return st;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(dO) || !aligned16(dK) ||
        !aligned16(dV))
        return ATTN_ERR_MISALIGNED;
    // head dim 256 walks 64-row query blocks: Q and dO boxes of 64 rows
    const int qrows = d == 256 ? 64 : kTileRows;
    CUtensorMap tq, tk, tv, tdo, tdk, tdv;
    if (!make_tmap(&tq, Q, dtype, B, lq, d, qrows) || !make_tmap(&tk, K, dtype, B, lk, d) ||
        !make_tmap(&tv, V, dtype, B, lk, d) || !make_tmap(&tdo, dO, dtype, B, lq, d, qrows) ||
        !make_tmap(&tdk, dK, dtype, B, lk, d) || !make_tmap(&tdv, dV, dtype, B, lk, d))
        return ATTN_ERR_CUDA;
    const Workspace w = carve(workspace, B, lq.H, lq.N);
    BwdParams p{};
    p.dK = dK;
    p.dV = dV;
    p.key_lens = key_lens;
    p.dev_status = dev_status;
    p.dq_acc = w.dq_acc;
    p.lse2 = w.lse2;
    p.Drow = w.Drow;
    p.B = B;
    p.H = lq.H;
    p.N = lq.N;
    p.Nk = lk.N;
    p.Npad = npad_of(lq.N);
    p.nkb = (lk.N + kTileRows - 1) / kTileRows;
    p.scale_log2 = scale * 1.4426950408889634f;
    p.scale = scale;
    p.drop_scale = 1.0f / (1.0f - dropout_p);
    p.drop_threshold = drop_threshold(dropout_p);
    p.seed_lo = static_cast<uint32_t>(seed & 0xFFFFFFFFu);
    p.seed_hi = static_cast<uint32_t>(seed >> 32);
    p.window = window > 0 ? window : 0;
    p.lq = lq;
    p.lk = lk;
    if (d == 256)
        return from_cuda(launch_bwd_main_d256(tq, tk, tv, tdo, tdk, tdv, p,
                                              dtype == ATTN_DTYPE_FP16, causal != 0,
                                              dropout_p > 0.f, static_cast<cudaStream_t>(stream)));
    return from_cuda(launch_bwd_main(tq, tk, tv, tdo, tdk, tdv, p, d, dtype == ATTN_DTYPE_FP16,
                                     causal != 0, dropout_p > 0.f,
                                     static_cast<cudaStream_t>(stream)));
}

attn_status convert_impl(void* dQ, int B, const SeqLayout& lq, int d, attn_dtype dtype,
                         float scale, const void* workspace, void* stream) {
    if (!aligned16(dQ)) return ATTN_ERR_MISALIGNED;
    const Workspace w = carve(const_cast<void*>(workspace), B, lq.H, lq.N);
    return from_cuda(launch_bwd_dq_convert(dQ, w.dq_acc, B * lq.H, lq, npad_of(lq.N), d,
                                           dtype == ATTN_DTYPE_FP16, scale,
                                           static_cast<cudaStream_t>(stream)));
}

// The whole backward for validated shapes: every argument is checked before
// the first launch so that errors leave the outputs untouched.
attn_status bwd_impl(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* LSE, void* dQ, void* dK, void* dV, int B, const SeqLayout& lq,
                     const SeqLayout& lk, int d, attn_dtype dtype, float scale, int causal,
                     int window, const int32_t* key_lens, float dropout_p, uint64_t seed,
                     void* workspace, size_t workspace_bytes, int* dev_status, void* stream) {
    attn_status st = check_math(scale, dropout_p);
    if (st != ATTN_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, B, lq.H, lq.N, d)) != ATTN_OK) return st;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) ||
        !aligned16(LSE) || !aligned16(dQ) || !aligned16(dK) || !aligned16(dV))
        return ATTN_ERR_MISALIGNED;
    if ((st = pre_impl(O, dO, LSE, B, lq, d, dtype, workspace, stream)) != ATTN_OK) return st;
    if ((st = main_impl(Q, K, V, dO, dK, dV, B, lq, lk, d, dtype, scale, causal, window, key_lens,
                        dropout_p, seed, workspace, dev_status, stream)) != ATTN_OK)
        return st;
    return convert_impl(dQ, B, lq, d, dtype, scale, workspace, stream);
}

SeqLayout dense(int H, int N) { return SeqLayout{nullptr, H, N, 0}; }

}  // namespace

attn_status check_bwd_args(const void* Q, const void* K, const void* V, const void* O,
                           const void* dO, const float* LSE, const void* dQ, const void* dK,
                           const void* dV, int B, int H, int N, int Nk, int d, attn_dtype dtype,
                           float scale, float dropout_p) {
    if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV) return ATTN_ERR_INVALID_ARG;
    attn_status st = check_shape(B, H, N, d, dtype, true);
    if (st != ATTN_OK) return st;
    if ((st = check_keys(B, H, Nk, d)) != ATTN_OK) return st;
    if ((st = check_math(scale, dropout_p)) != ATTN_OK) return st;
    if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(O) || !aligned16(dO) ||
        !aligned16(LSE) || !aligned16(dQ) || !aligned16(dK) || !aligned16(dV))
        return ATTN_ERR_MISALIGNED;
    return ATTN_OK;
}

}  // namespace gbattn

using namespace gbattn;

extern "C" {

attn_status attn_fwd(const void* Q, const void* K, const void* V, void* O, float* LSE, int B,
                     int H, int N, int Nk, int d, attn_dtype dtype, float scale, int causal,
                     int window, const int32_t* key_lens, float dropout_p, uint64_t seed,
                     int* dev_status, void* stream) {
    if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
    attn_status st = check_shape(B, H, N, d, dtype, false);
    if (st != ATTN_OK) return st;
    if ((st = check_keys(B, H, Nk, d)) != ATTN_OK) return st;
    return fwd_impl(Q, K, V, O, LSE, B, dense(H, N), dense(H, Nk), d, dtype, scale, causal, window,
                    key_lens, dropout_p, seed, dev_status, stream);
}

attn_status attn_fwd_varlen(const void* Q, const void* K, const void* V, void* O, float* LSE,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B, int H,
                            int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                            attn_dtype dtype, float scale, int causal, int window,
                            float dropout_p, uint64_t seed, int* dev_status, void* stream) {
    if (!Q || !K || !V || !O || !LSE) return ATTN_ERR_INVALID_ARG;
    const attn_status st = check_varlen(cu_seqlens_q, cu_seqlens_k, B, H, total_q, total_k,
                                        max_seqlen_q, max_seqlen_k, d, dtype, false);
    if (st != ATTN_OK) return st;
    return fwd_impl(Q, K, V, O, LSE, B, SeqLayout{cu_seqlens_q, H, max_seqlen_q, total_q},
                    SeqLayout{cu_seqlens_k, H, max_seqlen_k, total_k}, d, dtype, scale, causal,
                    window, nullptr, dropout_p, seed, dev_status, stream);
}

size_t attn_bwd_workspace_size(int B, int H, int N, int d) {
    if (check_shape(B, H, N, d, ATTN_DTYPE_BF16, true) != ATTN_OK) return 0;
    return workspace_bytes_of(B, H, N, d);
}

attn_status attn_bwd_preprocess(const void* O, const void* dO, const float* LSE, int B, int H,
                                int N, int d, attn_dtype dtype, void* workspace,
                                size_t workspace_bytes, void* stream) {
    if (!O || !dO || !LSE) return ATTN_ERR_INVALID_ARG;
    attn_status st = check_shape(B, H, N, d, dtype, true);
    if (st != ATTN_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, B, H, N, d)) != ATTN_OK) return st;
    return pre_impl(O, dO, LSE, B, dense(H, N), d, dtype, workspace, stream);
}

attn_status attn_bwd_main(const void* Q, const void* K, const void* V, const void* dO, void* dK,
                          void* dV, int B, int H, int N, int Nk, int d, attn_dtype dtype,
                          float scale, int causal, int window, const int32_t* key_lens,
                          float dropout_p, uint64_t seed, void* workspace,
                          size_t workspace_bytes, int* dev_status, void* stream) {
    if (!Q || !K || !V || !dO || !dK || !dV) return ATTN_ERR_INVALID_ARG;
    attn_status st = check_shape(B, H, N, d, dtype, true);
    if (st != ATTN_OK) return st;
    if ((st = check_keys(B, H, Nk, d)) != ATTN_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, B, H, N, d)) != ATTN_OK) return st;
    return main_impl(Q, K, V, dO, dK, dV, B, dense(H, N), dense(H, Nk), d, dtype, scale, causal,
                     window, key_lens, dropout_p, seed, workspace, dev_status, stream);
}

attn_status attn_bwd_dq_convert(void* dQ, int B, int H, int N, int d, attn_dtype dtype,
                                float scale, const void* workspace, size_t workspace_bytes,
                                void* stream) {
    if (!dQ) return ATTN_ERR_INVALID_ARG;
    attn_status st = check_shape(B, H, N, d, dtype, true);
    if (st != ATTN_OK) return st;
    if ((st = check_math(scale, 0.f)) != ATTN_OK) return st;
    if ((st = check_workspace(workspace, workspace_bytes, B, H, N, d)) != ATTN_OK) return st;
    return convert_impl(dQ, B, dense(H, N), d, dtype, scale, workspace, stream);
}

attn_status attn_bwd(const void* Q, const void* K, const void* V, const void* O, const void* dO,
                     const float* LSE, void* dQ, void* dK, void* dV, int B, int H, int N, int Nk,
                     int d, attn_dtype dtype, float scale, int causal, int window,
                     const int32_t* key_lens, float dropout_p, uint64_t seed, void* workspace,
                     size_t workspace_bytes, int* dev_status, void* stream) {
    const attn_status st = check_bwd_args(Q, K, V, O, dO, LSE, dQ, dK, dV, B, H, N, Nk, d, dtype,
                                          scale, dropout_p);
    if (st != ATTN_OK) return st;
    return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B, dense(H, N), dense(H, Nk), d, dtype, scale,
                    causal, window, key_lens, dropout_p, seed, workspace, workspace_bytes,
                    dev_status, stream);
}

attn_status attn_bwd_varlen(const void* Q, const void* K, const void* V, const void* O,
                            const void* dO, const float* LSE, void* dQ, void* dK, void* dV,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int B, int H,
                            int total_q, int total_k, int max_seqlen_q, int max_seqlen_k, int d,
                            attn_dtype dtype, float scale, int causal, int window,
                            float dropout_p, uint64_t seed, void* workspace,
                            size_t workspace_bytes, int* dev_status, void* stream) {
    if (!Q || !K || !V || !O || !dO || !LSE || !dQ || !dK || !dV) return ATTN_ERR_INVALID_ARG;
    const attn_status st = check_varlen(cu_seqlens_q, cu_seqlens_k, B, H, total_q, total_k,
                                        max_seqlen_q, max_seqlen_k, d, dtype, true);
    if (st != ATTN_OK) return st;
    return bwd_impl(Q, K, V, O, dO, LSE, dQ, dK, dV, B,
                    SeqLayout{cu_seqlens_q, H, max_seqlen_q, total_q},
                    SeqLayout{cu_seqlens_k, H, max_seqlen_k, total_k}, d, dtype, scale, causal,
                    window, nullptr, dropout_p, seed, workspace, workspace_bytes, dev_status,
                    stream);
}

const char* attn_status_string(attn_status status) {
    switch (status) {
        case ATTN_OK: return "ok";
        case ATTN_ERR_INVALID_ARG: return "invalid argument";
        case ATTN_ERR_UNSUPPORTED: return "unsupported head dimension, dtype or pass";
        case ATTN_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
        case ATTN_ERR_WORKSPACE: return "workspace missing or too small";
        case ATTN_ERR_CUDA: return "CUDA runtime or driver call failed";
        case ATTN_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

int attn_version(void) { return 200; }

}  // extern "C"
