// attn_bwd.cu — backward of the fused exact attention for sm_103a.
//
// Three launches:
//   preprocess  D_i = dO_i . O_i, -LSE_i * log2(e) into a padded workspace,
//               and a cleared fp32 dQ accumulator;
//   main        one CTA per (head, 128-key block): recomputes P tile by tile
//               from Q, K and the stored log-sum-exp (the recomputation of
//               "Why FlashAttention Is a Kernel Story", "When it falls down"),
//               accumulates dK, dV in tensor memory and adds dQ partials into
//               the workspace;
//   dq_convert  dQ = scale * accumulator, rounded to the output type.
// The main kernel is in attn_bwd_kernel.cuh; its packed-sequence
// instantiations are compiled in attn_bwd_packed.cu.
#include "attn_bwd_kernel.cuh"

namespace gbattn {
namespace {

constexpr float kLog2e = 1.4426950408889634f;

// D_i = dO_i . O_i and lse2_i = -LSE_i log2(e) for every padded row, and the
// row's fp32 dQ accumulator cleared.  Rows past the sequence's end (and rows
// whose LSE is -inf, which have no valid key) get lse2 = -inf so that the
// main kernel's P = exp2(s + lse2) is exactly 0 there; for packed sequences
// this also cancels the next sequence's rows that a tile load brings in.
// The workspace is [B*H][Npad] rows whatever the placement of O, dO, LSE.
//
// Bandwidth layout: a row is handled by D / 8 consecutive threads, each
// loading 16 bytes (8 elements) of O and of dO and clearing 32 bytes of the
// accumulator; every thread covers kPreRows rows, whose loads are all issued
// before the first product so that enough bytes are in flight.
constexpr int kPreThreads = 256;
constexpr int kPreRows = 2;

template <int D, bool kF16>
__global__ void __launch_bounds__(kPreThreads) bwd_pre_kernel(const uint16_t* __restrict__ O,
                                                              const uint16_t* __restrict__ dO,
                                                              const float* __restrict__ LSE,
                                                              float* __restrict__ lse2,
                                                              float* __restrict__ Drow,
                                                              float* __restrict__ dq_acc, int BH,
                                                              const SeqLayout lq, int Npad) {
    // O and LSE come from the kernel before.  The main kernel is let in only
    // after this wait: it loads Q, K, V and dO before its own wait, and may do
    // so only once every grid before this one has completed.
    grid_dep_wait();
    grid_dep_launch_dependents();
    constexpr int TPR = D / 8;                          // threads per row
    constexpr int ROWS_PER_PASS = kPreThreads / TPR;    // rows one pass of the block covers
    const int sub = threadIdx.x % TPR;                  // 8-element slice of the row
    const long long total = static_cast<long long>(BH) * Npad;
    long long prow[kPreRows];
    uint4 a[kPreRows], g[kPreRows];
#pragma unroll
    for (int k = 0; k < kPreRows; ++k) {
        prow[k] = (static_cast<long long>(blockIdx.x) * kPreRows + k) * ROWS_PER_PASS + threadIdx.x / TPR;
        a[k] = make_uint4(0, 0, 0, 0);
        g[k] = make_uint4(0, 0, 0, 0);
        if (prow[k] < total) {
            const int bh = static_cast<int>(prow[k] / Npad);
            const int row = static_cast<int>(prow[k] % Npad);
            int h;
            const SeqSpan sq = seq_span_bh(lq, bh, h);
            if (row < sq.len) {
                const size_t off = act_offset(lq, bh, h, sq.start, row, D) + 8 * sub;
                a[k] = *reinterpret_cast<const uint4*>(O + off);
                g[k] = *reinterpret_cast<const uint4*>(dO + off);
            }
        }
    }
#pragma unroll
    for (int k = 0; k < kPreRows; ++k) {
        const uint32_t av[4] = {a[k].x, a[k].y, a[k].z, a[k].w};
        const uint32_t gv[4] = {g[k].x, g[k].y, g[k].z, g[k].w};
        float acc = 0.f;
#pragma unroll
        for (int e = 0; e < 4; ++e)
            acc += h2lo_to_f32<kF16>(av[e]) * h2lo_to_f32<kF16>(gv[e]) +
                   h2hi_to_f32<kF16>(av[e]) * h2hi_to_f32<kF16>(gv[e]);
#pragma unroll
        for (int off = TPR / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (prow[k] >= total) continue;
        float4* qa = reinterpret_cast<float4*>(dq_acc + static_cast<size_t>(prow[k]) * D + 8 * sub);
        qa[0] = make_float4(0.f, 0.f, 0.f, 0.f);
        qa[1] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (sub == 0) {
            const int bh = static_cast<int>(prow[k] / Npad);
            const int row = static_cast<int>(prow[k] % Npad);
            int h;
            const SeqSpan sq = seq_span_bh(lq, bh, h);
            float nl2 = -INFINITY;   // -LSE log2e; -inf: the row takes no part
            if (row < sq.len) {
                const float lse = LSE[rowval_offset(lq, bh, h, sq.start, row)];
                if (lse != -INFINITY) nl2 = -lse * kLog2e;
            }
            lse2[prow[k]] = nl2;
            Drow[prow[k]] = acc;
        }
    }
}

// dQ = scale * acc for the rows of every sequence, walking the
// [B*H][Npad][D] workspace in groups of 8 elements (two 16-byte loads, one
// 16-byte store).  A thread takes kConvGroups groups 256 groups apart (each
// warp access stays one contiguous kilobyte) and issues all their loads
// before the first store; the workspace is read once, with the evict-first
// hint.  One group per thread (many small blocks) was the fastest: 2, 4 and
// 8 groups took 6% longer and more at the 4 x 16 x 4096 x 128 shape, up to
// 20% longer at the short-sequence shapes.
constexpr int kConvGroups = 1;

template <bool kF16>
__global__ void __launch_bounds__(256) bwd_dq_convert_kernel(uint16_t* __restrict__ dQ,
                                                             const float* __restrict__ dq_acc,
                                                             long long n8, const SeqLayout lq,
                                                             int Npad, int D, float scale) {
    grid_dep_launch_dependents();
    grid_dep_wait();   // the accumulator is complete once the main kernel is
    const long long g0 = static_cast<long long>(blockIdx.x) * (256 * kConvGroups) + threadIdx.x;
    float4 x[kConvGroups], y[kConvGroups];
#pragma unroll
    for (int u = 0; u < kConvGroups; ++u) {
        const long long i8 = g0 + 256 * u;
        if (i8 < n8) {
            const float4* src = reinterpret_cast<const float4*>(dq_acc + i8 * 8);
            x[u] = __ldcs(src);
            y[u] = __ldcs(src + 1);
        }
    }
#pragma unroll
    for (int u = 0; u < kConvGroups; ++u) {
        const long long i8 = g0 + 256 * u;
        if (i8 >= n8) break;
        const long long e = i8 * 8;                 // element index in [BH][Npad][D]
        const long long rowg = e / D;               // bh * Npad + row
        const int c = static_cast<int>(e % D);
        const int bh = static_cast<int>(rowg / Npad);
        const int row = static_cast<int>(rowg % Npad);
        int h;
        const SeqSpan sq = seq_span_bh(lq, bh, h);
        if (row >= sq.len) continue;
        uint4 out;
        out.x = pack_h2<kF16>(x[u].x * scale, x[u].y * scale);
        out.y = pack_h2<kF16>(x[u].z * scale, x[u].w * scale);
        out.z = pack_h2<kF16>(y[u].x * scale, y[u].y * scale);
        out.w = pack_h2<kF16>(y[u].z * scale, y[u].w * scale);
        *reinterpret_cast<uint4*>(dQ + act_offset(lq, bh, h, sq.start, row, D) + c) = out;
    }
}

template <int D, bool kF16>
void launch_pre_t(unsigned grid, const void* O, const void* dO, const float* LSE, float* lse2,
                  float* Drow, float* dq_acc, int BH, const SeqLayout& lq, int Npad,
                  cudaStream_t stream) {
    launch_overlapped(bwd_pre_kernel<D, kF16>, grid, kPreThreads, 0, stream,
                      static_cast<const uint16_t*>(O), static_cast<const uint16_t*>(dO), LSE, lse2,
                      Drow, dq_acc, BH, lq, Npad);
}

}  // namespace

cudaError_t launch_bwd_pre(const void* O, const void* dO, const float* LSE, float* lse2,
                           float* Drow, float* dq_acc, int BH, const SeqLayout& lq, int Npad,
                           int d, bool f16, cudaStream_t stream) {
    const long long rows = static_cast<long long>(BH) * Npad;
    const int rows_per_block = (kPreThreads / (d / 8)) * kPreRows;
    const unsigned grid = static_cast<unsigned>((rows + rows_per_block - 1) / rows_per_block);
    if (d == 64) {
        if (f16) launch_pre_t<64, true>(grid, O, dO, LSE, lse2, Drow, dq_acc, BH, lq, Npad, stream);
        else launch_pre_t<64, false>(grid, O, dO, LSE, lse2, Drow, dq_acc, BH, lq, Npad, stream);
    } else if (d == 128) {
        if (f16) launch_pre_t<128, true>(grid, O, dO, LSE, lse2, Drow, dq_acc, BH, lq, Npad, stream);
        else launch_pre_t<128, false>(grid, O, dO, LSE, lse2, Drow, dq_acc, BH, lq, Npad, stream);
    } else if (d == 256) {
        if (f16) launch_pre_t<256, true>(grid, O, dO, LSE, lse2, Drow, dq_acc, BH, lq, Npad, stream);
        else launch_pre_t<256, false>(grid, O, dO, LSE, lse2, Drow, dq_acc, BH, lq, Npad, stream);
    } else {
        return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

cudaError_t launch_bwd_dq_convert(void* dQ, const float* dq_acc, int BH, const SeqLayout& lq,
                                  int Npad, int d, bool f16, float scale, cudaStream_t stream) {
    const long long n8 = static_cast<long long>(BH) * Npad * d / 8;
    const unsigned grid = static_cast<unsigned>((n8 + 256 * kConvGroups - 1) / (256 * kConvGroups));
    if (f16)
        return launch_overlapped(bwd_dq_convert_kernel<true>, grid, 256, 0, stream,
                                 static_cast<uint16_t*>(dQ), dq_acc, n8, lq, Npad, d, scale);
    return launch_overlapped(bwd_dq_convert_kernel<false>, grid, 256, 0, stream,
                             static_cast<uint16_t*>(dQ), dq_acc, n8, lq, Npad, d, scale);
}

cudaError_t launch_bwd_main(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                            const BwdParams& p, int d, bool f16, bool causal, bool dropout,
                            cudaStream_t stream) {
    if (p.lq.cu != nullptr)
        return launch_bwd_main_packed(tq, tk, tv, tdo, tdk, tdv, p, d, f16, causal, dropout, stream);
    if (d == 64)
        return f16 ? dispatch_bwd<64, true, false>(tq, tk, tv, tdo, tdk, tdv, p, causal, dropout, stream)
                   : dispatch_bwd<64, false, false>(tq, tk, tv, tdo, tdk, tdv, p, causal, dropout, stream);
    if (d == 128)
        return f16 ? dispatch_bwd<128, true, false>(tq, tk, tv, tdo, tdk, tdv, p, causal, dropout, stream)
                   : dispatch_bwd<128, false, false>(tq, tk, tv, tdo, tdk, tdv, p, causal, dropout, stream);
    return cudaErrorInvalidValue;
}

}  // namespace gbattn
