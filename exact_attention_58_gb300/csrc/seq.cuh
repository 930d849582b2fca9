// seq.cuh — device-side placement of a sequence's rows: dense [B, H, N, d]
// tensors or packed sequences [T, H, d] located by cumulative offsets.
#pragma once

#include "internal.h"

namespace gbattn {

struct SeqSpan {
    int start;   // first token of the sequence (packed), 0 when dense
    int len;     // rows of the sequence
};

// Token range of sequence b.  Offsets outside [0, T], decreasing offsets and
// sequences longer than L.N are clamped so that every access stays inside
// the tensors, and reported as ATTN_ERR_INVALID_ARG through dev_status when
// `report` is set.
__device__ __forceinline__ SeqSpan seq_span(const SeqLayout& L, int b, int* dev_status,
                                            bool report) {
    if (L.cu == nullptr) return {0, L.N};
    const int s0 = L.cu[b], s1 = L.cu[b + 1];
    const int a = min(max(s0, 0), L.total);
    const int e = min(max(s1, a), L.total);
    const int len = min(e - a, L.N);
    if (report && dev_status != nullptr && (a != s0 || e != s1 || e - a > L.N))
        atomicCAS(dev_status, 0, static_cast<int>(ATTN_ERR_INVALID_ARG));
    return {a, len};
}

// Span of the sequence of head row bh = b * H + h, and its head h (left 0
// when dense, where the offsets below need bh alone).  Reports nothing.
__device__ __forceinline__ SeqSpan seq_span_bh(const SeqLayout& L, int bh, int& h) {
    h = 0;
    if (L.cu == nullptr) return {0, L.N};
    const int b = bh / L.H;
    h = bh - b * L.H;
    return seq_span(L, b, nullptr, false);
}

// Element offset of row `row` (counted within the sequence) of head h of
// sequence b (bh = b * H + h) in an activation tensor whose rows hold D
// elements; kPacked says at compile time which placement L describes.
template <bool kPacked>
__device__ __forceinline__ size_t act_offset_t(const SeqLayout& L, int bh, int h, int start,
                                               int row, int D) {
    if constexpr (kPacked) return (static_cast<size_t>(start + row) * L.H + h) * D;
    else return (static_cast<size_t>(bh) * L.N + row) * D;
}

// Offset of the same row in a per-row float array (LSE).
template <bool kPacked>
__device__ __forceinline__ size_t rowval_offset_t(const SeqLayout& L, int bh, int h, int start,
                                                  int row) {
    if constexpr (kPacked) return static_cast<size_t>(h) * L.total + start + row;
    else return static_cast<size_t>(bh) * L.N + row;
}

// TMA box coordinates (y, z) of the 128-row tile that starts at `row`: dense
// maps are {d, N, B*H}, packed maps {d, H, T}.
template <bool kPacked>
__device__ __forceinline__ void tma_rows_t(int bh, int h, int start, int row, int& y, int& z) {
    if constexpr (kPacked) {
        y = h;
        z = start + row;
    } else {
        y = row;
        z = bh;
    }
}

// The same with the placement decided at run time (L.cu), for the light
// kernels that serve both.
__device__ __forceinline__ size_t act_offset(const SeqLayout& L, int bh, int h, int start,
                                             int row, int D) {
    return L.cu ? act_offset_t<true>(L, bh, h, start, row, D)
                : act_offset_t<false>(L, bh, h, start, row, D);
}

__device__ __forceinline__ size_t rowval_offset(const SeqLayout& L, int bh, int h, int start,
                                                int row) {
    return L.cu ? rowval_offset_t<true>(L, bh, h, start, row)
                : rowval_offset_t<false>(L, bh, h, start, row);
}

}  // namespace gbattn
