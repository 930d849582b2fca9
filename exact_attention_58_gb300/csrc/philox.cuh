// philox.cuh — Philox4x32-10 counter-based generator for the fused dropout.
//
// Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2, 3"
// (SC'11): ten rounds, each multiplying counter words 0 and 2 by the two
// round multipliers and mixing the high halves with the other two words and
// the key; the key advances by the two Weyl increments between rounds.
#pragma once

#include <cstdint>

namespace gbattn {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        const uint32_t lo0 = 0xD2511F53u * c.x;
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return c;
}

// Dropout draws of scores (i, j0..j0+7) of head (b, h), j0 a multiple of 8:
// one Philox4x32-10 block at counter (i, j0>>3, h, b) under key
// (seed_lo, seed_hi).  Its four 32-bit words hold eight 16-bit draws: key
// j0+e's is word e>>1, the low half for even e and the high half for odd e.
// A score is dropped iff its draw < threshold (threshold < 2^16).
__device__ __forceinline__ uint4 dropout_draws8(uint32_t seed_lo, uint32_t seed_hi, int i, int j0,
                                                int h, int b) {
    return philox4x32_10(make_uint4(static_cast<uint32_t>(i), static_cast<uint32_t>(j0) >> 3,
                                    static_cast<uint32_t>(h), static_cast<uint32_t>(b)),
                         seed_lo, seed_hi);
}

// Keep bits of the two draws of one word: bit 0 the low half's, bit 1 the
// high half's.
__device__ __forceinline__ uint32_t keep_pair(uint32_t w, uint32_t threshold) {
    return static_cast<uint32_t>((w & 0xFFFFu) >= threshold) |
           (static_cast<uint32_t>((w >> 16) >= threshold) << 1);
}

// AND-mask of a packed pair of 16-bit values whose keys' draws are the two
// halves of w: each half all ones if kept, zero if dropped.
__device__ __forceinline__ uint32_t keep_mask_h2(uint32_t w, uint32_t threshold) {
    return ((w & 0xFFFFu) >= threshold ? 0x0000FFFFu : 0u) |
           ((w >> 16) >= threshold ? 0xFFFF0000u : 0u);
}

// Keep bits of keys j0..j0+7 from their block of draws: bit e for key j0+e.
__device__ __forceinline__ uint32_t keep8(uint4 r, uint32_t threshold) {
    return keep_pair(r.x, threshold) | (keep_pair(r.y, threshold) << 2) |
           (keep_pair(r.z, threshold) << 4) | (keep_pair(r.w, threshold) << 6);
}

// Keep bits of one key against 16 consecutive queries, for a warp whose 32
// lanes own 32 consecutive keys starting at a multiple of 8 (lane L owns key
// j, the 8 lanes of an octet share j & ~7).  Lane a of an octet draws the
// blocks of queries q0+a and q0+8+a, so each lane holds a row of two 8 x 8
// bit matrices (query, key); three butterfly rounds across the octet
// transpose both, each swapping the bit-s digit of the lane and of the bit
// position where they differ.  Returns bit x = keep(query q0+x, key j).
// Warp-collective: all 32 lanes must call it together.
__device__ __forceinline__ uint32_t dropout_keep16_t(uint32_t seed_lo, uint32_t seed_hi,
                                                     uint32_t threshold, int q0, int j, int h,
                                                     int b, int lane) {
    const int a = lane & 7;
    const int j0 = j & ~7;
    uint32_t v = keep8(dropout_draws8(seed_lo, seed_hi, q0 + a, j0, h, b), threshold) |
                 (keep8(dropout_draws8(seed_lo, seed_hi, q0 + 8 + a, j0, h, b), threshold) << 8);
#pragma unroll
    for (int s = 4; s >= 1; s >>= 1) {
        // bit positions whose digit s is set, in both bytes
        const uint32_t m = s == 4 ? 0xF0F0u : (s == 2 ? 0xCCCCu : 0xAAAAu);
        const uint32_t y = __shfl_xor_sync(0xffffffffu, v, s);
        v = (a & s) ? ((v & m) | ((y >> s) & ~m & 0xFFFFu)) : ((v & ~m & 0xFFFFu) | ((y << s) & m));
    }
    return v;
}

}  // namespace gbattn
