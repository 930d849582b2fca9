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

// Keep bits of scores (i, j0..j0+3) of head (b, h), j0 a multiple of 4:
// bit e set iff score (i, j0+e) is kept (its Philox word is >= threshold).
__device__ __forceinline__ uint32_t dropout_keep4(uint32_t seed_lo, uint32_t seed_hi,
                                                  uint32_t threshold, int i, int j0, int h,
                                                  int b) {
    const uint4 r = philox4x32_10(
        make_uint4(static_cast<uint32_t>(i), static_cast<uint32_t>(j0) >> 2,
                   static_cast<uint32_t>(h), static_cast<uint32_t>(b)),
        seed_lo, seed_hi);
    return static_cast<uint32_t>(r.x >= threshold) | (static_cast<uint32_t>(r.y >= threshold) << 1) |
           (static_cast<uint32_t>(r.z >= threshold) << 2) |
           (static_cast<uint32_t>(r.w >= threshold) << 3);
}

}  // namespace gbattn
