// attn_fwd_kernel.cuh — fused exact-attention forward for sm_103a.
//
// One CTA owns 256 query rows (two 128-row tiles, A and B) of one (b, h) head
// — one 128-row tile at head dim 256, whose fp32 O alone takes 256 tensor-
// memory columns — and walks the key/value sequence in 128-row blocks,
// keeping everything on chip: the online-softmax recurrence of "Why
// FlashAttention Is a Kernel Story" (section "Tiling": running row max m,
// running denominator l, output rescaled when m grows, O / l at the end) with
// S = Q K^T and O += P V on the tcgen05 tensor cores.  Only O and the per-row
// log-sum-exp reach HBM.  Queries stand at key positions i + Nk - N (cross-
// attention); a sequence's rows are placed densely or packed (seq.cuh).
//
// Warp roles (320 threads with two tiles, 192 with one):
//   warps 0-3   softmax for tile A, one thread per query row (TMEM lane)
//   warps 4-7   softmax for tile B (two tiles only)
//   next warp   TMA producer: Q once, then K_j, V_j into a ring of smem slots
//   last warp   MMA issuer: S_t = Q_t K_j^T (both operands in smem) and
//               O_t += P_t V_j (P read from tensor memory, V from smem), as
//               kind::f16, kind::tf32 or kind::f8f6f4 products by input type
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   [0,128)   S_A, later P_A (16-bit pairs in the first 64 columns, e4m3
//             quads in the first 32, or fp32)
//   [128,256) S_B / P_B
//   [256, 256+d) O_A,  [256+d, 256+2d) O_B   (fp32 accumulators)
//   one tile: S in [0,128), O in [128, 128+d)
// P aliases S: the MMA warp issues S_t(j+1) only after O_t += P_t(j) V_j,
// and tcgen05 MMAs from one thread execute in issue order.
//
// Rescaling follows the recurrence exactly but lazily: a row keeps its
// reference max until the block max exceeds it by more than 8 (log2 units),
// so P <= 2^8 and O, l stay consistent with the same reference; the final
// O / l is unchanged.
//
// Every wait is bounded (kWaitLimitNs); on expiry the CTA drains its own
// TMA loads and MMAs, frees tensor memory and reports
// ATTN_ERR_DEVICE_TIMEOUT through dev_status.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"
#include "philox.cuh"
#include "ptx.cuh"
#include "seq.cuh"

namespace gbattn {
namespace {

template <int D, bool kTF32, bool kF16, bool kFP8, int kTiles>
struct FwdCfg {
    static constexpr int ES = kTF32 ? 4 : (kFP8 ? 1 : 2);  // element bytes of Q, K, V
    static constexpr int ROWB = D * ES;                    // bytes per row
    static constexpr int NCB = ROWB / 128;                 // 128-byte column blocks
    static constexpr int BOXW = 128 / ES;                  // elements per column block
    static constexpr int TILE = kTileRows * ROWB;          // bytes per 128-row tile
    static constexpr int CB_BYTES = kTileRows * 128;       // bytes per column block
    // Query tiles per CTA: two tiles share each K/V block in one CTA, or one
    // tile per CTA with two CTAs resident on an SM.  d = 256 takes one tile:
    // its O accumulator alone fills half of tensor memory.
    static constexpr int TILES = kTiles;
    static_assert(kTiles == 1 || (kTiles == 2 && D <= 128), "two tiles fit tensor memory up to d = 128");
    static constexpr int NSLOT = (TILES == 2 ? 4 : 2) * ((ROWB == 128) ? 2 : 1);   // K/V ring slots
    static constexpr int THREADS = 32 * (4 * TILES + 2);   // softmax warps, producer, MMA
    static constexpr int PRODUCER_WARP = 4 * TILES;
    static constexpr int MMA_WARP = 4 * TILES + 1;
    static constexpr uint32_t TMEM_COLS = (TILES == 2 || D > 128) ? 512 : 256;
    static constexpr int CTAS_PER_SM = TMEM_COLS == 512 ? 1 : 2;
    static constexpr uint32_t O_COL = 128 * TILES;          // first O column (S tiles below)
    static constexpr int KSTEP = 32 / ES;                  // K elements per MMA
    static constexpr int QK_STEPS = ROWB / 32;             // MMAs per S tile
    static constexpr int PV_STEPS = kTileRows / KSTEP;     // MMAs per P V
    static constexpr int SMEM = (TILES + NSLOT) * TILE + 1024 /*barriers*/ + 1024 /*align*/;
    static constexpr uint32_t FMT = kTF32 ? kFmtTF32 : (kFP8 ? kFmtE4M3 : fmt16<kF16>());
    static constexpr uint32_t IDESC_QK = idesc_f32acc(128, 128, FMT, false, false);
    static constexpr uint32_t IDESC_PV = idesc_f32acc(128, D, FMT, false, !kTF32);
    static_assert(ROWB == 128 || ROWB == 256 || ROWB == 512, "tile rows of 128, 256 or 512 bytes");
    static_assert(O_COL + TILES * D <= TMEM_COLS, "S and O tiles must fit in tensor memory");
};


// fp32 V_j (keys k0..k0+127 of one head, [N][D] in global memory) written into
// a shared-memory slot as the K-major B operand of O += P V: D rows (one per
// head-dim column) of 128 keys, in 32-key column blocks of D x 128 bytes,
// 128-byte swizzle.  Keys past N are written as zeros.  One warp.
template <int D>
__device__ __forceinline__ void store_v_transposed(const float* __restrict__ Vh, uint8_t* dst,
                                                   int k0, int N, int lane) {
#pragma unroll 1
    for (int t = 0; t < 4; ++t) {
        const int k = lane + 32 * t;       // key within the block; column block t
        const int key = k0 + k;
        const uint32_t kb_off = t * (D * 128) + (static_cast<uint32_t>(k & 3) << 2);
#pragma unroll 4
        for (int c4 = 0; c4 < D / 4; ++c4) {
            const float4 v = (key < N) ? *reinterpret_cast<const float4*>(Vh + static_cast<size_t>(key) * D + 4 * c4)
                                       : make_float4(0.f, 0.f, 0.f, 0.f);
            const float vv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = 4 * c4 + e;
                const uint32_t byte = kb_off + c * 128 + ((((k & 31) >> 2) ^ (c & 7)) << 4);
                *reinterpret_cast<float*>(dst + byte) = vv[e];
            }
        }
    }
}
constexpr float kRescaleThreshold = 8.0f;   // log2 units
constexpr float kLn2 = 0.69314718055994530942f;

// kSelfTest (one test instantiation only, never the attn_fwd path): the
// producer withholds the K tile of key block p.withhold_block and every wait
// gives up after p.wait_ns, so that a wait expires with copies and products
// in flight and the abort path below runs on the GPU.
template <int D, bool kTF32, bool kF16, bool kFP8, bool kCausal, bool kDropout, bool kWindow,
          bool kPacked, int kTiles, bool kSelfTest = false>
__global__ void __launch_bounds__(FwdCfg<D, kTF32, kF16, kFP8, kTiles>::THREADS,
                                  FwdCfg<D, kTF32, kF16, kFP8, kTiles>::CTAS_PER_SM)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const FwdParams p) {
    using C = FwdCfg<D, kTF32, kF16, kFP8, kTiles>;
    // Launched overlapped with the kernel before it: touch no global memory
    // before that one is done.  The forward does not let its own dependents in
    // early (their CTAs, parked next to the forward's last wave, cost it 0.4%
    // at N = 4096 and 16384 in an A/B on one GPU).
    grid_dep_wait();
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;                                   // C::TILES tiles
    uint8_t* sKV = smem + C::TILES * C::TILE;             // NSLOT tiles
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (C::TILES + C::NSLOT) * C::TILE);
    uint64_t* bar_q = bars;               // [2] one per query tile
    uint64_t* full = bars + 2;
    // Ring slots are freed by tensor-pipe commits.  A ring of kPairs >= 2 K/V
    // pairs takes one commit per key block j (after its last S, so K_j and
    // V_{j-1} are both read) on empty[(j - jbeg) % kPairs]: one commit fewer per
    // block than a commit per slot, and each commit costs the MMA warp a
    // queue slot (an extra one was 0.85% slower at C3).  A one-pair ring keeps
    // a barrier per slot.
    constexpr int kPairs = C::NSLOT / 2;
    constexpr bool kBlockRelease = kPairs >= 2;
    uint64_t* empty = full + C::NSLOT;
    uint64_t* bar_s = empty + C::NSLOT;   // [2]
    uint64_t* bar_p = bar_s + 2;          // [2]
    uint64_t* bar_o = bar_p + 2;          // [2]
    uint64_t* bar_fin = bar_o + 2;
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bar_fin + 1);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const unsigned long long lim = kSelfTest ? p.wait_ns : kWaitLimitNs;

    // ---- which 256 query rows of which head ----
    const int BH = p.B * p.H;
    int qb, bh;
    grouped_schedule(static_cast<int>(blockIdx.x), BH, p.nqb, bh, qb);
    if (kCausal) qb = p.nqb - 1 - qb;   // the last query blocks see the most keys
    const int b = bh / p.H, h = bh % p.H;
    // rows of this sequence: all N (Nk) when dense; when packed, the
    // sequence's own token range
    const bool report = threadIdx.x == 0 && h == 0 && qb == 0;
    const SeqSpan sq = kPacked ? seq_span(p.lq, b, p.dev_status, report) : SeqSpan{0, p.N};
    const SeqSpan sk = kPacked ? seq_span(p.lk, b, p.dev_status, report) : SeqSpan{0, p.Nk};
    const int N = sq.len;    // query rows
    const int Nk = sk.len;   // keys
    // Queries continue the key sequence: query i stands at key position
    // i + off for the causal and window tests (off = 0 when N == Nk).
    const int off = Nk - N;
    int L = Nk;
    if (p.key_lens != nullptr) {
        const int raw = p.key_lens[b];
        L = raw < 0 ? 0 : (raw > Nk ? Nk : raw);
        if (raw != L && threadIdx.x == 0 && p.dev_status != nullptr)
            atomicCAS(p.dev_status, 0, static_cast<int>(ATTN_ERR_INVALID_ARG));
    }
    const int q0 = qb * kTileRows * C::TILES;
    const int nkv_all = (L + kTileRows - 1) / kTileRows;
    // > 0: sliding window, keys with row - key < W (and key - row < W unless
    // causal); a compile-time 0 in the instantiations without a window
    const int W = kWindow ? p.window : 0;
    // Key blocks [jlo(t), jhi(t)) tile t needs (causal and window bounds skip
    // the rest).  Scalars and selects, not arrays: a loop-indexed array would
    // live in local memory inside the MMA issue loop.
    int jlo0 = 0, jlo1 = 0, jhi0 = 0, jhi1 = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        const int first = q0 + t * kTileRows;
        int lo = 0, hi = 0;
        if (first < N && t < C::TILES) {
            const int last = min(first + kTileRows - 1, N - 1);
            hi = kCausal ? (last + off >= 0 ? min(nkv_all, (last + off) / kTileRows + 1) : 0)
                         : nkv_all;
            if (W > 0) {
                lo = max(0, first + off - W + 1) / kTileRows;
                if (!kCausal) hi = max(0, min(nkv_all, (last + off + W - 1) / kTileRows + 1));
            }
            lo = min(lo, hi);
        }
        if (t == 0) { jlo0 = lo; jhi0 = hi; } else { jlo1 = lo; jhi1 = hi; }
    }
    auto jlo = [&](int t) { return t ? jlo1 : jlo0; };
    auto jhi = [&](int t) { return t ? jhi1 : jhi0; };
    auto nkv_t = [&](int t) { return jhi(t) - jlo(t); };   // blocks tile t sees
    // blocks the CTA walks: tile A's window starts no later than tile B's
    const int jbeg = (nkv_t(0) > 0) ? jlo0 : jlo1;
    const int jend = max(jhi0, jhi1);
    const int nkv = (nkv_t(0) > 0 || nkv_t(1) > 0) ? jend - jbeg : 0;

    // ---- set-up ----
    if (threadIdx.x == 0) {
        mbar_init(&bar_q[0], 1);
        mbar_init(&bar_q[1], 1);
        for (int s = 0; s < C::NSLOT; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int t = 0; t < 2; ++t) {
            mbar_init(&bar_s[t], 1);
            mbar_init(&bar_p[t], kTileRows);
            mbar_init(&bar_o[t], 1);
        }
        mbar_init(bar_fin, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == C::MMA_WARP) {
        tmem_alloc(s_tmem, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    if (warp == C::PRODUCER_WARP) {
        // ================= TMA producer =================
        // The whole warp walks the ring (waits are warp-collective); lane 0
        // issues the TMA copies.  TF32 products only take a K-major B, so for
        // fp32 inputs the warp itself writes V_j transposed (keys along K)
        // into its slot instead of a TMA copy.
        if (nkv > 0) {
            if (lane == 0) {
                tma_prefetch_desc(&tmQ);
                tma_prefetch_desc(&tmK);
                tma_prefetch_desc(&tmV);
            }
            // Issue order Q_0, K_jbeg, Q_1, V_jbeg, ... at d = 64, so that the
            // first S product waits for two of them only (1.9% faster at
            // N = 4096, 0.45% at N = 16384 in an A/B on one GPU); Q_0, Q_1,
            // K_jbeg, ... at d >= 128, where the early order measured 0.4%
            // slower at N = 4096.
            constexpr bool kQ1AfterK = (D == 64);
            const int ntiles = (nkv_t(1) > 0) ? 2 : 1;
            auto load_q = [&](int t) {
                int y, z;
                tma_rows_t<kPacked>(bh, h, sq.start, q0 + t * kTileRows, y, z);
                mbar_arrive_expect_tx(&bar_q[t], C::TILE);
                for (int cb = 0; cb < C::NCB; ++cb)
                    tma_load_3d(sQ + t * C::TILE + cb * C::CB_BYTES, &tmQ, &bar_q[t],
                                cb * C::BOXW, y, z);
            };
            bool q1_issued = false;
            if (lane == 0) {
                load_q(0);
                if (!kQ1AfterK && ntiles == 2) load_q(1);
            }
            if (!kQ1AfterK && ntiles == 2) q1_issued = true;
            int seq = 0;
            int withheld = -1;   // the fill left out (self test only)
            bool ok = true;
            for (int j = jbeg; j < jbeg + nkv && ok; ++j) {
                for (int which = 0; which < 2; ++which) {
                    if (which == 1 && ntiles == 2 && !q1_issued) {   // after the first K
                        if (lane == 0) load_q(1);
                        q1_issued = true;
                    }
                    const int slot = seq % C::NSLOT;
                    const uint32_t ph = (seq / C::NSLOT) & 1;
                    bool free_ok;
                    if constexpr (kBlockRelease) {
                        // the slot's previous tile (K or V of block bi - P) is
                        // free once block bi - P (K) or bi - P + 1 (V) has
                        // released its pair
                        const int bi = j - jbeg;
                        const int wb = which == 0 ? bi - kPairs : bi - kPairs + 1;
                        free_ok = bi < kPairs ||
                                  mbar_wait_warp(&empty[wb % kPairs], (wb / kPairs) & 1, s_abort, lim);
                    } else {
                        free_ok = mbar_wait_warp(&empty[slot], ph ^ 1, s_abort, lim);
                    }
                    if (!free_ok) {
                        ok = false;
                        break;
                    }
                    if (kSelfTest && which == 0 && j == p.withhold_block) {   // no copy, no arrival
                        withheld = seq++;
                        continue;
                    }
                    if (kTF32 && which == 1) {
                        store_v_transposed<D>(static_cast<const float*>(p.V) +
                                                  static_cast<size_t>(bh) * Nk * D,
                                              sKV + slot * C::TILE, j * kTileRows, Nk, lane);
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0) mbar_arrive(&full[slot]);
                    } else if (lane == 0) {
                        mbar_arrive_expect_tx(&full[slot], C::TILE);
                        const CUtensorMap* m = which ? &tmV : &tmK;
                        int y, z;
                        tma_rows_t<kPacked>(bh, h, sk.start, j * kTileRows, y, z);
                        for (int cb = 0; cb < C::NCB; ++cb)
                            tma_load_3d(sKV + slot * C::TILE + cb * C::CB_BYTES, m, &full[slot],
                                        cb * C::BOXW, y, z);
                    }
                    ++seq;
                }
            }
            // Drain: every load this warp issued has landed before teardown.
            if (lane == 0) {
                volatile int no_abort = 0;
                mbar_wait(&bar_q[0], 0, &no_abort, lim);
                if (q1_issued) mbar_wait(&bar_q[1], 0, &no_abort, lim);
                for (int s = 0; s < C::NSLOT && s < seq; ++s) {
                    const int uses = (seq - s + C::NSLOT - 1) / C::NSLOT;
                    // a withheld fill is always its slot's last: nothing refills
                    // a slot whose consumer never got its tile
                    if (s + (uses - 1) * C::NSLOT == withheld) continue;
                    mbar_wait(&full[s], (uses - 1) & 1, &no_abort, lim);
                }
            }
        }
        __syncwarp();
    } else if (warp == C::MMA_WARP) {
        // ================= MMA issuer =================
        if (lane == 0 && nkv > 0) {
            // Descriptor bases built once; each MMA only adds a constant.
            const uint64_t dq0 = sdesc_sw128(smem_u32(sQ), 16, 1024);
            const uint64_t dq1 = sdesc_adv(dq0, C::TILE);
            const uint64_t dk0 = sdesc_sw128(smem_u32(sKV), 16, 1024);   // K-major, slot 0
            const uint64_t dv0 = kTF32 ? dk0 : sdesc_sw128(smem_u32(sKV), C::CB_BYTES, 1024);
            auto issue_qk = [&](int t, int slot) {
                const uint32_t d_tmem = tmem + 128u * t;
                const uint64_t ad = t ? dq1 : dq0;
                const uint64_t bd = sdesc_adv(dk0, slot * C::TILE);
                // 16-bit inputs: one run of MMAs (32-byte K steps, the next
                // 128-byte column block after four)
                constexpr uint32_t CB = C::CB_BYTES / 16 - 6;
                if constexpr (!kTF32 && !kFP8 && C::QK_STEPS == 8) {
                    mma8_ss_f16<2, 2, 2, CB, 2, 2, 2, 2, 2, 2, CB, 2, 2, 2>(d_tmem, ad, bd, C::IDESC_QK, 0u);
                    return;
                } else if constexpr (!kTF32 && !kFP8 && C::QK_STEPS == 4) {
                    mma4_ss_f16<2, 2, 2, 2, 2, 2>(d_tmem, ad, bd, C::IDESC_QK, 0u);
                    return;
                } else if constexpr (!kTF32 && !kFP8 && C::QK_STEPS == 16) {   // d = 256: two runs
                    mma8_ss_f16<2, 2, 2, CB, 2, 2, 2, 2, 2, 2, CB, 2, 2, 2>(d_tmem, ad, bd, C::IDESC_QK, 0u);
                    mma8_ss_f16<2, 2, 2, CB, 2, 2, 2, 2, 2, 2, CB, 2, 2, 2>(
                        d_tmem, sdesc_adv(ad, 2 * C::CB_BYTES), sdesc_adv(bd, 2 * C::CB_BYTES),
                        C::IDESC_QK, 1u);
                    return;
                }
#pragma unroll
                for (int kk = 0; kk < C::QK_STEPS; ++kk) {
                    const uint32_t off = (kk >> 2) * C::CB_BYTES + (kk & 3) * 32;
                    if constexpr (kFP8)
                        mma_ss_f8(d_tmem, sdesc_adv(ad, off), sdesc_adv(bd, off), C::IDESC_QK,
                                  kk > 0 ? 1u : 0u);
                    else
                        mma_ss<kTF32>(d_tmem, sdesc_adv(ad, off), sdesc_adv(bd, off), C::IDESC_QK,
                                      kk > 0 ? 1u : 0u);
                }
            };
            auto issue_pv = [&](int t, int slot, bool accumulate) {
                const uint32_t d_tmem = tmem + C::O_COL + D * t;
                const uint32_t a_tmem = tmem + 128u * t;
                const uint64_t bd = sdesc_adv(dv0, slot * C::TILE);
                if constexpr (!kTF32 && !kFP8 && C::PV_STEPS == 8) {   // 16-bit: 8 x 16 keys
                    mma_run_ts_f16<8, 8, C::KSTEP * 128 / 16>(d_tmem, a_tmem, bd, C::IDESC_PV,
                                                              accumulate ? 1u : 0u);
                    return;
                }
#pragma unroll
                for (int kk = 0; kk < C::PV_STEPS; ++kk) {
                    // bf16: V as stored (MN-major); fp32: V transposed (K-major)
                    const uint32_t off = kTF32 ? (kk >> 2) * (D * 128) + (kk & 3) * 32
                                               : kk * C::KSTEP * 128;
                    if constexpr (kFP8)
                        mma_ts_f8(d_tmem, a_tmem + kk * 8, sdesc_adv(bd, off), C::IDESC_PV,
                                  (accumulate || kk > 0) ? 1u : 0u);
                    else
                        mma_ts<kTF32>(d_tmem, a_tmem + kk * 8, sdesc_adv(bd, off), C::IDESC_PV,
                                      (accumulate || kk > 0) ? 1u : 0u);
                }
            };
            bool ok = true;
            bool q_ready[2] = {false, false};
            int seq = 0;
            int v_slot = 0;
            uint32_t v_phase = 0;
            bool v_ready = false;
            for (int j = jbeg; j < jbeg + nkv && ok; ++j) {
                const int kslot = seq % C::NSLOT;
                const uint32_t kph = (seq / C::NSLOT) & 1;
                ++seq;
                const int next_v_slot = seq % C::NSLOT;
                const uint32_t next_v_phase = (seq / C::NSLOT) & 1;
                ++seq;
                bool k_ready = false;
                // With a ring of one K/V pair (d = 256, one-tile d = 128) V_{j-1}'s
                // slot is released right behind the last P V that reads it, so
                // that V_j's refill starts before S_j (5.6% faster at d = 256,
                // N = 4096); with deeper rings the commit between the products
                // costs more than it saves (2.6% slower at C3), so the slot goes
                // after the block's last S.
                constexpr bool kEarlyVRelease = C::NSLOT == 2;
                int v_last = -1;
                for (int t = 0; t < C::TILES; ++t)
                    if (kEarlyVRelease && j - 1 >= jlo(t) && j - 1 < jhi(t)) v_last = t;
                for (int t = 0; t < C::TILES && ok; ++t) {
                    const bool qk = j >= jlo(t) && j < jhi(t);
                    const bool prev = j - 1 >= jlo(t) && j - 1 < jhi(t);   // tile t saw block j-1
                    const bool last_pv = prev && j == jhi(t);
                    if (prev) {   // O_t += P_t(j-1) V_{j-1}, once the softmax of j-1 is done
                        ok = mbar_wait(&bar_p[t], (j - 1 - jlo(t)) & 1, s_abort, lim);
                        if (!ok) break;
                        tc_fence_after();
                        if (!v_ready) {
                            ok = mbar_wait(&full[v_slot], v_phase, s_abort, lim);
                            v_ready = true;
                            if (!ok) break;
                            tc_fence_after();
                        }
                        issue_pv(t, v_slot, j - 1 > jlo(t));
                        if (last_pv) tc_commit(&bar_o[t]);
                        if (t == v_last) tc_commit(&empty[v_slot]);
                    }
                    if (qk) {                         // S_t = Q_t K_j^T
                        if (!q_ready[t]) {
                            ok = mbar_wait(&bar_q[t], 0, s_abort, lim);
                            q_ready[t] = true;
                            if (!ok) break;
                            tc_fence_after();
                        }
                        if (!k_ready) {
                            ok = mbar_wait(&full[kslot], kph, s_abort, lim);
                            k_ready = true;
                            if (!ok) break;
                            tc_fence_after();
                        }
                        issue_qk(t, kslot);
                        tc_commit(&bar_s[t]);
                    }
                }
                if (!ok) break;
                if constexpr (kBlockRelease) {
                    tc_commit(&empty[(j - jbeg) % kPairs]);
                } else {
                    tc_commit(&empty[kslot]);
                    if (j > jbeg && v_last < 0) tc_commit(&empty[v_slot]);   // unless released above
                }
                v_slot = next_v_slot;
                v_phase = next_v_phase;
                v_ready = false;
            }
            for (int t = 0; t < C::TILES && ok; ++t) {   // tiles whose last block is the CTA's last
                if (nkv_t(t) == 0 || jhi(t) != jbeg + nkv) continue;
                ok = mbar_wait(&bar_p[t], (jhi(t) - 1 - jlo(t)) & 1, s_abort, lim);
                if (ok && !v_ready) {
                    ok = mbar_wait(&full[v_slot], v_phase, s_abort, lim);
                    v_ready = true;
                }
                if (!ok) break;
                tc_fence_after();
                issue_pv(t, v_slot, jhi(t) - 1 > jlo(t));
                tc_commit(&bar_o[t]);
            }
            // Drain: no MMA of this CTA is in flight at teardown.
            tc_commit(bar_fin);
            volatile int no_abort = 0;
            mbar_wait(bar_fin, 0, &no_abort, lim);
        }
        __syncwarp();
    } else {
        // ================= softmax (warps 0-7) =================
        const int t = warp >> 2;
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int row = q0 + t * kTileRows + r;
        const int ntile = nkv_t(t);
        const int tile_first_row = q0 + t * kTileRows;
        const uint32_t t_lane = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t t_S = t_lane + 128u * t;
        const uint32_t t_O = t_lane + C::O_COL + D * t;
        float m_ref = -INFINITY;   // reference max, log2 units of scaled scores
        float l = 0.f;
        bool ok = true;
        for (int j = jlo(t); j < jhi(t); ++j) {
            if (!mbar_wait_warp(&bar_s[t], (j - jlo(t)) & 1, s_abort, lim)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const int k0 = j * kTileRows;
            const int tile_last_row = tile_first_row + kTileRows - 1;
            const bool wmask = W > 0 && (k0 < tile_last_row + off - W + 1 ||
                                         (!kCausal && k0 + kTileRows - 1 > tile_first_row + off + W - 1));
            const bool tile_mask = (k0 + kTileRows > L) ||
                                   (kCausal && k0 + kTileRows - 1 > tile_first_row + off) || wmask;
            // columns >= lim and < lo of this row are masked (only on masked tiles)
            int lim = tile_mask ? (kCausal ? min(L, row + off + 1) : L) - k0 : kTileRows;
            int lo = 0;
            if (wmask) {
                lo = row + off - W + 1 - k0;
                if (!kCausal) lim = min(lim, row + off + W - k0);
            }

            // ---- pass 1: row max (S read from TMEM, eight independent chains) ----
            float mx;
            uint32_t sr[4][32];   // all of S stays in registers for pass 2
            {
#pragma unroll
                for (int c = 0; c < 4; ++c) tmem_ld32(t_S + 32 * c, sr[c]);
                tmem_ld_wait();
#pragma unroll
                for (int c = 0; c < 4; ++c) reg_fence(sr[c]);
                if (tile_mask) {
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= lim || c < lo) sr[c >> 5][c & 31] = __float_as_uint(-INFINITY);
                }
                float mp[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mp[k] = -INFINITY;
#pragma unroll
                for (int c = 0; c < 128; c += 2)
                    mp[(c >> 1) & 7] = max3f(mp[(c >> 1) & 7], __uint_as_float(sr[c >> 5][c & 31]),
                                             __uint_as_float(sr[c >> 5][(c & 31) + 1]));
                mx = max3f(max3f(mp[0], mp[1], mp[2]), max3f(mp[3], mp[4], mp[5]),
                           fmaxf(mp[6], mp[7]));
            }
            const float m_new = fmaxf(m_ref, mx * p.scale_log2);
            const bool want = (m_ref != -INFINITY) && (m_new > m_ref + kRescaleThreshold);
            const bool warp_rescale = __any_sync(0xffffffffu, want);
            float alpha = 1.f;
            if (m_ref == -INFINITY) {
                m_ref = m_new;   // O and l are still zero: adopt without rescaling
            } else if (warp_rescale) {
                alpha = ex2_approx(m_ref - m_new);
                m_ref = m_new;
            }
            const float neg_m = (m_ref == -INFINITY) ? 0.f : -m_ref;

            // ---- pass 2: P = exp2(s scale log2e - m), 32 keys at a time, from
            // the scores pass 1 left in registers (re-reading them from tensor
            // memory put a load latency on the chain of every chunk; keeping
            // them was 2% faster at C3, 5% at N = 1024 and d = 64) ----
            float rowsum = 0.f;
            const uint64_t sc2 = f2_pack(p.scale_log2, p.scale_log2);
            const uint64_t nm2 = f2_pack(neg_m, neg_m);
            uint64_t acc2[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) acc2[k] = f2_pack(0.f, 0.f);
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t* sv = sr[cc];   // masked in pass 1
                if constexpr (kFP8) {
                    // P rounded to e4m3, four keys per word, 32 keys in 8
                    // columns; the row sum adds the unrounded P.
                    uint32_t pk[8];
                    uint4 dr = make_uint4(0u, 0u, 0u, 0u);   // draws of this group pair's 8 keys
#pragma unroll
                    for (int g = 0; g < 8; ++g) {   // 4 keys per group
                        float x[4];
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[4 * g + 2 * e]),
                                                     __uint_as_float(sv[4 * g + 2 * e + 1])),
                                             sc2, nm2),
                                      x[2 * e], x[2 * e + 1]);
                            x[2 * e] = ex2_approx(x[2 * e]);
                            x[2 * e + 1] = ex2_approx(x[2 * e + 1]);
                            acc2[(2 * g + e) & 3] =
                                f2_add(acc2[(2 * g + e) & 3], f2_pack(x[2 * e], x[2 * e + 1]));
                        }
                        uint32_t u = pack_e4m3x4(x[0], x[1], x[2], x[3]);
                        if constexpr (kDropout) {
                            if ((g & 1) == 0)
                                dr = dropout_draws8(p.seed_lo, p.seed_hi, row, k0 + 32 * cc + 4 * g, h, b);
                            const uint32_t keep = keep_pair((g & 1) ? dr.z : dr.x, p.drop_threshold) |
                                                  (keep_pair((g & 1) ? dr.w : dr.y, p.drop_threshold) << 2);
                            u &= ((keep & 1u) ? 0x000000FFu : 0u) | ((keep & 2u) ? 0x0000FF00u : 0u) |
                                 ((keep & 4u) ? 0x00FF0000u : 0u) | ((keep & 8u) ? 0xFF000000u : 0u);
                        }
                        pk[g] = u;
                    }
                    tmem_st8(t_S + 8 * cc, pk);
                } else if constexpr (!kTF32) {
                    // exp2 arguments two at a time (paired FMA); the row sum adds
                    // the unrounded P (fp32) in four independent paired chains.
#pragma unroll
                    for (int half = 0; half < 2; ++half) {   // 16 keys, 8 packed words
                        uint32_t pk[8];
                        uint4 dr = make_uint4(0u, 0u, 0u, 0u);   // draws of this group pair's 8 keys
#pragma unroll
                        for (int g = 4 * half; g < 4 * half + 4; ++g) {   // 4 keys per group
                            if constexpr (kDropout)
                                if ((g & 1) == 0)
                                    dr = dropout_draws8(p.seed_lo, p.seed_hi, row, k0 + 32 * cc + 4 * g,
                                                        h, b);
#pragma unroll
                            for (int e = 0; e < 2; ++e) {
                                float x0, x1;
                                f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[4 * g + 2 * e]),
                                                         __uint_as_float(sv[4 * g + 2 * e + 1])),
                                                 sc2, nm2),
                                          x0, x1);
                                x0 = ex2_approx(x0);
                                x1 = ex2_approx(x1);
                                uint32_t u = pack_h2<kF16>(x0, x1);
                                acc2[(2 * g + e) & 3] = f2_add(acc2[(2 * g + e) & 3], f2_pack(x0, x1));
                                if constexpr (kDropout)   // the pair's draws are the halves of one word
                                    u &= keep_mask_h2((g & 1) ? (e ? dr.w : dr.z) : (e ? dr.y : dr.x),
                                                      p.drop_threshold);
                                pk[2 * (g - 4 * half) + e] = u;
                            }
                        }
                        tmem_st8(t_S + 16 * cc + 8 * half, pk);
                    }
                } else {
                    uint32_t pf[32];
                    uint4 dr = make_uint4(0u, 0u, 0u, 0u);   // draws of this group pair's 8 keys
#pragma unroll
                    for (int g = 0; g < 8; ++g) {
                        uint32_t keep = 0xFu;
                        if constexpr (kDropout) {
                            if ((g & 1) == 0)
                                dr = dropout_draws8(p.seed_lo, p.seed_hi, row, k0 + 32 * cc + 4 * g, h, b);
                            keep = keep_pair((g & 1) ? dr.z : dr.x, p.drop_threshold) |
                                   (keep_pair((g & 1) ? dr.w : dr.y, p.drop_threshold) << 2);
                        }
#pragma unroll
                        for (int e = 0; e < 2; ++e) {
                            float x0, x1;
                            f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[4 * g + 2 * e]),
                                                     __uint_as_float(sv[4 * g + 2 * e + 1])),
                                             sc2, nm2),
                                      x0, x1);
                            x0 = ex2_approx(x0);
                            x1 = ex2_approx(x1);
                            acc2[(2 * g + e) & 3] = f2_add(acc2[(2 * g + e) & 3], f2_pack(x0, x1));
                            pf[4 * g + 2 * e] = ((keep >> (2 * e)) & 1u) ? __float_as_uint(x0) : 0u;
                            pf[4 * g + 2 * e + 1] =
                                ((keep >> (2 * e + 1)) & 1u) ? __float_as_uint(x1) : 0u;
                        }
                    }
                    tmem_st32(t_S + 32 * cc, pf);
                }
            }
            {
                float a0, a1, a2, a3;
                f2_unpack(f2_add(acc2[0], acc2[1]), a0, a1);
                f2_unpack(f2_add(acc2[2], acc2[3]), a2, a3);
                rowsum = (a0 + a1) + (a2 + a3);
            }
            l = l * alpha + rowsum;
            if (warp_rescale && j > jlo(t)) {   // O row *= alpha (PV of block j-1 is complete)
#pragma unroll
                for (int c = 0; c < D / 32; ++c) {
                    uint32_t o[32];
                    tmem_ld32(t_O + 32 * c, o);
                    tmem_ld_wait();
                    reg_fence(o);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st32(t_O + 32 * c, o);
                }
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive_warp(&bar_p[t]);
        }
        // ---- epilogue: O = acc / l (times 1/(1-p)), LSE = (m + log2 l) ln 2 ----
        if (ok && ntile > 0) {
            ok = mbar_wait_warp(&bar_o[t], 0, s_abort, lim);
            tc_fence_after();
        }
        if (ok) {
            const float inv = (l > 0.f) ? p.out_scale / l : 0.f;
            const size_t row_off = act_offset_t<kPacked>(p.lq, bh, h, sq.start, row, D);
            // O in 32-column chunks, the next chunk's TMEM load overlapping this
            // chunk's conversion and stores
            uint32_t ob[2][32];
            if (ntile > 0) {
                tmem_ld32(t_O, ob[0]);
                tmem_ld_wait();
                reg_fence(ob[0]);
            }
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
                if (ntile > 0 && c + 1 < D / 32) tmem_ld32(t_O + 32 * (c + 1), ob[(c + 1) & 1]);
                uint32_t* o = ob[c & 1];
                if (ntile == 0) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = 0u;
                }
                if (row < N) {
                    if constexpr (kTF32) {
                        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.O) + row_off + 32 * c);
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            dst[v] = make_float4(__uint_as_float(o[4 * v]) * inv,
                                                 __uint_as_float(o[4 * v + 1]) * inv,
                                                 __uint_as_float(o[4 * v + 2]) * inv,
                                                 __uint_as_float(o[4 * v + 3]) * inv);
                    } else {
                        uint4* dst = reinterpret_cast<uint4*>(
                            static_cast<uint16_t*>(p.O) + row_off + 32 * c);
#pragma unroll
                        for (int v = 0; v < 4; ++v) {
                            uint32_t w[4];
#pragma unroll
                            for (int e = 0; e < 4; ++e)
                                w[e] = pack_h2<kF16>(__uint_as_float(o[8 * v + 2 * e]) * inv,
                                                     __uint_as_float(o[8 * v + 2 * e + 1]) * inv);
                            dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
                if (ntile > 0 && c + 1 < D / 32) {
                    tmem_ld_wait();
                    reg_fence(ob[(c + 1) & 1]);
                }
            }
            if (row < N)
                p.LSE[rowval_offset_t<kPacked>(p.lq, bh, h, sq.start, row)] =
                    (l > 0.f) ? (m_ref + log2f(l)) * kLn2 : -INFINITY;
        }
    }

    // ---- teardown ----
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == C::MMA_WARP) tmem_dealloc(tmem, C::TMEM_COLS);
    if (threadIdx.x == 0 && *s_abort && p.dev_status != nullptr)
        atomicCAS(p.dev_status, 0, static_cast<int>(ATTN_ERR_DEVICE_TIMEOUT));
}

template <int D, bool kTF32, bool kF16, bool kFP8, bool kCausal, bool kDropout, bool kWindow,
          bool kPacked, int kTiles, bool kSelfTest = false>
cudaError_t launch_fwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const FwdParams& p, cudaStream_t stream) {
    using C = FwdCfg<D, kTF32, kF16, kFP8, kTiles>;
    auto kern = attn_fwd_kernel<D, kTF32, kF16, kFP8, kCausal, kDropout, kWindow, kPacked, kTiles,
                                kSelfTest>;
    static std::atomic<unsigned long long> smem_ready{0};
    const cudaError_t e = enable_smem_per_device(kern, C::SMEM, smem_ready);
    if (e != cudaSuccess) return e;
    FwdParams pp = p;
    pp.nqb = (p.N + kTileRows * C::TILES - 1) / (kTileRows * C::TILES);
    const unsigned grid = static_cast<unsigned>(pp.nqb) * static_cast<unsigned>(p.B * p.H);
    return launch_overlapped(kern, grid, C::THREADS, C::SMEM, stream, tq, tk, tv, pp);
}

template <int D, bool kTF32, bool kF16, bool kFP8, bool kPacked, bool kWindow, int kTiles>
cudaError_t dispatch_mask_w(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                            const FwdParams& p, bool causal, bool dropout, cudaStream_t s) {
    if (causal)
        return dropout ? launch_fwd_t<D, kTF32, kF16, kFP8, true, true, kWindow, kPacked, kTiles>(tq, tk, tv, p, s)
                       : launch_fwd_t<D, kTF32, kF16, kFP8, true, false, kWindow, kPacked, kTiles>(tq, tk, tv, p, s);
    return dropout ? launch_fwd_t<D, kTF32, kF16, kFP8, false, true, kWindow, kPacked, kTiles>(tq, tk, tv, p, s)
                   : launch_fwd_t<D, kTF32, kF16, kFP8, false, false, kWindow, kPacked, kTiles>(tq, tk, tv, p, s);
}

// kTiles query tiles per CTA; head dim 256 always takes one.
template <int D, bool kTF32, bool kF16, bool kFP8, bool kPacked, int kTiles = (D == 256 ? 1 : 2)>
cudaError_t dispatch_mask(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                          const FwdParams& p, bool causal, bool dropout, cudaStream_t s) {
    return p.window > 0 ? dispatch_mask_w<D, kTF32, kF16, kFP8, kPacked, true, kTiles>(tq, tk, tv, p, causal, dropout, s)
                        : dispatch_mask_w<D, kTF32, kF16, kFP8, kPacked, false, kTiles>(tq, tk, tv, p, causal, dropout, s);
}

}  // namespace
}  // namespace gbattn
