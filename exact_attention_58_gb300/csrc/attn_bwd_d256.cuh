// attn_bwd_d256.cuh — main kernel of the fused exact-attention backward for
// head dim 256 (bf16 or fp16), sm_103a.
//
// At d = 256 the dK and dV accumulators of one 128-key block (fp32, 256
// columns each) would fill tensor memory on their own, and 128-row Q, dO
// tiles next to the resident K and V no longer fit in shared memory.  The
// work is therefore split over the head dim: each CTA owns one (head, 128-key
// block, half of d) and accumulates dK, dV for its 128 output columns in
// tensor memory, recomputing S^T = K Q^T and dP^T = V dO^T (contractions over
// the whole d) from full-width tiles; query blocks are 64 rows.  The two
// halves of a key block run as neighbouring CTAs.  The recomputation of P from
// Q, K and the stored log-sum-exp is the one of "Why FlashAttention Is a
// Kernel Story" ("When it falls down", backward pass); that page names
// d = 256 as the case that needs smaller tiles.
//
// Per query block i (64 rows), for the CTA's half h of d:
//   S^T  = K_j Q_i^T,  dP^T = V_j dO_i^T              (N = 64, K = 256)
//   P^T  = exp2(S^T scale log2e - LSE_i log2e)        (masked, dropout bits)
//   dS^T = P^T (dP^T Z/(1-p) - D_i)
//   dV_h += (P Z/(1-p))^T dO_i[:, h]                  (P read from TMEM)
//   dK_h += dS^T Q_i[:, h]                            (dS from smem)
//   dQ_i[:, h] += dS K_j[:, h]                        (as dQ^T = K^T dS^T, added
//                                                      into the fp32 workspace)
//
// Warp roles (448 threads):
//   warps 0-3  compute, queries 0-31 of the block: one thread per key row
//   warps 4-7  compute, queries 32-63
//   warps 8-11 dQ: dQ^T out of TMEM (lane = one of the 128 columns of the
//              half), one 128-byte add per warp instruction
//   warp  12   TMA producer: K_j, V_j once; per block Q_i with LSE_i and D_i
//              (freed once dK_h of the block is done) and dO_i (freed once
//              dV_h is done), one buffer each
//   warp  13   MMA issuer
//
// Tensor memory: dK_h [0,128) dV_h [128,256) S [256,320) dP [320,384)
// dQ^T [384,448).  Each compute warpgroup writes its P (16-bit pairs) over
// the first 16 columns of its 32-column part of S.
#pragma once

#include "internal.h"
#include "philox.cuh"
#include "ptx.cuh"
#include "seq.cuh"

namespace gbattn {
namespace {

template <bool kF16>
struct Bwd256Cfg {
    static constexpr int D = 256;
    static constexpr int QR = 64;                  // query rows per block
    static constexpr int THREADS = 448;
    static constexpr int NCB = D * 2 / 128;        // 128-byte column blocks per row (4)
    static constexpr int KCB = kTileRows * 128;    // one column block of a 128-row tile
    static constexpr int QCB = QR * 128;           // one column block of a 64-row tile
    static constexpr int KTILE = NCB * KCB;        // 64 KB
    static constexpr int QTILE = NCB * QCB;        // 32 KB
    static constexpr int DS_BYTES = kTileRows * QR * 2;   // [128 keys][64 queries]
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = KTILE;
    // Q in two parts: the half of d this CTA does not own (read by S only,
    // refilled as soon as S of the block has run) and two buffers for the
    // owned half (read by S and dK), so that the next block's Q is in place
    // before its S; LSE and D double-buffered with the owned half.
    static constexpr int QHALF = 2 * QCB;               // 16 KB: two column blocks
    static constexpr int OFF_Q = 2 * KTILE;             // the other half
    static constexpr int OFF_QOWN = OFF_Q + QHALF;      // [2] the owned half
    static constexpr int OFF_DO = OFF_QOWN + 2 * QHALF;
    static constexpr int OFF_DS = OFF_DO + QTILE;
    static constexpr int OFF_LSE = OFF_DS + DS_BYTES;   // [2][64] float
    static constexpr int OFF_D = OFF_LSE + 2 * QR * 4;  // [2][64] float
    static constexpr int OFF_BAR = OFF_D + 2 * QR * 4;
    static constexpr int SMEM = OFF_BAR + 256;
    static constexpr uint32_t C_DK = 0, C_DV = 128, C_S = 256, C_DP = 320, C_DQ = 384;
    static constexpr uint32_t FMT = fmt16<kF16>();
    static constexpr uint32_t IDESC_SDP = idesc_f32acc(128, QR, FMT, false, false);
    static constexpr uint32_t IDESC_DKV = idesc_f32acc(128, 128, FMT, false, true);
    // dQ^T = K^T dS^T: M = 128 columns of the half, N = 64 queries
    static constexpr uint32_t IDESC_DQ = idesc_f32acc(128, QR, FMT, true, true);
    static_assert(SMEM <= 232448, "shared memory budget");
    static_assert(OFF_Q % 1024 == 0 && OFF_QOWN % 1024 == 0 && OFF_DO % 1024 == 0 &&
                      OFF_DS % 1024 == 0,
                  "swizzled tiles start on 1024-byte boundaries");
    static_assert(OFF_DO - OFF_Q >= KTILE / 2, "the dK staging tile fits over the Q buffers");
};

template <bool kF16, bool kCausal, bool kDropout, bool kWindow, bool kPacked>
__global__ void __launch_bounds__(448, 1)
    attn_bwd_d256_kernel(const __grid_constant__ CUtensorMap tmQ,   // 64-row boxes
                         const __grid_constant__ CUtensorMap tmK,   // 128-row boxes
                         const __grid_constant__ CUtensorMap tmV,
                         const __grid_constant__ CUtensorMap tmdO,  // 64-row boxes
                         const __grid_constant__ CUtensorMap tmdK,
                         const __grid_constant__ CUtensorMap tmdV, const BwdParams p) {
    using C = Bwd256Cfg<kF16>;
    constexpr int D = C::D;
    constexpr int QR = C::QR;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    grid_dep_launch_dependents();   // as in the d <= 128 kernel: waits before the workspace

    const int BH = p.B * p.H;
    int rank, bh;   // rank / 2: key block (0 = heaviest under causal), rank % 2: half of d
    grouped_schedule(static_cast<int>(blockIdx.x), BH, 2 * p.nkb, bh, rank);
    const int kb = rank >> 1;
    const int half = rank & 1;
    const int b = bh / p.H, h = bh % p.H;
    const bool report = threadIdx.x == 0 && h == 0 && rank == 0;
    const SeqSpan sq = kPacked ? seq_span(p.lq, b, p.dev_status, report) : SeqSpan{0, p.N};
    const SeqSpan sk = kPacked ? seq_span(p.lk, b, p.dev_status, report) : SeqSpan{0, p.Nk};
    const int N = sq.len;    // query rows
    const int Nk = sk.len;   // keys
    const int off = Nk - N;  // query i stands at key position i + off
    const int nqb = (N + QR - 1) / QR;
    int L = Nk;
    if (p.key_lens != nullptr) {
        const int raw = p.key_lens[b];
        L = raw < 0 ? 0 : (raw > Nk ? Nk : raw);
        if (raw != L && threadIdx.x == 0 && p.dev_status != nullptr)
            atomicCAS(p.dev_status, 0, static_cast<int>(ATTN_ERR_INVALID_ARG));
    }
    const int k0 = kb * kTileRows;
    const int W = kWindow ? p.window : 0;
    int q_begin = kCausal ? max(0, k0 - off) / QR : 0;
    int q_end = nqb;
    if (W > 0) {
        const int last_q = k0 + kTileRows - 1 - off + W - 1;   // last query the block's keys reach
        q_end = last_q < 0 ? 0 : min(nqb, last_q / QR + 1);
        if (!kCausal) q_begin = max(0, k0 - off - W + 1) / QR;
    }
    const int nq = q_end - q_begin;
    const int c0 = 128 * half;   // first column of this CTA's half of d
    if (k0 >= L || nq <= 0) {    // no key of this block is attended: this half of dK, dV is 0
        grid_dep_wait();
        const int rows = min(kTileRows, Nk - k0);
        for (int x = threadIdx.x; x < rows * 16; x += blockDim.x) {   // 16 x 8 elements a row
            const size_t e = act_offset_t<kPacked>(p.lk, bh, h, sk.start, k0 + x / 16, D) + c0 + 8 * (x % 16);
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dK) + e) = make_uint4(0, 0, 0, 0);
            *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dV) + e) = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    if ((smem_u32(smem) & 1023u) != 0) {   // the swizzled tiles need 1024-byte alignment
        if (threadIdx.x == 0 && p.dev_status != nullptr)
            atomicCAS(p.dev_status, 0, static_cast<int>(ATTN_ERR_CUDA));
        return;
    }

    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::OFF_BAR);
    uint64_t* bar_kv = bars + 0;
    uint64_t* full_q0 = bars + 1;     // Q_i, LSE_i, D_i loaded (stage i & 1; [1] at bars + 15)
    uint64_t* full_do = bars + 2;     // dO_i loaded
    uint64_t* empty_q0 = bars + 3;    // dK_h of the block done: its stage free ([1] at bars + 16)
    uint64_t* empty_do = bars + 4;    // dV_h of the block done (dO free)
    uint64_t* bar_S = bars + 5;       // S^T in TMEM
    uint64_t* bar_dP = bars + 6;      // dP^T in TMEM
    uint64_t* bar_P = bars + 7;       // [2] P of a warpgroup's 32 queries in TMEM
    uint64_t* bar_dS = bars + 9;      // [2] dS of a warpgroup's 32 queries in smem
    uint64_t* bar_dQ = bars + 11;     // dQ^T in TMEM
    uint64_t* bar_dQfree = bars + 12; // the dQ warps have read it out
    uint64_t* bar_dkdv = bars + 13;
    uint64_t* bar_fin = bars + 14;
    uint64_t* full_q1 = bars + 15;
    uint64_t* empty_q1 = bars + 16;
    auto full_q = [&](int st) { return st ? full_q1 : full_q0; };
    auto empty_q = [&](int st) { return st ? empty_q1 : empty_q0; };
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 17);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    float* sLSE = reinterpret_cast<float*>(smem + C::OFF_LSE);
    float* sD = reinterpret_cast<float*>(smem + C::OFF_D);

    if (threadIdx.x == 0) {
        mbar_init(bar_kv, 1);
        mbar_init(full_q0, 1);
        mbar_init(full_q1, 1);
        mbar_init(full_do, 1);
        mbar_init(empty_q0, 1);
        mbar_init(empty_q1, 1);
        mbar_init(empty_do, 1);
        mbar_init(bar_S, 1);
        mbar_init(bar_dP, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&bar_P[s], kTileRows);
            mbar_init(&bar_dS[s], kTileRows);
        }
        mbar_init(bar_dQ, 1);
        mbar_init(bar_dQfree, kTileRows);
        mbar_init(bar_dkdv, 1);
        mbar_init(bar_fin, 1);
        *s_abort = 0;
        fence_mbar_init();
    }
    if (warp == 13) {
        tmem_alloc(s_tmem, 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *s_tmem;

    if (warp == 12) {
        // ================= TMA producer =================
        if (lane == 0) {
            tma_prefetch_desc(&tmQ);
            tma_prefetch_desc(&tmK);
            tma_prefetch_desc(&tmV);
            tma_prefetch_desc(&tmdO);
            mbar_arrive_expect_tx(bar_kv, 2 * C::KTILE);
            int ky, kz;
            tma_rows_t<kPacked>(bh, h, sk.start, k0, ky, kz);
            for (int cb = 0; cb < C::NCB; ++cb) {
                tma_load_3d(smem + C::OFF_K + cb * C::KCB, &tmK, bar_kv, cb * 64, ky, kz);
                tma_load_3d(smem + C::OFF_V + cb * C::KCB, &tmV, bar_kv, cb * 64, ky, kz);
            }
            int do_issued = 0, q_issued = 0;
            for (int it = 0; it < nq; ++it) {
                const int qi = q_begin + it;
                const int st = it & 1;
                int qy, qz;
                tma_rows_t<kPacked>(bh, h, sq.start, qi * QR, qy, qz);
                // The owned half of Q_i with LSE_i, D_i into stage st once dK_h of
                // block i-2 is done; the other half once S of block i-1 has read
                // it; then dO_i once dV_h of block i-1 is done.  One arrival on
                // full_q(st) covers both halves.
                if (!mbar_wait(empty_q(st), ((it >> 1) & 1) ^ 1, s_abort)) break;
                mbar_arrive_expect_tx(full_q(st), C::QTILE + 2 * QR * 4);
                for (int c = 0; c < 2; ++c)
                    tma_load_3d(smem + C::OFF_QOWN + st * C::QHALF + c * C::QCB, &tmQ, full_q(st),
                                (2 * half + c) * 64, qy, qz);
                const size_t roff = static_cast<size_t>(bh) * p.Npad + static_cast<size_t>(qi) * QR;
                if (it == 0) grid_dep_wait();   // LSE and D come from the preprocess
                bulk_load(sLSE + st * QR, p.lse2 + roff, QR * 4, full_q(st));
                bulk_load(sD + st * QR, p.Drow + roff, QR * 4, full_q(st));
                // (the other half is issued even if the wait gives up, so that
                // the stage's phase can complete for the drain below)
                const bool s_ok = it == 0 || mbar_wait(bar_S, (it - 1) & 1, s_abort);
                for (int c = 0; c < 2; ++c)
                    tma_load_3d(smem + C::OFF_Q + c * C::QCB, &tmQ, full_q(st),
                                (2 * (1 - half) + c) * 64, qy, qz);
                ++q_issued;
                if (!s_ok) break;
                if (!mbar_wait(empty_do, (it & 1) ^ 1, s_abort)) break;
                mbar_arrive_expect_tx(full_do, C::QTILE);
                for (int cb = 0; cb < C::NCB; ++cb)
                    tma_load_3d(smem + C::OFF_DO + cb * C::QCB, &tmdO, full_do, cb * 64, qy, qz);
                ++do_issued;
            }
            // Drain: every copy issued has landed before teardown.
            volatile int no_abort = 0;
            mbar_wait(bar_kv, 0, &no_abort);
            if (do_issued > 0) mbar_wait(full_do, (do_issued - 1) & 1, &no_abort);
            for (int st = 0; st < 2 && st < q_issued; ++st) {
                const int uses = (q_issued - st + 1) / 2;
                mbar_wait(full_q(st), (uses - 1) & 1, &no_abort);
            }
        }
        __syncwarp();
    } else if (warp == 13) {
        // ================= MMA issuer =================
        if (lane == 0) {
            const uint64_t dK_k = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);   // K-major
            const uint64_t dV_k = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);
            // S^T reads Q as K-major column blocks: the owned half from its
            // stage buffer, the other half from the shared one
            const uint64_t dQo_k = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
            const uint64_t dQown_k0 = sdesc_sw128(smem_u32(smem + C::OFF_QOWN), 16, 1024);
            const uint64_t dO_k = sdesc_sw128(smem_u32(smem + C::OFF_DO), 16, 1024);
            // MN-major views of this CTA's half: Q_h, dO_h (N = 128 columns as two
            // 64-column blocks of a 64-row tile), K_h (M = 128 columns of a
            // 128-row tile) and dS^T (N = 64 queries, one column block)
            const uint64_t dQ_mn0 = sdesc_sw128(smem_u32(smem + C::OFF_QOWN), C::QCB, 1024);
            const uint64_t dO_mn = sdesc_sw128(smem_u32(smem + C::OFF_DO + 2 * half * C::QCB), C::QCB, 1024);
            const uint64_t dK_mn = sdesc_sw128(smem_u32(smem + C::OFF_K + 2 * half * C::KCB), C::KCB, 1024);
            const uint64_t dS_mn = sdesc_sw128(smem_u32(smem + C::OFF_DS), C::QCB, 1024);
            const uint64_t dS_k = sdesc_sw128(smem_u32(smem + C::OFF_DS), 16, 1024);   // keys as rows
            // Each group of MMAs goes out as runs of inline PTX (ptx.cuh) whose
            // descriptors advance by constants: 32 bytes per K step inside a
            // 128-byte column block, then on to the next column block.
            constexpr uint32_t KJ = C::KCB / 16 - 6, QJ = C::QCB / 16 - 6;
            // K = 256 as two runs over column blocks {0, 1} and {2, 3}; b_lo
            // and b_hi are the B operand's descriptors for the two pairs
            auto issue_full_d = [&](uint32_t d_tmem, uint64_t a_k, uint64_t b_lo, uint64_t b_hi) {
                mma8_ss_f16<2, 2, 2, KJ, 2, 2, 2, 2, 2, 2, QJ, 2, 2, 2>(d_tmem, a_k, b_lo, C::IDESC_SDP, 0u);
                mma8_ss_f16<2, 2, 2, KJ, 2, 2, 2, 2, 2, 2, QJ, 2, 2, 2>(
                    d_tmem, sdesc_adv(a_k, 2 * C::KCB), b_hi, C::IDESC_SDP, 1u);
            };
            bool ok = mbar_wait(bar_kv, 0, s_abort);
            for (int it = 0; it < nq && ok; ++it) {
                const uint32_t ph = it & 1;
                const int st = it & 1;
                const uint64_t dQown_k = sdesc_adv(dQown_k0, st * C::QHALF);
                const uint64_t dQ_mn = sdesc_adv(dQ_mn0, st * C::QHALF);
                // S^T = K Q^T and dP^T = V dO^T over the whole head dim
                ok = mbar_wait(full_q(st), (it >> 1) & 1, s_abort);
                if (!ok) break;
                tc_fence_after();
                issue_full_d(tmem + C::C_S, dK_k, half == 0 ? dQown_k : dQo_k,
                             half == 0 ? dQo_k : dQown_k);
                tc_commit(bar_S);
                ok = mbar_wait(full_do, ph, s_abort);
                if (!ok) break;
                tc_fence_after();
                issue_full_d(tmem + C::C_DP, dV_k, dO_k, sdesc_adv(dO_k, 2 * C::QCB));
                tc_commit(bar_dP);
                // dV_h += P^T dO_h, each warpgroup's 32 queries as soon as its P is in
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    ok = mbar_wait(&bar_P[hh], ph, s_abort);
                    if (!ok) break;
                    tc_fence_after();
#pragma unroll
                    for (int k2 = 0; k2 < 2; ++k2) {
                        const int kk = 2 * hh + k2;   // 16 queries
                        mma_ts<false>(tmem + C::C_DV, tmem + C::C_S + 32 * hh + 8 * k2,
                                      sdesc_adv(dO_mn, kk * 2048), C::IDESC_DKV,
                                      (it == 0 && kk == 0) ? 0u : 1u);
                    }
                }
                if (!ok) break;
                tc_commit(empty_do);
                // dK_h += dS^T Q_h and dQ^T_h = K_h^T dS^T once all of dS is in
                ok = mbar_wait(&bar_dS[0], ph, s_abort) && mbar_wait(&bar_dS[1], ph, s_abort);
                if (!ok) break;
                tc_fence_after();
                mma4_ss_f16<2, 2, 2, 128, 128, 128>(tmem + C::C_DK, dS_k, dQ_mn, C::IDESC_DKV,
                                                    it == 0 ? 0u : 1u);
                tc_commit(empty_q(st));
                if (it > 0) {   // the dQ warps have read the previous block's dQ^T
                    ok = mbar_wait(bar_dQfree, (it - 1) & 1, s_abort);
                    if (!ok) break;
                    tc_fence_after();
                }
                static_assert(kTileRows / 16 == 8, "dQ^T: 8 K steps of 16 keys");
                mma8_ss_f16<128, 128, 128, 128, 128, 128, 128, 128, 128, 128, 128, 128, 128, 128>(
                    tmem + C::C_DQ, dK_mn, dS_mn, C::IDESC_DQ, 0u);   // K = keys
                tc_commit(bar_dQ);
            }
            if (ok) tc_commit(bar_dkdv);
            tc_commit(bar_fin);
            volatile int no_abort = 0;
            mbar_wait(bar_fin, 0, &no_abort);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ================= compute: P and dS, one key row per thread =================
        const int hh = warp >> 2;          // which 32 queries of the block
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int j = k0 + r;
        const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t tS = tl + C::C_S + 32 * hh;
        const uint32_t tdP = tl + C::C_DP + 32 * hh;
        const bool row_valid = j < L;
        const int jo = j - off;   // this key's position on the query axis
        uint8_t* rowp = smem + C::OFF_DS + r * 128;
        bool ok = true;
        for (int it = 0; it < nq; ++it) {
            const uint32_t ph = it & 1;
            const int qi = q_begin + it;
            if (!mbar_wait_warp(bar_S, ph, s_abort) ||
                !mbar_wait_warp(full_q(it & 1), (it >> 1) & 1, s_abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float* lse_s = sLSE + (it & 1) * QR + 32 * hh;
            const float* d_s = sD + (it & 1) * QR + 32 * hh;
            const int q0h = qi * QR + 32 * hh;   // first query of this warpgroup's part
            const bool diag = kCausal && (k0 + kTileRows - 1 > qi * QR + off);
            const bool wmask = W > 0 && (qi * QR + QR - 1 + off - k0 >= W ||
                                         (!kCausal && k0 + kTileRows - 1 - qi * QR - off >= W));
            // ---- P from S (32 queries, two 16-column chunks) ----
            float pr[32];
            uint32_t keepw[2];
            uint32_t sv[32];
            tmem_ld32(tS, sv);
            tmem_ld_wait();
            reg_fence(sv);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t keep = 0xFFFFu;   // bit e: query 16c+e of this part kept
                if constexpr (kDropout)   // the octet of lanes sharing j & ~7 transposes its draws
                    keep = dropout_keep16_t(p.seed_lo, p.seed_hi, p.drop_threshold, q0h + 16 * c, j, h,
                                            b, lane);
                keepw[c] = keep;
                uint32_t pk[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float pd[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int col = 16 * c + 2 * e + u;
                        float x = ex2_approx(fmaf(__uint_as_float(sv[col]), p.scale_log2, lse_s[col]));
                        const int iq = q0h + col;
                        const bool valid = row_valid && (!diag || jo <= iq) &&
                                           (!wmask || (iq - jo < W && (kCausal || jo - iq < W)));
                        x = valid ? x : 0.f;
                        pr[col] = x;
                        pd[u] = x;
                        if constexpr (kDropout)
                            pd[u] = ((keep >> (2 * e + u)) & 1u) ? x * p.drop_scale : 0.f;
                    }
                    pk[e] = pack_h2<kF16>(pd[0], pd[1]);
                }
                tmem_st8(tS + 8 * c, pk);
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar_P[hh]);
            // ---- dS = P (dP Z/(1-p) - D) ----
            if (!mbar_wait_warp(bar_dP, ph, s_abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t dpv[32];
            tmem_ld32(tdP, dpv);
            tmem_ld_wait();
            reg_fence(dpv);
#pragma unroll
            for (int c = 0; c < 2; ++c) {
                uint32_t dk[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    float ds[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int col = 16 * c + 2 * e + u;
                        float dp = __uint_as_float(dpv[col]);
                        if constexpr (kDropout)
                            dp = ((keepw[c] >> (2 * e + u)) & 1u) ? dp * p.drop_scale : 0.f;
                        ds[u] = pr[col] * (dp - d_s[col]);
                    }
                    dk[e] = pack_h2<kF16>(ds[0], ds[1]);
                }
                // dS (16-bit) into shared memory: keys as rows, the 64 queries
                // of the block along a 128-byte row, 128-byte swizzle.  bar_dP
                // of this block also means every MMA of the previous block (the
                // dS readers dK and dQ among them) has completed.
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int chunk = (4 * hh + 2 * c + u) ^ (r & 7);
                    *reinterpret_cast<uint4*>(rowp + chunk * 16) =
                        make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar_dS[hh]);
        }
        // ---- epilogue: warpgroup 0 writes dK_h = scale * acc, warpgroup 1 dV_h ----
        if (ok) {
            ok = mbar_wait_warp(bar_dkdv, 0, s_abort);
            tc_fence_after();
        }
        // The Q (warpgroup 0) and dO (warpgroup 1) buffers are free once
        // bar_dkdv has fired: each holds one 128-row x 128-column tile as two
        // 128-byte-swizzled column blocks of 16 KB.
        uint8_t* stg = smem + (hh == 0 ? C::OFF_Q : C::OFF_DO);
        const bool direct = kPacked && k0 + kTileRows > Nk;   // last block of a packed sequence
        uint16_t* gout = static_cast<uint16_t*>(hh == 0 ? p.dK : p.dV);
        const bool row_in = k0 + r < Nk;
        const size_t grow = row_in ? act_offset_t<kPacked>(p.lk, bh, h, sk.start, k0 + r, D) + c0 : 0;
        if (ok) {
            const uint32_t src = tl + (hh == 0 ? C::C_DK : C::C_DV);
            const float mul = (hh == 0) ? p.scale : 1.f;
#pragma unroll 1
            for (int c = 0; c < 4; ++c) {   // 32 columns = half a 128-byte column block
                uint32_t a[32];
                tmem_ld32(src + 32 * c, a);
                tmem_ld_wait();
                reg_fence(a);
                uint8_t* rp = stg + (c >> 1) * C::KCB + r * 128;
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    uint32_t w[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        w[e] = pack_h2<kF16>(__uint_as_float(a[8 * q4 + 2 * e]) * mul,
                                             __uint_as_float(a[8 * q4 + 2 * e + 1]) * mul);
                    if (direct) {
                        if (row_in)
                            *reinterpret_cast<uint4*>(gout + grow + 32 * c + 8 * q4) =
                                make_uint4(w[0], w[1], w[2], w[3]);
                    } else {
                        const int chunk = (4 * (c & 1) + q4) ^ (r & 7);
                        *reinterpret_cast<uint4*>(rp + chunk * 16) = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
            fence_proxy_async_smem();
        }
        named_barrier_sync(1 + hh, 128);
        if (ok && !direct && quarter == 0 && lane == 0) {
            const CUtensorMap* m = (hh == 0) ? &tmdK : &tmdV;
            int y, z;
            tma_rows_t<kPacked>(bh, h, sk.start, k0, y, z);
            for (int cb = 0; cb < 2; ++cb) tma_store_3d(m, stg + cb * C::KCB, c0 + cb * 64, y, z);
            bulk_commit_group();
            bulk_wait_group_read_all();
        }
    } else {
        // ================= dQ: dQ^T out of TMEM, added into the workspace =================
        // lane = one of the 128 columns of this half; TMEM columns are the 64
        // queries of the block; each warp instruction adds 32 consecutive floats
        // of one query row.
        grid_dep_wait();   // the accumulator is cleared by the preprocess
        const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const int dc = c0 + (warp & 3) * 32 + lane;
        for (int it = 0; it < nq; ++it) {
            const int qi = q_begin + it;
            const size_t row0 = static_cast<size_t>(bh) * p.Npad + static_cast<size_t>(qi) * QR;
            const int nvalid = min(QR, N - qi * QR);
            if (!mbar_wait_warp(bar_dQ, it & 1, s_abort)) break;
            tc_fence_after();
            uint32_t x[2][32];
            tmem_ld32(tl + C::C_DQ, x[0]);
            tmem_ld32(tl + C::C_DQ + 32, x[1]);
            tmem_ld_wait();
            reg_fence(x[0]);
            reg_fence(x[1]);
            tc_fence_before();
            mbar_arrive(bar_dQfree);
            float* col = p.dq_acc + row0 * D + dc;
#pragma unroll
            for (int c = 0; c < 2; ++c)
#pragma unroll
                for (int e = 0; e < 32; ++e)
                    if (32 * c + e < nvalid)
                        red_add_f32(col + static_cast<size_t>(32 * c + e) * D, __uint_as_float(x[c][e]));
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 13) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0 && *s_abort && p.dev_status != nullptr)
        atomicCAS(p.dev_status, 0, static_cast<int>(ATTN_ERR_DEVICE_TIMEOUT));
}

template <bool kF16, bool kCausal, bool kDropout, bool kWindow, bool kPacked>
cudaError_t launch_bwd_d256_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdk,
                              const CUtensorMap& tdv, const BwdParams& p, cudaStream_t stream) {
    using C = Bwd256Cfg<kF16>;
    auto kern = attn_bwd_d256_kernel<kF16, kCausal, kDropout, kWindow, kPacked>;
    static std::atomic<unsigned long long> smem_ready{0};
    const cudaError_t e = enable_smem_per_device(kern, C::SMEM, smem_ready);
    if (e != cudaSuccess) return e;
    const unsigned grid = 2u * static_cast<unsigned>(p.nkb) * static_cast<unsigned>(p.B * p.H);
    return launch_overlapped(kern, grid, C::THREADS, C::SMEM, stream, tq, tk, tv, tdo, tdk, tdv, p);
}

template <bool kF16, bool kPacked, bool kWindow>
cudaError_t dispatch_bwd_d256_w(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                                const BwdParams& p, bool causal, bool dropout, cudaStream_t s) {
    if (causal)
        return dropout ? launch_bwd_d256_t<kF16, true, true, kWindow, kPacked>(tq, tk, tv, tdo, tdk, tdv, p, s)
                       : launch_bwd_d256_t<kF16, true, false, kWindow, kPacked>(tq, tk, tv, tdo, tdk, tdv, p, s);
    return dropout ? launch_bwd_d256_t<kF16, false, true, kWindow, kPacked>(tq, tk, tv, tdo, tdk, tdv, p, s)
                   : launch_bwd_d256_t<kF16, false, false, kWindow, kPacked>(tq, tk, tv, tdo, tdk, tdv, p, s);
}

template <bool kF16, bool kPacked>
cudaError_t dispatch_bwd_d256(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                              const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                              const BwdParams& p, bool causal, bool dropout, cudaStream_t s) {
    return p.window > 0
               ? dispatch_bwd_d256_w<kF16, kPacked, true>(tq, tk, tv, tdo, tdk, tdv, p, causal, dropout, s)
               : dispatch_bwd_d256_w<kF16, kPacked, false>(tq, tk, tv, tdo, tdk, tdv, p, causal, dropout, s);
}

}  // namespace
}  // namespace gbattn
