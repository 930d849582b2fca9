// attn_bwd_kernel.cuh — main kernel of the fused exact-attention backward
// for sm_103a (the preprocess and dQ conversion kernels are in attn_bwd.cu).
#pragma once

#include <cuda_bf16.h>

#include <type_traits>

#include "internal.h"
#include "philox.cuh"
#include "ptx.cuh"
#include "seq.cuh"

namespace gbattn {
namespace {

// ---------------------------------------------------------------------------
// main kernel
// ---------------------------------------------------------------------------
// One CTA per (head, 128-key block j).  K_j and V_j stay in shared memory;
// the CTA walks the query blocks i (from the diagonal on when causal):
//   S^T  = K_j Q_i^T          dP^T = V_j dO_i^T          (tcgen05, smem x smem)
//   P^T  = exp2(S^T scale log2e - LSE_i log2e)           (masked, dropout bits)
//   dS^T = P^T (dP^T Z/(1-p) - D_i)
//   dQ_i += dS K_j            (smem x smem, added into the fp32 workspace)
//   dV_j += (P Z/(1-p))^T dO_i                           (P read from TMEM)
//   dK_j += dS^T Q_i                                     (dS read from smem)
// dK_j (times scale) and dV_j leave the chip once, at the end.  Queries stand
// at key positions i + Nk - N (cross-attention), which shifts the causal and
// window bounds of the query-block range; rows of a packed sequence are
// located through seq.cuh, and the last key block of a packed sequence writes
// dK, dV row by row so that nothing lands in the next sequence's rows.
//
// Warp roles (448 threads):
//   warps 0-3  compute, query columns 0-63 of the block: one thread per key
//              row (TMEM lane) builds P and dS
//   warps 4-7  compute, query columns 64-127
//   warps 8-11 dQ: read dQ out of TMEM and add it into the fp32 workspace
//              with fire-and-forget reductions (d = 64: one thread per query
//              row, 16-byte adds; d = 128: one thread per head-dim column,
//              one 128-byte contiguous add per warp instruction)
//   warp  12   TMA producer: K_j, V_j once; Q_i, dO_i, LSE_i, D_i per block
//   warp  13   MMA issuer.  S^T and dP^T are committed separately: the
//              compute warps build P from S^T while dP^T runs, dV for each
//              query half starts as soon as its P is in TMEM, and dQ and dK
//              for each half as soon as its dS is in shared memory.  Across
//              blocks the issue order is  dV_i, S_{i+1}, dK_i, dQ_i, dP_{i+1}
//              at d = 64 and  dV_i, dQ_i and dK_i of query half 0, S_{i+1},
//              dQ_i and dK_i of half 1, dP_{i+1}  at d = 128, where the dQ
//              warps' fp32 adds (64 KB a block) set the pace: their first
//              half is handed over as early as possible.
//
// Tensor memory (512 columns):
//   d = 64:  dK [0,64) dV [64,128) S [128,256) dP [256,384) dQ [384,448)
//   d = 128: dK [0,128) dV [128,256) S [256,384) dP [384,512); dQ^T reuses
//            the dP columns, so the next dP^T waits until the dQ warps have
//            read it out.
// Each compute warpgroup writes its P (bf16 pairs) over the first 32 columns
// of its 64-column half of S.  dS goes to shared memory only: it is the
// MN-major operand of the dQ product and, read as K-major with keys as rows,
// the A operand of dK += dS^T Q.
template <int D, bool kF16>
struct BwdCfg {
    static constexpr int THREADS = 448;
    static constexpr int ROWB = D * 2;
    static constexpr int NCB = ROWB / 128;
    static constexpr int TILE = kTileRows * ROWB;
    static constexpr int CB_BYTES = kTileRows * 128;
    static constexpr int HALF_BYTES = CB_BYTES / 2;   // 64 rows of one 128-byte column block
    static constexpr int DS_BYTES = kTileRows * kTileRows * 2;
    static constexpr int OFF_K = 0;
    static constexpr int OFF_V = TILE;
    static constexpr int OFF_Q = 2 * TILE;    // 2 stages
    static constexpr int OFF_DO = 4 * TILE;   // 2 stages
    static constexpr int OFF_DS = 6 * TILE;
    static constexpr int OFF_LSE = OFF_DS + DS_BYTES;   // [2][128] float
    static constexpr int OFF_D = OFF_LSE + 1024;        // [2][128] float
    static constexpr int OFF_BAR = OFF_D + 1024;
    static constexpr int SMEM = OFF_BAR + 256;
    static constexpr int QK_STEPS = ROWB / 32;
    static constexpr uint32_t C_DK = 0;
    static constexpr uint32_t C_DV = D;
    static constexpr uint32_t C_S = 2 * D;
    static constexpr uint32_t C_DP = 2 * D + 128;
    // dQ, fp32: its own columns for d = 64; for d = 128 it reuses the dP
    // columns, which are free once P and dS have been built.
    static constexpr uint32_t C_DQ = (D == 64) ? 2 * D + 256 : C_DP;
    static constexpr uint32_t FMT = fmt16<kF16>();   // every operand has the storage type
    static constexpr uint32_t IDESC_SDP = idesc_f32acc(128, 128, FMT, false, false);
    static constexpr uint32_t IDESC_DP_HALF = idesc_f32acc(128, 64, FMT, false, false);
    static constexpr uint32_t IDESC_DKV = idesc_f32acc(128, D, FMT, false, true);
    // d = 64: dQ = dS K (lanes = queries, N = 64).  d = 128: dQ^T = K^T dS^T
    // (lanes = head-dim columns), one N = 64 product per query half.
    static constexpr uint32_t IDESC_DQ = idesc_f32acc(128, 64, FMT, true, true);
    static_assert(SMEM <= 232448, "shared memory budget");
};

template <int D, bool kF16, bool kCausal, bool kDropout, bool kWindow, bool kPacked>
__global__ void __launch_bounds__(448, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ,
                    const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV,
                    const __grid_constant__ CUtensorMap tmdO,
                    const __grid_constant__ CUtensorMap tmdK,
                    const __grid_constant__ CUtensorMap tmdV, const BwdParams p) {
    using C = BwdCfg<D, kF16>;
    extern __shared__ __align__(1024) uint8_t smem[];
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // Launched overlapped with the preprocess: K, V, Q and dO (inputs) load
    // while it finishes; the workspace it writes (LSE, D, the cleared dQ
    // accumulator) and the outputs are touched only after grid_dep_wait().
    grid_dep_launch_dependents();

    const int BH = p.B * p.H;
    int kb, bh;   // causal: key block 0 meets every query block, so rank 0 is heaviest
    grouped_schedule(static_cast<int>(blockIdx.x), BH, p.nkb, bh, kb);
    const int b = bh / p.H, h = bh % p.H;
    // rows of this sequence: all N (Nk) when dense; when packed, the
    // sequence's own token range
    const bool report = threadIdx.x == 0 && h == 0 && kb == 0;
    const SeqSpan sq = kPacked ? seq_span(p.lq, b, p.dev_status, report) : SeqSpan{0, p.N};
    const SeqSpan sk = kPacked ? seq_span(p.lk, b, p.dev_status, report) : SeqSpan{0, p.Nk};
    const int N = sq.len;    // query rows
    const int Nk = sk.len;   // keys
    // Queries continue the key sequence: query i stands at key position
    // i + off for the causal and window tests (off = 0 when N == Nk).
    const int off = Nk - N;
    const int nqb = (N + kTileRows - 1) / kTileRows;
    int L = Nk;
    if (p.key_lens != nullptr) {
        const int raw = p.key_lens[b];
        L = raw < 0 ? 0 : (raw > Nk ? Nk : raw);
        if (raw != L && threadIdx.x == 0 && p.dev_status != nullptr)
            atomicCAS(p.dev_status, 0, static_cast<int>(ATTN_ERR_INVALID_ARG));
    }
    const int k0 = kb * kTileRows;
    // Query blocks that see some key of this block: from the diagonal on when
    // causal; a sliding window of W keys also bounds them from the other side.
    const int W = kWindow ? p.window : 0;   // compile-time 0 without a window
    int q_begin = kCausal ? max(0, k0 - off) / kTileRows : 0;
    int q_end = nqb;
    if (W > 0) {
        const int last_q = k0 + kTileRows - 1 - off + W - 1;   // last query the block's keys reach
        q_end = last_q < 0 ? 0 : min(nqb, last_q / kTileRows + 1);
        if (!kCausal) q_begin = max(0, k0 - off - W + 1) / kTileRows;
    }
    const int nq = q_end - q_begin;
    if (k0 >= L || nq <= 0) {   // no key of this block is attended: dK = dV = 0
        grid_dep_wait();
        const int rows = min(kTileRows, Nk - k0);
        constexpr int kRow16 = D / 8;   // uint4 per row
        for (int x = threadIdx.x; x < rows * kRow16; x += blockDim.x) {
            const size_t e = act_offset_t<kPacked>(p.lk, bh, h, sk.start, k0 + x / kRow16, D) + 8 * (x % kRow16);
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
    uint64_t* full_q = bars + 1;      // [2]
    // bars + 3, bars + 4: unused (a Q/dO stage is released by bar_dP[0])
    uint64_t* bar_S = bars + 5;       // S^T in TMEM
    uint64_t* bar_P = bars + 6;       // [2] P of a query half in TMEM (one per warpgroup)
    uint64_t* bar_dQ = bars + 8;       // [2] dQ (d = 128: each query half of dQ^T) in TMEM
    uint64_t* bar_dQfree = bars + 10;  // [2] the dQ warps have read it out
    uint64_t* bar_dkdv = bars + 12;
    uint64_t* bar_fin = bars + 13;
    uint64_t* bar_dP = bars + 14;      // [2] dP^T of a query half in TMEM
    uint64_t* bar_dS = bars + 16;      // [2] dS of a query half in smem
    uint32_t* s_tmem = reinterpret_cast<uint32_t*>(bars + 18);
    volatile int* s_abort = reinterpret_cast<volatile int*>(s_tmem + 1);
    float* sLSE = reinterpret_cast<float*>(smem + C::OFF_LSE);
    float* sD = reinterpret_cast<float*>(smem + C::OFF_D);

    if (threadIdx.x == 0) {
        mbar_init(bar_kv, 1);
        for (int s = 0; s < 2; ++s) {
            mbar_init(&full_q[s], 1);
            mbar_init(&bar_P[s], kTileRows);
            mbar_init(&bar_dS[s], kTileRows);
            mbar_init(&bar_dP[s], 1);
            mbar_init(&bar_dQ[s], 1);
            mbar_init(&bar_dQfree[s], kTileRows);
        }
        mbar_init(bar_S, 1);
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
            mbar_arrive_expect_tx(bar_kv, 2 * C::TILE);
            int ky, kz;
            tma_rows_t<kPacked>(bh, h, sk.start, k0, ky, kz);
            for (int cb = 0; cb < C::NCB; ++cb) {
                tma_load_3d(smem + C::OFF_K + cb * C::CB_BYTES, &tmK, bar_kv, cb * 64, ky, kz);
                tma_load_3d(smem + C::OFF_V + cb * C::CB_BYTES, &tmV, bar_kv, cb * 64, ky, kz);
            }
            int issued = 0;
            for (int it = 0; it < nq; ++it) {
                const int stage = it & 1;
                // The stage's previous block (it - 2) is done with it once dK of
                // that block has run, which the commit of the next dP^T half 0
                // (dP of block it - 1, completion it - 1 of bar_dP[0]) covers:
                // the MMA warp spends no commit of its own on the release.
                // (A parity wait must name the phase in progress or the one just
                // completed: block 2 first waits for completion 0, after which
                // each block's wait is at most one phase ahead of the last.)
                if (it == 2 && !mbar_wait(&bar_dP[0], 0, s_abort)) break;
                if (it >= 2 && !mbar_wait(&bar_dP[0], (it - 1) & 1, s_abort)) break;
                const int qi = q_begin + it;
                mbar_arrive_expect_tx(&full_q[stage], 2 * C::TILE + 1024);
                int qy, qz;
                tma_rows_t<kPacked>(bh, h, sq.start, qi * kTileRows, qy, qz);
                for (int cb = 0; cb < C::NCB; ++cb) {
                    tma_load_3d(smem + C::OFF_Q + stage * C::TILE + cb * C::CB_BYTES, &tmQ,
                                &full_q[stage], cb * 64, qy, qz);
                    tma_load_3d(smem + C::OFF_DO + stage * C::TILE + cb * C::CB_BYTES, &tmdO,
                                &full_q[stage], cb * 64, qy, qz);
                }
                const size_t roff = static_cast<size_t>(bh) * p.Npad + static_cast<size_t>(qi) * kTileRows;
                if (it == 0) grid_dep_wait();   // LSE and D come from the preprocess
                bulk_load(sLSE + stage * kTileRows, p.lse2 + roff, 512, &full_q[stage]);
                bulk_load(sD + stage * kTileRows, p.Drow + roff, 512, &full_q[stage]);
                ++issued;
            }
            volatile int no_abort = 0;
            mbar_wait(bar_kv, 0, &no_abort);
            for (int s = 0; s < 2 && s < issued; ++s) {
                const int uses = (issued - s + 1) / 2;
                mbar_wait(&full_q[s], (uses - 1) & 1, &no_abort);
            }
        }
        __syncwarp();
    } else if (warp == 13) {
        // ================= MMA issuer =================
        if (lane == 0) {
            // Descriptor bases built once; each MMA only adds a constant.
            const uint64_t dK_k = sdesc_sw128(smem_u32(smem + C::OFF_K), 16, 1024);    // K-major
            const uint64_t dV_k = sdesc_sw128(smem_u32(smem + C::OFF_V), 16, 1024);
            const uint64_t dK_mn = sdesc_sw128(smem_u32(smem + C::OFF_K), C::CB_BYTES, 1024);
            const uint64_t dS_mn = sdesc_sw128(smem_u32(smem + C::OFF_DS), C::CB_BYTES, 1024);
            const uint64_t dS_k = sdesc_sw128(smem_u32(smem + C::OFF_DS), 16, 1024);  // keys as rows
            const uint64_t dQ_k0 = sdesc_sw128(smem_u32(smem + C::OFF_Q), 16, 1024);
            const uint64_t dQ_mn0 = sdesc_sw128(smem_u32(smem + C::OFF_Q), C::CB_BYTES, 1024);
            const uint64_t dO_k0 = sdesc_sw128(smem_u32(smem + C::OFF_DO), 16, 1024);
            const uint64_t dO_mn0 = sdesc_sw128(smem_u32(smem + C::OFF_DO), C::CB_BYTES, 1024);
            // dV += P^T dO (P from TMEM) and dK += dS^T Q (dS from smem) over the
            // query columns [64 hh, 64 hh + 64)
            // Each group of MMAs is issued as one run (ptx.cuh): the MMA warp
            // shares its sub-partition with busy compute warps, so its own
            // instruction count sets how fast the products reach the queue.
            constexpr uint32_t CB = C::CB_BYTES / 16 - 6;   // K-major: next column block after 4 steps
            auto issue_dv_half = [&](int hh, uint64_t do_mn, bool first) {
                // dV += P^T dO: 4 x 16 queries, P from TMEM, dO MN-major
                mma_run_ts_f16<4, 8, 128>(tmem + C::C_DV, tmem + C::C_S + 64 * hh,
                                          sdesc_adv(do_mn, 4 * hh * 2048), C::IDESC_DKV,
                                          first ? 0u : 1u);
            };
            auto issue_dk_half = [&](int hh, uint64_t q_mn, bool first) {
                // dK += dS^T Q: A = dS read with keys as rows (32-byte steps), Q MN-major
                mma4_ss_f16<2, 2, 2, 128, 128, 128>(tmem + C::C_DK, sdesc_adv(dS_k, hh * C::CB_BYTES),
                                                    sdesc_adv(q_mn, 4 * hh * 2048), C::IDESC_DKV,
                                                    first ? 0u : 1u);
            };
            auto issue_s = [&](int stage) {   // S^T = K Q^T
                const uint64_t q_k = sdesc_adv(dQ_k0, stage * C::TILE);
                if constexpr (C::QK_STEPS == 8)
                    mma8_ss_f16<2, 2, 2, CB, 2, 2, 2, 2, 2, 2, CB, 2, 2, 2>(tmem + C::C_S, dK_k, q_k,
                                                                          C::IDESC_SDP, 0u);
                else
                    mma4_ss_f16<2, 2, 2, 2, 2, 2>(tmem + C::C_S, dK_k, q_k, C::IDESC_SDP, 0u);
            };
            // dP^T = V dO^T for the query columns [64 hh, 64 hh + 64) (N = 64:
            // B is rows 64 hh.. of the dO tile)
            auto issue_dp_half = [&](int stage, int hh) {
                const uint64_t do_k = sdesc_adv(dO_k0, stage * C::TILE + hh * C::HALF_BYTES);
                if constexpr (C::QK_STEPS == 8)
                    mma8_ss_f16<2, 2, 2, CB, 2, 2, 2, 2, 2, 2, CB, 2, 2, 2>(
                        tmem + C::C_DP + 64 * hh, dV_k, do_k, C::IDESC_DP_HALF, 0u);
                else
                    mma4_ss_f16<2, 2, 2, 2, 2, 2>(tmem + C::C_DP + 64 * hh, dV_k, do_k,
                                                  C::IDESC_DP_HALF, 0u);
            };
            // dP^T of block it_prev + 1, half by half.  d = 128: the next dP^T
            // half may only land once the dQ warps have read the dQ^T half that
            // shares its columns, and P of a half is usually in before that, so
            // each dP^T half is followed by the block's dV += P^T dO for the
            // same query half, which fills the tensor pipe while the dQ warps
            // drain dQ (0.9% faster at C3, 1% slower with 512- and 1024-key
            // windows, whose CTAs walk few blocks; testing for P without
            // waiting and otherwise leaving dV for the top of the iteration was
            // 1% slower at C3).  dV of the second half waits until dQ and dK of
            // the first half are issued: the dQ warps, the slowest path, get
            // their dQ^T half sooner (0.6% faster at C3).  d = 64 has no such
            // wait, and there dV goes at the top of the block's iteration
            // (interleaving it delayed the second dP^T half: 5% slower at C5).
            constexpr bool kDvInDp = D == 128;
            bool dv1_late = false;
            auto issue_dp = [&](int stage, int it_prev) {
                const int itb = it_prev + 1;
                const uint64_t do_mn = sdesc_adv(dO_mn0, stage * C::TILE);
                auto issue_dv = [&](int hh) {
                    if (!mbar_wait(&bar_P[hh], itb & 1, s_abort)) return false;
                    tc_fence_after();
                    issue_dv_half(hh, do_mn, itb == 0 && hh == 0);
                    return true;
                };
                // A CTA's first block has no dQ^T to wait for: both its dP^T
                // halves go at once (the start-up is on the critical path), dV
                // after them.
                const bool interleave = kDvInDp && it_prev >= 0;
                dv1_late = interleave;   // dV of the second half follows dQ, dK of half 0
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    if (D == 128 && it_prev >= 0 &&
                        !mbar_wait(&bar_dQfree[hh], it_prev & 1, s_abort))
                        return false;
                    tc_fence_after();
                    issue_dp_half(stage, hh);
                    tc_commit(&bar_dP[hh]);
                    if (interleave && hh == 0 && !issue_dv(0)) return false;
                }
                if (kDvInDp && !interleave)
                    for (int hh = 0; hh < 2; ++hh)
                        if (!issue_dv(hh)) return false;
                return true;
            };
            // Software pipeline over query blocks: S^T of block i+1 is issued
            // behind dV of block i (the tensor pipe runs one thread's MMAs in
            // issue order, so it reads P_i before S^T_{i+1} overwrites it), and
            // dP^T of block i+1 right behind dQ and dK of block i, each half of
            // it followed by dV of block i+1 for that half.  The compute warps
            // then find the next S^T on its way while they build dS.
            bool ok = mbar_wait(bar_kv, 0, s_abort) && mbar_wait(&full_q[0], 0, s_abort);
            if (ok) {
                tc_fence_after();
                issue_s(0);
                tc_commit(bar_S);
                ok = issue_dp(0, -1);
            }
            for (int it = 0; it < nq && ok; ++it) {
                const int stage = it & 1;
                const bool more = it + 1 < nq;
                const int nstage = stage ^ 1;
                const uint64_t q_mn = sdesc_adv(dQ_mn0, stage * C::TILE);
                if constexpr (!kDvInDp) {
                    const uint64_t do_mn = sdesc_adv(dO_mn0, stage * C::TILE);
#pragma unroll
                    for (int hh = 0; hh < 2; ++hh) {   // dV += P^T dO as each half of P is in
                        ok = mbar_wait(&bar_P[hh], it & 1, s_abort);
                        if (!ok) break;
                        tc_fence_after();
                        issue_dv_half(hh, do_mn, it == 0 && hh == 0);
                    }
                    if (!ok) break;
                }
                auto issue_next_s = [&]() {
                    ok = mbar_wait(&full_q[nstage], ((it + 1) >> 1) & 1, s_abort);
                    if (!ok) return;
                    tc_fence_after();
                    issue_s(nstage);
                    tc_commit(bar_S);
                };
                // d = 64: the next S^T right behind dV (the compute warps need it
                // soonest); d = 128: after dQ and dK of the first query half, so
                // that dQ^T half 0 (which the dQ warps then drain) goes first
                if (D == 64 && more) {
                    issue_next_s();
                    if (!ok) break;
                }
                // d = 128: dQ^T = K^T dS^T for one query half needs only that
                // half of dS, so it follows dK of the half straight away.
                auto issue_dq_half = [&](int hh) {   // K = keys, 8 x 16 rows
                    mma8_ss_f16<128, 128, 128, 128, 128, 128, 128, 128, 128, 128, 128, 128, 128, 128>(
                        tmem + C::C_DQ + 64 * hh, dK_mn, sdesc_adv(dS_mn, hh * C::CB_BYTES), C::IDESC_DQ, 0u);
                    tc_commit(&bar_dQ[hh]);
                };
                ok = mbar_wait(&bar_dS[0], it & 1, s_abort);
                if (!ok) break;
                tc_fence_after();
                if constexpr (D == 128) issue_dq_half(0);
                issue_dk_half(0, q_mn, it == 0);
                if (dv1_late) {   // before S^T of the next block overwrites P
                    ok = mbar_wait(&bar_P[1], it & 1, s_abort);
                    if (!ok) break;
                    tc_fence_after();
                    issue_dv_half(1, sdesc_adv(dO_mn0, stage * C::TILE), false);
                    dv1_late = false;
                }
                if (D == 128 && more) {
                    issue_next_s();
                    if (!ok) break;
                }
                ok = mbar_wait(&bar_dS[1], it & 1, s_abort);
                if (ok && D == 64 && it > 0) ok = mbar_wait(&bar_dQfree[0], (it - 1) & 1, s_abort);
                if (!ok) break;
                tc_fence_after();
                if constexpr (D == 64) {   // dQ = dS K (lanes = queries), K = keys
                    mma8_ss_f16<128, 128, 128, 128, 128, 128, 128, 128, 128, 128, 128, 128, 128, 128>(
                        tmem + C::C_DQ, dS_mn, dK_mn, C::IDESC_DQ, 0u);
                    tc_commit(&bar_dQ[0]);
                } else {
                    issue_dq_half(1);
                }
                issue_dk_half(1, q_mn, false);   // runs while the dQ warps drain dQ
                if (more) {
                    // dP^T of the next block.  Its commits also cover dK and dQ
                    // of this block: when they fire, the dS buffer is free.
                    ok = issue_dp(nstage, it);
                    if (!ok) break;
                }
            }
            if (ok) tc_commit(bar_dkdv);
            tc_commit(bar_fin);
            volatile int no_abort = 0;
            mbar_wait(bar_fin, 0, &no_abort);
        }
        __syncwarp();
    } else if (warp < 8) {
        // ================= compute: P and dS, one key row per thread =================
        const int hh = warp >> 2;          // query-column half of this warpgroup
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const int j = k0 + r;
        const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t tS = tl + C::C_S + 64 * hh;
        const uint32_t tdP = tl + C::C_DP + 64 * hh;   // this half's dP^T columns
        const bool row_valid = j < L;
        const bool warp_has_invalid_row = __any_sync(0xffffffffu, !row_valid);
        const int jo = j - off;   // this key's position on the query axis
        uint8_t* rowp = smem + C::OFF_DS + hh * C::CB_BYTES + r * 128;
        bool ok = true;
        for (int it = 0; it < nq; ++it) {
            const int stage = it & 1;
            const uint32_t ph = (it >> 1) & 1;
            const int qi = q_begin + it;
            // Keep bits of this key against the half's 64 queries (16 per
            // chunk), drawn before S^T is awaited: they do not depend on it.
            uint32_t keepw[4] = {0xFFFFu, 0xFFFFu, 0xFFFFu, 0xFFFFu};
            if constexpr (kDropout) {
#pragma unroll
                for (int c = 0; c < 4; ++c)   // the octet of lanes sharing j & ~7 transposes its draws
                    keepw[c] = dropout_keep16_t(p.seed_lo, p.seed_hi, p.drop_threshold,
                                                qi * kTileRows + 64 * hh + 16 * c, j, h, b, lane);
            }
            if (!mbar_wait_warp(bar_S, it & 1, s_abort) ||
                !mbar_wait_warp(&full_q[stage], ph, s_abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const float* lse_s = sLSE + stage * kTileRows + 64 * hh;
            const float* d_s = sD + stage * kTileRows + 64 * hh;
            const int q0h = qi * kTileRows + 64 * hh;   // first query of this half
            // some key of this block lies past some query's causal limit
            const bool diag = kCausal && (k0 + kTileRows - 1 > qi * kTileRows + off);
            // some (query, key) pair of this block lies outside the window
            const bool wmask = W > 0 && (qi * kTileRows + kTileRows - 1 + off - k0 >= W ||
                                         (!kCausal && k0 + kTileRows - 1 - qi * kTileRows - off >= W));
            // ---- phase 1 (while dP^T is still on the tensor pipe): P from S ----
            // 16-column chunks; the next chunk's TMEM load overlaps this chunk's
            // math.  P (undropped, fp32) stays in registers for phase 2.  The
            // exponents scale s - LSE log2e are formed two columns per
            // instruction; blocks without a masked pair take a copy of the loop
            // with no mask tests.
            float pr[64];
            uint32_t buf[2][16];
            const uint64_t scale2 = f2_pack(p.scale_log2, p.scale_log2);
            auto phase1 = [&](auto masked_tag) {
                constexpr bool kMasked = decltype(masked_tag)::value;
                tmem_ld16(tS, buf[0]);
                tmem_ld_wait();
                reg_fence(buf[0]);
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    if (c < 3) tmem_ld16(tS + 16 * (c + 1), buf[(c + 1) & 1]);
                    const uint32_t* sv = buf[c & 1];
                    const uint32_t keep = keepw[c];   // bit e: column 16c+e of this half kept
                    float nl[16];   // this chunk's -LSE log2e values, four 16-byte shared loads
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        const float4 t4 = reinterpret_cast<const float4*>(lse_s + 16 * c)[v];
                        nl[4 * v] = t4.x;
                        nl[4 * v + 1] = t4.y;
                        nl[4 * v + 2] = t4.z;
                        nl[4 * v + 3] = t4.w;
                    }
                    uint32_t pk[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int col = 16 * c + 2 * e;
                        float x[2];
                        f2_unpack(f2_fma(f2_pack(__uint_as_float(sv[2 * e]), __uint_as_float(sv[2 * e + 1])),
                                         scale2, f2_pack(nl[2 * e], nl[2 * e + 1])),
                                  x[0], x[1]);
                        float pd[2];
#pragma unroll
                        for (int u = 0; u < 2; ++u) {
                            x[u] = ex2_approx(x[u]);
                            if constexpr (kMasked) {
                                const int iq = q0h + col + u;   // query index
                                const bool valid = row_valid && (!diag || jo <= iq) &&
                                                   (!wmask || (iq - jo < W && (kCausal || jo - iq < W)));
                                x[u] = valid ? x[u] : 0.f;
                            }
                            pr[col + u] = x[u];
                            pd[u] = x[u];
                            if constexpr (kDropout)
                                pd[u] = ((keep >> (2 * e + u)) & 1u) ? x[u] * p.drop_scale : 0.f;
                        }
                        pk[e] = pack_h2<kF16>(pd[0], pd[1]);
                    }
                    tmem_st8(tS + 8 * c, pk);
                    if (c < 3) {
                        tmem_ld_wait();
                        reg_fence(buf[(c + 1) & 1]);
                    }
                }
            };
            // The choice must be the same in all 32 lanes: the tensor-memory
            // loads and stores and the shuffles inside are warp-collective.
            if (diag || wmask || warp_has_invalid_row)
                phase1(std::true_type{});
            else
                phase1(std::false_type{});
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(&bar_P[hh]);

            // ---- phase 2: dS = P (dP Z/(1-p) - D) once dP^T is in ----
            if (!mbar_wait_warp(&bar_dP[hh], it & 1, s_abort)) {
                ok = false;
                break;
            }
            tc_fence_after();
            tmem_ld16(tdP, buf[0]);
            tmem_ld_wait();
            reg_fence(buf[0]);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (c < 3) tmem_ld16(tdP + 16 * (c + 1), buf[(c + 1) & 1]);
                const uint32_t* dpv = buf[c & 1];
                float dv[16];   // this chunk's D values
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    const float4 t4 = reinterpret_cast<const float4*>(d_s + 16 * c)[v];
                    dv[4 * v] = t4.x;
                    dv[4 * v + 1] = t4.y;
                    dv[4 * v + 2] = t4.z;
                    dv[4 * v + 3] = t4.w;
                }
                uint32_t dk[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {   // two columns per instruction
                    const int col = 16 * c + 2 * e;
                    float dp[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        dp[u] = __uint_as_float(dpv[2 * e + u]);
                        if constexpr (kDropout)
                            dp[u] = ((keepw[c] >> (2 * e + u)) & 1u) ? dp[u] * p.drop_scale : 0.f;
                    }
                    float ds[2];
                    f2_unpack(f2_mul(f2_pack(pr[col], pr[col + 1]),
                                     f2_sub(f2_pack(dp[0], dp[1]), f2_pack(dv[2 * e], dv[2 * e + 1]))),
                              ds[0], ds[1]);
                    dk[e] = pack_h2<kF16>(ds[0], ds[1]);
                }
                // dS (bf16) into shared memory: query index innermost (one
                // 64-query block per half), 128-byte swizzle.  bar_dP of this
                // block also means every MMA of the previous block (among them
                // the buffer's readers, dK and dQ) has completed.
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int chunk = (2 * c + u) ^ (r & 7);
                    *reinterpret_cast<uint4*>(rowp + chunk * 16) =
                        make_uint4(dk[4 * u], dk[4 * u + 1], dk[4 * u + 2], dk[4 * u + 3]);
                }
                if (c < 3) {
                    tmem_ld_wait();
                    reg_fence(buf[(c + 1) & 1]);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(&bar_dS[hh]);
        }
        // ---- epilogue: warpgroup 0 writes dK = scale * acc, warpgroup 1 dV ----
        // Each thread puts its key row (bf16) into the freed Q stage buffers in
        // the tensor map's 128-byte swizzled layout; one thread per warpgroup
        // then stores the whole 128-row tile with TMA (full-line writes; rows
        // past N are clipped by the map).
        if (ok) {
            ok = mbar_wait_warp(bar_dkdv, 0, s_abort);
            tc_fence_after();
        }
        uint8_t* stg = smem + C::OFF_Q + hh * C::TILE;   // free once bar_dkdv has fired
        // The last block of a packed sequence is written row by row: a TMA
        // store of the whole box would also write the next sequence's rows.
        const bool direct = kPacked && k0 + kTileRows > Nk;
        uint16_t* gout = static_cast<uint16_t*>(hh == 0 ? p.dK : p.dV);
        const bool row_in = k0 + r < Nk;
        const size_t grow = row_in ? act_offset_t<kPacked>(p.lk, bh, h, sk.start, k0 + r, D) : 0;
        if (ok) {
            const uint32_t src = tl + (hh == 0 ? C::C_DK : C::C_DV);
            const float mul = (hh == 0) ? p.scale : 1.f;
#pragma unroll 1
            for (int c = 0; c < D / 32; ++c) {   // 32 columns = half a 128-byte column block
                uint32_t a[32];
                tmem_ld32(src + 32 * c, a);
                tmem_ld_wait();
                reg_fence(a);
                uint8_t* rowp = stg + (c >> 1) * C::CB_BYTES + r * 128;
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
                        *reinterpret_cast<uint4*>(rowp + chunk * 16) =
                            make_uint4(w[0], w[1], w[2], w[3]);
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
            for (int cb = 0; cb < C::NCB; ++cb) tma_store_3d(m, stg + cb * C::CB_BYTES, cb * 64, y, z);
            bulk_commit_group();
            bulk_wait_group_read_all();
        }
    } else {
        // ================= dQ: read dQ out of TMEM, add into the workspace =================
        grid_dep_wait();   // the accumulator is cleared by the preprocess
        const uint32_t tl = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        for (int it = 0; it < nq; ++it) {
            const size_t row0 = static_cast<size_t>(bh) * p.Npad + static_cast<size_t>(q_begin + it) * kTileRows;
            if constexpr (D == 64) {
                // lane = query row rq; 64 head-dim columns as 16-byte adds
                if (!mbar_wait_warp(&bar_dQ[0], it & 1, s_abort)) break;
                tc_fence_after();
                const int rq = (warp & 3) * 32 + lane;
                uint32_t x[2][32];
                tmem_ld32(tl + C::C_DQ, x[0]);
                tmem_ld32(tl + C::C_DQ + 32, x[1]);
                tmem_ld_wait();
                reg_fence(x[0]);
                reg_fence(x[1]);
                tc_fence_before();
                mbar_arrive(&bar_dQfree[0]);
                if ((q_begin + it) * kTileRows + rq < N) {
                    float* dst = p.dq_acc + (row0 + rq) * D;
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int v = 0; v < 8; ++v)
                            red_add_v4(dst + 32 * c + 4 * v, __uint_as_float(x[c][4 * v]),
                                       __uint_as_float(x[c][4 * v + 1]),
                                       __uint_as_float(x[c][4 * v + 2]),
                                       __uint_as_float(x[c][4 * v + 3]));
                }
            } else {
                // lane = head-dim column dc; TMEM columns are queries.  Each
                // query half goes to registers whole, so its columns are released
                // (for the next dP^T half) before the reductions start; each warp
                // instruction then adds one query row's 32 consecutive floats.
                // Holding one half (64 values) rather than all 128 keeps the
                // warp inside its register budget.
                const int dc = (warp & 3) * 32 + lane;
                const int nvalid = min(kTileRows, N - (q_begin + it) * kTileRows);
                float* col = p.dq_acc + row0 * D + dc;
                bool ok = true;
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    if (!mbar_wait_warp(&bar_dQ[hh], it & 1, s_abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    uint32_t x[2][32];
                    tmem_ld32(tl + C::C_DQ + 64 * hh, x[0]);
                    tmem_ld32(tl + C::C_DQ + 64 * hh + 32, x[1]);
                    tmem_ld_wait();
                    reg_fence(x[0]);
                    reg_fence(x[1]);
                    tc_fence_before();
                    mbar_arrive(&bar_dQfree[hh]);
                    const int nv = nvalid - 64 * hh;   // valid query rows of this half
                    float* colh = col + static_cast<size_t>(64 * hh) * D;
#pragma unroll
                    for (int c = 0; c < 2; ++c)
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            if (32 * c + e < nv)
                                red_add_f32(colh + static_cast<size_t>(32 * c + e) * D,
                                            __uint_as_float(x[c][e]));
                }
                if (!ok) break;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 13) tmem_dealloc(tmem, 512);
    if (threadIdx.x == 0 && *s_abort && p.dev_status != nullptr)
        atomicCAS(p.dev_status, 0, static_cast<int>(ATTN_ERR_DEVICE_TIMEOUT));
}

template <int D, bool kF16, bool kCausal, bool kDropout, bool kWindow, bool kPacked>
cudaError_t launch_bwd_t(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                         const BwdParams& p, cudaStream_t stream) {
    using C = BwdCfg<D, kF16>;
    auto kern = attn_bwd_kernel<D, kF16, kCausal, kDropout, kWindow, kPacked>;
    static std::atomic<unsigned long long> smem_ready{0};
    const cudaError_t e = enable_smem_per_device(kern, C::SMEM, smem_ready);
    if (e != cudaSuccess) return e;
    const unsigned grid = static_cast<unsigned>(p.nkb) * static_cast<unsigned>(p.B * p.H);
    return launch_overlapped(kern, grid, C::THREADS, C::SMEM, stream, tq, tk, tv, tdo, tdk, tdv, p);
}

template <int D, bool kF16, bool kPacked, bool kWindow>
cudaError_t dispatch_bwd_w(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                           const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                           const BwdParams& p, bool causal, bool dropout, cudaStream_t s) {
    if (causal)
        return dropout ? launch_bwd_t<D, kF16, true, true, kWindow, kPacked>(tq, tk, tv, tdo, tdk, tdv, p, s)
                       : launch_bwd_t<D, kF16, true, false, kWindow, kPacked>(tq, tk, tv, tdo, tdk, tdv, p, s);
    return dropout ? launch_bwd_t<D, kF16, false, true, kWindow, kPacked>(tq, tk, tv, tdo, tdk, tdv, p, s)
                   : launch_bwd_t<D, kF16, false, false, kWindow, kPacked>(tq, tk, tv, tdo, tdk, tdv, p, s);
}

template <int D, bool kF16, bool kPacked>
cudaError_t dispatch_bwd(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                         const CUtensorMap& tdo, const CUtensorMap& tdk, const CUtensorMap& tdv,
                         const BwdParams& p, bool causal, bool dropout, cudaStream_t s) {
    return p.window > 0
               ? dispatch_bwd_w<D, kF16, kPacked, true>(tq, tk, tv, tdo, tdk, tdv, p, causal, dropout, s)
               : dispatch_bwd_w<D, kF16, kPacked, false>(tq, tk, tv, tdo, tdk, tdv, p, causal, dropout, s);
}

}  // namespace
}  // namespace gbattn
