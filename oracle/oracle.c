/*
 * oracle.c — float64 CPU oracle for exact scaled-dot-product attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * What it computes (and where the pages fix it):
 *
 *   * The attention chain written out in full, one head at a time:
 *     matmul -> scale -> mask -> softmax -> dropout -> matmul
 *     (anthology-of-the-sota, practice SOTA-114, "The general form of the
 *     practice above it"; "Why FlashAttention Is a Kernel Story", "The real
 *     bottleneck: memory bandwidth, not FLOPs", the standard-attention IO
 *     listing).  S and P are materialised as N x N float64 arrays.  The fused
 *     method returns exactly this result up to rounding (SOTA-085, "What 'when
 *     hardware supports it' is carrying", Theorem 1; "Why FlashAttention Is a
 *     Kernel Story", "Tiling", final rescale), so the plain definition is the
 *     oracle.
 *
 *   * The backward pass as the derivative of that chain (the pages only say
 *     that the backward recomputes S and P from O and the log-sum-exp: "Why
 *     FlashAttention Is a Kernel Story", "When it falls down", backward-pass
 *     complexity).  The gradient formulas below are the chain rule applied to
 *     the forward definition; they are pinned by finite differences in the
 *     tests.
 *
 *   * A tiled variant that follows the online-softmax recurrence of
 *     "Why FlashAttention Is a Kernel Story", "Tiling" (running max m,
 *     running denominator l, rescaled output), used only to show that the
 *     result does not depend on the tile size.
 *
 *   * Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
 *     easy as 1, 2, 3", SC'11), written from the paper's definition, used for
 *     the dropout keep/drop decision.
 *
 * Readings of points the pages leave open:
 *   - mask: key j of sequence b is valid iff j < key_len[b] and, when causal,
 *     j <= i, and, when window w > 0 (sliding-window attention, named as a
 *     variant in "Why FlashAttention Is a Kernel Story", "When it falls down"),
 *     i - j < w (and j - i < w when not causal).  Invalid scores are -inf
 *     before the softmax.
 *   - a row with no valid key has O = 0, LSE = -inf and zero gradients.
 *   - dropout is inverted dropout on the normalised P: kept entries are
 *     scaled by 1/(1-p); the log-sum-exp and the softmax denominator use the
 *     undropped P.
 *   - dropout bits: Philox4x32-10 with key (lo32(seed), hi32(seed)) and
 *     counter (i, j>>3, h, b); the output's four 32-bit words hold eight
 *     16-bit draws, word (j>>1)&3 holding key j's in its low half when j is
 *     even and in its high half when j is odd.  The draw is compared with
 *     the integer threshold t = min(floor(p * 2^16), 2^16-1); the entry is
 *     dropped iff draw < t.
 *   - LSE is the natural log of the sum over valid keys of exp(scale*q.k).
 *
 * Layout of every tensor argument: contiguous [heads][N][d] (or [heads][N]
 * for LSE), row-major, float64.  Functions return 0 on success and a
 * negative value on a bad argument or an allocation failure.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Philox4x32-10 (Salmon et al., SC'11, section 3.2).                       */
/* Each of the 10 rounds forms the 64-bit products M0*c0 and M1*c2 and maps  */
/* (c0, c1, c2, c3) to (hi(M1*c2) ^ c1 ^ k0, lo(M1*c2),                      */
/*                      hi(M0*c0) ^ c3 ^ k1, lo(M0*c0)),                      */
/* with M0 = 0xD2511F53, M1 = 0xCD9E8D57; between rounds the key (k0, k1) is */
/* bumped by the Weyl constants (0x9E3779B9, 0xBB67AE85).                     */
/* ------------------------------------------------------------------------ */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u
#define PHILOX_W1 0xBB67AE85u

void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    uint32_t c0 = ctr[0], c1 = ctr[1], c2 = ctr[2], c3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    for (int round = 0; round < 10; ++round) {
        uint64_t p0 = (uint64_t)PHILOX_M0 * (uint64_t)c0;
        uint64_t p1 = (uint64_t)PHILOX_M1 * (uint64_t)c2;
        uint32_t hi0 = (uint32_t)(p0 >> 32), lo0 = (uint32_t)p0;
        uint32_t hi1 = (uint32_t)(p1 >> 32), lo1 = (uint32_t)p1;
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
        if (round < 9) { k0 += PHILOX_W0; k1 += PHILOX_W1; }
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* Integer drop threshold on a 16-bit draw: floor(p * 2^16), clamped to
 * 2^16 - 1. */
uint32_t oracle_dropout_threshold(double p) {
    if (!(p > 0.0)) return 0u;
    double t = floor(p * 65536.0);
    if (t >= 65535.0) return 0xFFFFu;
    return (uint32_t)t;
}

/* 1 if score (i, j) of head (b, h) is kept, 0 if dropped. */
int oracle_dropout_keep(uint64_t seed, int b, int h, int i, int j, uint32_t threshold) {
    uint32_t ctr[4] = {(uint32_t)i, (uint32_t)j >> 3, (uint32_t)h, (uint32_t)b};
    uint32_t key[2] = {(uint32_t)(seed & 0xFFFFFFFFu), (uint32_t)(seed >> 32)};
    uint32_t r[4];
    oracle_philox4x32_10(ctr, key, r);
    uint32_t word = r[(j >> 1) & 3];
    uint32_t draw = (j & 1) ? (word >> 16) : (word & 0xFFFFu);
    return draw < threshold ? 0 : 1;
}

/* Keep mask Z[i][j] (0/1 bytes) of one head, rows x cols. */
void oracle_dropout_mask(uint64_t seed, int b, int h, int rows, int cols, double p, uint8_t* Z) {
    uint32_t t = oracle_dropout_threshold(p);
    for (int i = 0; i < rows; ++i)
        for (int j = 0; j < cols; ++j)
            Z[(size_t)i * cols + j] = (uint8_t)oracle_dropout_keep(seed, b, h, i, j, t);
}

/* ------------------------------------------------------------------------ */
/* Shared pieces of the materialised chain                                   */
/* ------------------------------------------------------------------------ */
static int valid_pair(int i, int j, int causal, int window, int key_len) {
    if (j >= key_len) return 0;
    if (causal && j > i) return 0;
    if (window > 0) {   /* local attention: keys within window - 1 of the query */
        if (i - j >= window) return 0;
        if (!causal && j - i >= window) return 0;
    }
    return 1;
}

static int check_args(int N, int d, double p, int key_len) {
    if (N < 1 || d < 1) return -1;
    if (!(p >= 0.0 && p < 1.0)) return -1;
    if (key_len < 0 || key_len > N) return -1;
    return 0;
}

/* S (scaled, masked to -inf), then P = softmax(S) row-wise, LSE per row.
 * Rows with no valid key get P = 0 and LSE = -inf. */
static void scores_and_probs(const double* q, const double* k, int N, int d, double scale,
                             int causal, int window, int key_len, double* P, double* lse) {
    for (int i = 0; i < N; ++i) {
        double* Pi = P + (size_t)i * N;
        double m = -INFINITY;
        for (int j = 0; j < N; ++j) {
            double s = -INFINITY;
            if (valid_pair(i, j, causal, window, key_len)) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += q[(size_t)i * d + c] * k[(size_t)j * d + c];
                s = scale * acc;
            }
            Pi[j] = s;
            if (s > m) m = s;
        }
        if (m == -INFINITY) {
            for (int j = 0; j < N; ++j) Pi[j] = 0.0;
            lse[i] = -INFINITY;
            continue;
        }
        double l = 0.0;
        for (int j = 0; j < N; ++j) {
            double e = (Pi[j] == -INFINITY) ? 0.0 : exp(Pi[j] - m);
            Pi[j] = e;
            l += e;
        }
        for (int j = 0; j < N; ++j) Pi[j] /= l;
        lse[i] = m + log(l);
    }
}

/* Dropout factor Z_ij / (1 - p) for every (i, j) of one head. */
static void dropout_factors(int N, double p, uint64_t seed, int b, int h, double* F) {
    if (p == 0.0) {
        for (size_t x = 0; x < (size_t)N * N; ++x) F[x] = 1.0;
        return;
    }
    uint32_t t = oracle_dropout_threshold(p);
    double inv = 1.0 / (1.0 - p);
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j)
            F[(size_t)i * N + j] = oracle_dropout_keep(seed, b, h, i, j, t) ? inv : 0.0;
}

/* ------------------------------------------------------------------------ */
/* One head, materialised                                                    */
/* ------------------------------------------------------------------------ */
int oracle_head_fwd(const double* q, const double* k, const double* v, double* o, double* lse,
                    int N, int d, double scale, int causal, int window, int key_len, double p,
                    uint64_t seed, int b, int h) {
    if (check_args(N, d, p, key_len)) return -1;
    double* P = (double*)malloc(sizeof(double) * (size_t)N * N);
    double* F = (double*)malloc(sizeof(double) * (size_t)N * N);
    if (!P || !F) { free(P); free(F); return -2; }
    scores_and_probs(q, k, N, d, scale, causal, window, key_len, P, lse);
    dropout_factors(N, p, seed, b, h, F);
    /* O_i = sum_j P_ij F_ij V_j, accumulated key by key (row-major access). */
    for (size_t x = 0; x < (size_t)N * d; ++x) o[x] = 0.0;
    for (int i = 0; i < N; ++i) {
        for (int j = 0; j < N; ++j) {
            double w = P[(size_t)i * N + j] * F[(size_t)i * N + j];
            if (w == 0.0) continue;
            for (int c = 0; c < d; ++c) o[(size_t)i * d + c] += w * v[(size_t)j * d + c];
        }
    }
    free(P); free(F);
    return 0;
}

/*
 * Backward of one head.  With Pd = P * F (F = Z/(1-p)) and O = Pd V:
 *   dV_j  = sum_i Pd_ij dO_i
 *   dP_ij = (dO_i . V_j) F_ij                  gradient w.r.t. P
 *   D_i   = sum_j P_ij dP_ij                   (equals dO_i . O_i)
 *   dS_ij = P_ij (dP_ij - D_i)                 softmax Jacobian
 *   dQ_i  = scale sum_j dS_ij K_j
 *   dK_j  = scale sum_i dS_ij Q_i
 * D is also returned (length N) when the pointer is not NULL.
 */
int oracle_head_bwd(const double* q, const double* k, const double* v, const double* dout,
                    double* dq, double* dk, double* dv, double* D_out,
                    int N, int d, double scale, int causal, int window, int key_len, double p,
                    uint64_t seed, int b, int h) {
    if (check_args(N, d, p, key_len)) return -1;
    double* P = (double*)malloc(sizeof(double) * (size_t)N * N);
    double* F = (double*)malloc(sizeof(double) * (size_t)N * N);
    double* dS = (double*)malloc(sizeof(double) * (size_t)N * N);
    double* lse = (double*)malloc(sizeof(double) * (size_t)N);
    if (!P || !F || !dS || !lse) { free(P); free(F); free(dS); free(lse); return -2; }
    scores_and_probs(q, k, N, d, scale, causal, window, key_len, P, lse);
    dropout_factors(N, p, seed, b, h, F);

    /* dV_j = sum_i P_ij F_ij dO_i, accumulated query by query */
    for (size_t x = 0; x < (size_t)N * d; ++x) dv[x] = 0.0;
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j) {
            double w = P[(size_t)i * N + j] * F[(size_t)i * N + j];
            if (w == 0.0) continue;
            for (int c = 0; c < d; ++c) dv[(size_t)j * d + c] += w * dout[(size_t)i * d + c];
        }
    /* dP, D, dS */
    for (int i = 0; i < N; ++i) {
        double Di = 0.0;
        for (int j = 0; j < N; ++j) {
            double dp = 0.0;
            if (P[(size_t)i * N + j] != 0.0) { /* dP_ij only enters through P_ij dP_ij */
                for (int c = 0; c < d; ++c) dp += dout[(size_t)i * d + c] * v[(size_t)j * d + c];
                dp *= F[(size_t)i * N + j];
            }
            dS[(size_t)i * N + j] = dp; /* holds dP for now */
            Di += P[(size_t)i * N + j] * dp;
        }
        if (D_out) D_out[i] = Di;
        for (int j = 0; j < N; ++j)
            dS[(size_t)i * N + j] = P[(size_t)i * N + j] * (dS[(size_t)i * N + j] - Di);
    }
    /* dQ */
    for (int i = 0; i < N; ++i)
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int j = 0; j < N; ++j) acc += dS[(size_t)i * N + j] * k[(size_t)j * d + c];
            dq[(size_t)i * d + c] = scale * acc;
        }
    /* dK_j = scale sum_i dS_ij Q_i, accumulated query by query */
    for (size_t x = 0; x < (size_t)N * d; ++x) dk[x] = 0.0;
    for (int i = 0; i < N; ++i)
        for (int j = 0; j < N; ++j) {
            double w = dS[(size_t)i * N + j];
            if (w == 0.0) continue;
            for (int c = 0; c < d; ++c) dk[(size_t)j * d + c] += w * q[(size_t)i * d + c];
        }
    for (size_t x = 0; x < (size_t)N * d; ++x) dk[x] *= scale;
    free(P); free(F); free(dS); free(lse);
    return 0;
}

/*
 * Selected rows of one head's forward, without an N x N array: each row is
 * the same definition evaluated on its own (O(N d) memory).  Used to check
 * outputs of workloads too large to materialise.
 */
int oracle_head_fwd_rows(const double* q, const double* k, const double* v,
                         const int32_t* rows, int nrows, double* o_rows, double* lse_rows,
                         int N, int d, double scale, int causal, int window, int key_len, double p,
                         uint64_t seed, int b, int h) {
    if (check_args(N, d, p, key_len)) return -1;
    double* s = (double*)malloc(sizeof(double) * (size_t)N);
    if (!s) return -2;
    uint32_t t = oracle_dropout_threshold(p);
    double inv = 1.0 / (1.0 - p);
    for (int r = 0; r < nrows; ++r) {
        int i = rows[r];
        if (i < 0 || i >= N) { free(s); return -1; }
        double m = -INFINITY;
        for (int j = 0; j < N; ++j) {
            double sc = -INFINITY;
            if (valid_pair(i, j, causal, window, key_len)) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += q[(size_t)i * d + c] * k[(size_t)j * d + c];
                sc = scale * acc;
            }
            s[j] = sc;
            if (sc > m) m = sc;
        }
        double* orow = o_rows + (size_t)r * d;
        for (int c = 0; c < d; ++c) orow[c] = 0.0;
        if (m == -INFINITY) { lse_rows[r] = -INFINITY; continue; }
        double l = 0.0;
        for (int j = 0; j < N; ++j) {
            s[j] = (s[j] == -INFINITY) ? 0.0 : exp(s[j] - m);
            l += s[j];
        }
        for (int j = 0; j < N; ++j) {
            if (s[j] == 0.0) continue;
            double f = 1.0;
            if (p > 0.0) f = oracle_dropout_keep(seed, b, h, i, j, t) ? inv : 0.0;
            double w = s[j] / l * f;
            if (w == 0.0) continue;
            for (int c = 0; c < d; ++c) orow[c] += w * v[(size_t)j * d + c];
        }
        lse_rows[r] = m + log(l);
    }
    free(s);
    return 0;
}

/*
 * Forward and backward of the query rows [row0, row0 + nrows) of one head,
 * row by row, without an Nq x Nk array: O, LSE and dQ of those rows, and the
 * rows' contributions to dK and dV added into dk_part and dv_part ([Nk][d],
 * zeroed by the caller).  The same definitions as oracle_head_fwd and
 * oracle_head_bwd, restricted to a slice of the rows; summed over a partition
 * of all rows, the contributions give the head's dK and dV.
 *
 * Nq query rows and Nk keys may differ (cross-attention).  Queries are then
 * aligned with the last keys: query i plays the part of position i + Nk - Nq
 * in the causal and window tests, so the last query sees every key when
 * causal (the usual convention when a shorter query block continues a longer
 * key sequence).  With Nq == Nk this is the square definition.
 */
int oracle_head_rows_fwd_bwd(const double* q, const double* k, const double* v,
                             const double* dout, int row0, int nrows, double* o_rows,
                             double* lse_rows, double* dq_rows, double* dk_part, double* dv_part,
                             int Nq, int Nk, int d, double scale, int causal, int window,
                             int key_len, double p, uint64_t seed, int b, int h) {
    if (check_args(Nk, d, p, key_len) || Nq < 1 || row0 < 0 || nrows < 0 || row0 + nrows > Nq)
        return -1;
    const int N = Nk;          /* keys */
    const int off = Nk - Nq;   /* query i sits at position i + off */
    double* P = (double*)malloc(sizeof(double) * (size_t)N);
    double* F = (double*)malloc(sizeof(double) * (size_t)N);
    if (!P || !F) { free(P); free(F); return -2; }
    uint32_t t = oracle_dropout_threshold(p);
    double inv = 1.0 / (1.0 - p);
    for (int r = 0; r < nrows; ++r) {
        const int i = row0 + r;
        const double* qi = q + (size_t)i * d;
        const double* gi = dout + (size_t)i * d;
        double* oi = o_rows + (size_t)r * d;
        double* dqi = dq_rows + (size_t)r * d;
        for (int c = 0; c < d; ++c) { oi[c] = 0.0; dqi[c] = 0.0; }
        double m = -INFINITY;
        for (int j = 0; j < N; ++j) {
            double sc = -INFINITY;
            if (valid_pair(i + off, j, causal, window, key_len)) {
                double acc = 0.0;
                for (int c = 0; c < d; ++c) acc += qi[c] * k[(size_t)j * d + c];
                sc = scale * acc;
            }
            P[j] = sc;
            if (sc > m) m = sc;
        }
        if (m == -INFINITY) { lse_rows[r] = -INFINITY; continue; }
        double l = 0.0;
        for (int j = 0; j < N; ++j) {
            P[j] = (P[j] == -INFINITY) ? 0.0 : exp(P[j] - m);
            l += P[j];
        }
        for (int j = 0; j < N; ++j) {
            P[j] /= l;
            F[j] = 1.0;
            if (p > 0.0) F[j] = oracle_dropout_keep(seed, b, h, i, j, t) ? inv : 0.0;
        }
        lse_rows[r] = m + log(l);
        for (int j = 0; j < N; ++j) {          /* O_i */
            double w = P[j] * F[j];
            if (w == 0.0) continue;
            for (int c = 0; c < d; ++c) oi[c] += w * v[(size_t)j * d + c];
        }
        double Di = 0.0;                        /* D_i = dO_i . O_i */
        for (int c = 0; c < d; ++c) Di += gi[c] * oi[c];
        for (int j = 0; j < N; ++j) {
            if (P[j] == 0.0) continue;
            double dp = 0.0;
            for (int c = 0; c < d; ++c) dp += gi[c] * v[(size_t)j * d + c];
            dp *= F[j];
            const double ds = P[j] * (dp - Di);
            const double w = P[j] * F[j];
            for (int c = 0; c < d; ++c) {
                dqi[c] += ds * k[(size_t)j * d + c];
                dk_part[(size_t)j * d + c] += scale * ds * qi[c];
                dv_part[(size_t)j * d + c] += w * gi[c];
            }
        }
        for (int c = 0; c < d; ++c) dqi[c] *= scale;
    }
    free(P); free(F);
    return 0;
}

/* Rows [row0, row0 + nrows) of nh heads (OpenMP over heads); Q, dO are
 * [nh][Nq][d], K, V [nh][Nk][d], the *_rows arrays [nh][nrows](...) and the
 * partial dK, dV arrays [nh][Nk][d] (zeroed here). */
int oracle_heads_rows_fwd_bwd(const double* Q, const double* K, const double* V,
                              const double* dO, int nh, const int32_t* b_idx,
                              const int32_t* h_idx, const int32_t* key_len, int Nq, int Nk, int d,
                              double scale, int causal, int window, double p, uint64_t seed, int row0,
                              int nrows, double* O_rows, double* LSE_rows, double* dQ_rows,
                              double* dK_part, double* dV_part, int nthreads);

/*
 * Tiled forward of one head following the online-softmax recurrence of
 * "Why FlashAttention Is a Kernel Story", "Tiling": rows are taken Br at a
 * time and keys Bc at a time; for each key tile the running max m, the
 * running denominator l and the unnormalised output are updated as
 *   m_new = max(m_old, rowmax(s)),
 *   l_new = exp(m_old - m_new) l_old + rowsum(exp(s - m_new)),
 *   O_new = exp(m_old - m_new) O_old + exp(s - m_new) V,
 * and after the last tile O = O / l.  Dropout multiplies the exp(s - m_new)
 * terms that enter O (not l) by Z/(1-p).
 */
int oracle_head_fwd_tiled(const double* q, const double* k, const double* v, double* o,
                          double* lse, int N, int d, double scale, int causal, int window, int key_len,
                          double p, uint64_t seed, int b, int h, int Br, int Bc) {
    if (check_args(N, d, p, key_len) || Br < 1 || Bc < 1) return -1;
    double* m = (double*)malloc(sizeof(double) * (size_t)Br);
    double* l = (double*)malloc(sizeof(double) * (size_t)Br);
    double* s = (double*)malloc(sizeof(double) * (size_t)Br * Bc);
    double* acc = (double*)malloc(sizeof(double) * (size_t)Br * d);
    if (!m || !l || !s || !acc) { free(m); free(l); free(s); free(acc); return -2; }
    uint32_t t = oracle_dropout_threshold(p);
    double inv = 1.0 / (1.0 - p);
    for (int i0 = 0; i0 < N; i0 += Br) {
        int br = (N - i0 < Br) ? N - i0 : Br;
        for (int r = 0; r < br; ++r) { m[r] = -INFINITY; l[r] = 0.0; }
        for (size_t x = 0; x < (size_t)br * d; ++x) acc[x] = 0.0;
        for (int j0 = 0; j0 < N; j0 += Bc) {
            int bc = (N - j0 < Bc) ? N - j0 : Bc;
            for (int r = 0; r < br; ++r) {
                int i = i0 + r;
                double rowmax = -INFINITY;
                for (int cc = 0; cc < bc; ++cc) {
                    int j = j0 + cc;
                    double sc = -INFINITY;
                    if (valid_pair(i, j, causal, window, key_len)) {
                        double a = 0.0;
                        for (int c = 0; c < d; ++c) a += q[(size_t)i * d + c] * k[(size_t)j * d + c];
                        sc = scale * a;
                    }
                    s[(size_t)r * Bc + cc] = sc;
                    if (sc > rowmax) rowmax = sc;
                }
                double m_new = (rowmax > m[r]) ? rowmax : m[r];
                if (m_new == -INFINITY) continue; /* nothing valid yet in this row */
                double alpha = (m[r] == -INFINITY) ? 0.0 : exp(m[r] - m_new);
                double rowsum = 0.0;
                for (int c = 0; c < d; ++c) acc[(size_t)r * d + c] *= alpha;
                for (int cc = 0; cc < bc; ++cc) {
                    double sc = s[(size_t)r * Bc + cc];
                    if (sc == -INFINITY) continue;
                    double e = exp(sc - m_new);
                    rowsum += e;
                    double f = 1.0;
                    if (p > 0.0) f = oracle_dropout_keep(seed, b, h, i, j0 + cc, t) ? inv : 0.0;
                    if (f == 0.0) continue;
                    for (int c = 0; c < d; ++c)
                        acc[(size_t)r * d + c] += e * f * v[(size_t)(j0 + cc) * d + c];
                }
                l[r] = alpha * l[r] + rowsum;
                m[r] = m_new;
            }
        }
        for (int r = 0; r < br; ++r) {
            int i = i0 + r;
            if (l[r] == 0.0) {
                for (int c = 0; c < d; ++c) o[(size_t)i * d + c] = 0.0;
                lse[i] = -INFINITY;
            } else {
                for (int c = 0; c < d; ++c) o[(size_t)i * d + c] = acc[(size_t)r * d + c] / l[r];
                lse[i] = m[r] + log(l[r]);
            }
        }
    }
    free(m); free(l); free(s); free(acc);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Many heads at once (OpenMP over heads).                                   */
/* Arrays hold nh heads back to back; head x has batch index b_idx[x], head  */
/* index h_idx[x] (both only feed the dropout counter) and key length        */
/* key_len[x].  nthreads <= 0 lets OpenMP choose.                            */
/* ------------------------------------------------------------------------ */
static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_heads_fwd(const double* Q, const double* K, const double* V, double* O, double* LSE,
                     int nh, const int32_t* b_idx, const int32_t* h_idx, const int32_t* key_len,
                     int N, int d, double scale, int causal, int window, double p, uint64_t seed,
                     int nthreads) {
    if (nh < 0) return -1;
    set_threads(nthreads);
    int err = 0;
    size_t hd = (size_t)N * d;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int x = 0; x < nh; ++x) {
        int r = oracle_head_fwd(Q + x * hd, K + x * hd, V + x * hd, O + x * hd, LSE + (size_t)x * N,
                                N, d, scale, causal, window, key_len[x], p, seed, b_idx[x], h_idx[x]);
        if (r) err |= 1;
    }
    return err ? -1 : 0;
}

int oracle_heads_bwd(const double* Q, const double* K, const double* V, const double* dO,
                     double* dQ, double* dK, double* dV, double* D,
                     int nh, const int32_t* b_idx, const int32_t* h_idx, const int32_t* key_len,
                     int N, int d, double scale, int causal, int window, double p, uint64_t seed,
                     int nthreads) {
    if (nh < 0) return -1;
    set_threads(nthreads);
    int err = 0;
    size_t hd = (size_t)N * d;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int x = 0; x < nh; ++x) {
        int r = oracle_head_bwd(Q + x * hd, K + x * hd, V + x * hd, dO + x * hd,
                                dQ + x * hd, dK + x * hd, dV + x * hd,
                                D ? D + (size_t)x * N : NULL,
                                N, d, scale, causal, window, key_len[x], p, seed, b_idx[x], h_idx[x]);
        if (r) err |= 1;
    }
    return err ? -1 : 0;
}

int oracle_heads_rows_fwd_bwd(const double* Q, const double* K, const double* V,
                              const double* dO, int nh, const int32_t* b_idx,
                              const int32_t* h_idx, const int32_t* key_len, int Nq, int Nk, int d,
                              double scale, int causal, int window, double p, uint64_t seed, int row0,
                              int nrows, double* O_rows, double* LSE_rows, double* dQ_rows,
                              double* dK_part, double* dV_part, int nthreads) {
    if (nh < 0) return -1;
    set_threads(nthreads);
    int err = 0;
    size_t qd = (size_t)Nq * d, kd = (size_t)Nk * d, rd = (size_t)nrows * d;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int x = 0; x < nh; ++x) {
        for (size_t y = 0; y < kd; ++y) { dK_part[x * kd + y] = 0.0; dV_part[x * kd + y] = 0.0; }
        int r = oracle_head_rows_fwd_bwd(Q + x * qd, K + x * kd, V + x * kd, dO + x * qd, row0,
                                         nrows, O_rows + x * rd, LSE_rows + (size_t)x * nrows,
                                         dQ_rows + x * rd, dK_part + x * kd, dV_part + x * kd, Nq,
                                         Nk, d, scale, causal, window, key_len[x], p, seed, b_idx[x],
                                         h_idx[x]);
        if (r) err |= 1;
    }
    return err ? -1 : 0;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
