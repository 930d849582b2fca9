"""Pins of the float64 oracle against facts that do not come from the oracle.

Each ``pin_*`` function takes a loaded oracle library (the normal build or a
deliberately broken build from the mutation test) and returns the largest
error it saw; the test asserts it is below the pin's bound.  The facts come
from the mathematics of the chain the pages describe (anthology-of-the-sota,
SOTA-114, "The general form of the practice above it"; "Why FlashAttention Is
a Kernel Story", "Tiling"), from library routines that compute the same thing
another way (torch float64 softmax and autograd, Triton's Philox), and from
brute force (central finite differences).
"""
from __future__ import annotations

import math
import os
import subprocess
import sys
import json

import numpy as np
import torch

import oracle

RNG = np.random.default_rng(12345)


def _rand(*shape, scale=1.0, seed=None):
    r = np.random.default_rng(seed) if seed is not None else RNG
    return r.standard_normal(shape) * scale


def _valid(N, causal, key_len, window=0):
    i = np.arange(N)[:, None]
    j = np.arange(N)[None, :]
    v = np.broadcast_to(j < key_len, (N, N))
    if causal:
        v = v & (j <= i)
    if window > 0:   # sliding window: keys within window - 1 of the query
        v = v & (i - j < window)
        if not causal:
            v = v & (j - i < window)
    return np.array(v)


# ---------------------------------------------------------------------------
# closed forms and special cases
# ---------------------------------------------------------------------------
def pin_zero_query(L) -> float:
    """Q = 0: every valid score is 0, so O_i is the mean of the valid V_j and
    LSE_i = ln(#valid keys).  With dropout, O_i = sum_j Z_ij V_j / ((1-p) #valid)."""
    worst = 0.0
    for causal in (False, True):
        for key_len in (11, 7, 1, 0):
            for p in (0.0, 0.3):
                N, d = 11, 5
                q = np.zeros((1, 1, N, d))
                k = _rand(1, 1, N, d, seed=1)
                v = _rand(1, 1, N, d, seed=2)
                O, LSE = oracle.attn_fwd(q, k, v, 0.7, causal, [key_len], p, 99, _lib=L)
                valid = _valid(N, causal, key_len)
                Z = oracle.dropout_mask(99, 0, 0, N, N, p, _lib=L) if p > 0 else np.ones((N, N))
                for i in range(N):
                    cnt = valid[i].sum()
                    if cnt == 0:
                        exp_o = np.zeros(d)
                        worst = max(worst, 0.0 if LSE[0, 0, i] == -math.inf else 1.0)
                    else:
                        w = valid[i] * Z[i] / ((1 - p) * cnt)
                        exp_o = w @ v[0, 0]
                        worst = max(worst, abs(LSE[0, 0, i] - math.log(cnt)))
                    worst = max(worst, np.abs(O[0, 0, i] - exp_o).max())
    return worst


def pin_causal_row0(L) -> float:
    """Causal row 0 sees only key 0: O_0 = V_0 and LSE_0 = scale q_0 . k_0."""
    worst = 0.0
    for N, d in ((1, 3), (9, 4), (33, 16)):
        q, k, v = _rand(2, 3, N, d), _rand(2, 3, N, d), _rand(2, 3, N, d)
        O, LSE = oracle.attn_fwd(q, k, v, 0.31, True, None, 0.0, 0, _lib=L)
        worst = max(worst, np.abs(O[:, :, 0] - v[:, :, 0]).max())
        lse0 = 0.31 * np.einsum("bhd,bhd->bh", q[:, :, 0], k[:, :, 0])
        worst = max(worst, np.abs(LSE[:, :, 0] - lse0).max())
    return worst


def pin_single_key(L) -> float:
    """N = 1 (or key_len = 1): the only key gets weight 1, so O = V_0 everywhere."""
    q, k, v = _rand(2, 2, 1, 8), _rand(2, 2, 1, 8), _rand(2, 2, 1, 8)
    O, _ = oracle.attn_fwd(q, k, v, 0.5, False, None, 0.0, 0, _lib=L)
    worst = np.abs(O - v).max()
    q, k, v = _rand(1, 2, 6, 8), _rand(1, 2, 6, 8), _rand(1, 2, 6, 8)
    O, _ = oracle.attn_fwd(q, k, v, 0.5, False, [1], 0.0, 0, _lib=L)
    worst = max(worst, np.abs(O - v[:, :, :1]).max())
    return float(worst)


def pin_rows_are_distributions(L) -> float:
    """With V = identity (d = N), O is P itself: rows are non-negative, sum to
    1, vanish exactly on masked pairs, and follow softmax's ratio law
    P_ij / P_ik = exp(scale (q_i.k_j - q_i.k_k))."""
    worst = 0.0
    N = 12
    for causal in (False, True):
        for key_len in (12, 5):
            q, k = _rand(1, 1, N, N), _rand(1, 1, N, N)
            v = np.eye(N)[None, None]
            O, _ = oracle.attn_fwd(q, k, v, 0.9, causal, [key_len], 0.0, 0, _lib=L)
            P = O[0, 0]
            valid = _valid(N, causal, key_len)
            worst = max(worst, np.abs(P.sum(1) - 1).max())
            worst = max(worst, np.abs(P[~valid]).max() if (~valid).any() else 0.0)
            worst = max(worst, -min(0.0, P.min()))
            s = 0.9 * (q[0, 0] @ k[0, 0].T)
            for i in range(N):
                js = np.nonzero(valid[i])[0]
                if len(js) >= 2:
                    r = P[i, js[1:]] / P[i, js[0]]
                    worst = max(worst, np.abs(np.log(r) - (s[i, js[1:]] - s[i, js[0]])).max())
    return worst


def pin_two_keys_sigmoid(L) -> float:
    """Two keys: the weight of key 0 is the logistic function
    1 / (1 + exp(scale q (k_1 - k_0))) and LSE = scale q k_0 + ln(1 + exp(...))."""
    worst = 0.0
    for qv, k0, k1 in ((0.3, -1.2, 2.0), (-2.5, 0.7, 0.1), (4.0, 3.0, -3.0)):
        q = np.array([[[[qv], [qv]]]])
        k = np.array([[[[k0], [k1]]]])
        v = np.array([[[[1.5], [-0.25]]]])
        sc = 0.8
        O, LSE = oracle.attn_fwd(q, k, v, sc, False, None, 0.0, 0, _lib=L)
        t = sc * qv * (k1 - k0)
        w0 = 1.0 / (1.0 + math.exp(t))
        worst = max(worst, abs(O[0, 0, 0, 0] - (w0 * 1.5 + (1 - w0) * -0.25)))
        worst = max(worst, abs(LSE[0, 0, 0] - (sc * qv * k0 + math.log1p(math.exp(t)))))
    return worst


def pin_key_shift_invariance(L) -> float:
    """Adding one vector c to every key shifts row i's scores by scale q_i . c,
    which the softmax removes: O is unchanged and LSE moves by scale q_i . c."""
    B, H, N, d = 1, 2, 10, 4
    q, k, v = _rand(B, H, N, d), _rand(B, H, N, d), _rand(B, H, N, d)
    c = _rand(d)
    O1, L1 = oracle.attn_fwd(q, k, v, 0.6, True, [8], 0.2, 5, _lib=L)
    O2, L2 = oracle.attn_fwd(q, k + c, v, 0.6, True, [8], 0.2, 5, _lib=L)
    shift = 0.6 * np.einsum("bhnd,d->bhn", q, c)
    fin = np.isfinite(L1)
    return float(max(np.abs(O1 - O2).max(), np.abs((L2 - L1 - shift)[fin]).max()))


# ---------------------------------------------------------------------------
# library routines computing the same chain another way
# ---------------------------------------------------------------------------
def _torch_chain(q, k, v, scale, causal, key_len, p, Z, window=0):
    """softmax(scale Q K^T + mask) * Z/(1-p) @ V with torch float64 library ops."""
    s = scale * torch.matmul(q, k.transpose(-1, -2))
    N = q.shape[-2]
    valid = torch.as_tensor(_valid(N, causal, key_len, window))
    s = s.masked_fill(~valid, float("-inf"))
    lse = torch.logsumexp(s, dim=-1)
    P = torch.softmax(s, dim=-1)
    P = torch.nan_to_num(P, nan=0.0)
    if p > 0:
        P = P * torch.as_tensor(Z, dtype=torch.float64) / (1 - p)
    return P @ v, lse


def pin_torch_autograd(L) -> float:
    """Forward against torch float64 softmax/logsumexp/matmul; backward against
    torch autograd of that chain (same dropout mask Z applied as a constant)."""
    worst = 0.0
    for N, d, causal, key_len, p in ((7, 4, False, 7, 0.0), (13, 8, True, 13, 0.0),
                                    (16, 8, False, 9, 0.25), (19, 4, True, 15, 0.4)):
        B, H = 1, 2
        q, k, v, do = (_rand(B, H, N, d) for _ in range(4))
        sc = 1 / math.sqrt(d)
        O, LSE = oracle.attn_fwd(q, k, v, sc, causal, [key_len], p, 7, _lib=L)
        dQ, dK, dV, _ = oracle.attn_bwd(q, k, v, do, sc, causal, [key_len], p, 7, _lib=L)
        for h in range(H):
            Z = oracle.dropout_mask(7, 0, h, N, N, p, _lib=L) if p > 0 else None
            tq, tk, tv = (torch.tensor(a[0, h], requires_grad=True) for a in (q, k, v))
            to, tl = _torch_chain(tq, tk, tv, sc, causal, key_len, p, Z)
            (to * torch.tensor(do[0, h])).sum().backward()
            worst = max(worst, np.abs(O[0, h] - to.detach().numpy()).max())
            worst = max(worst, np.abs(LSE[0, h] - tl.detach().numpy()).max())
            for g, tg in ((dQ, tq), (dK, tk), (dV, tv)):
                worst = max(worst, np.abs(g[0, h] - tg.grad.numpy()).max())
    return worst


def pin_window_one(L) -> float:
    """Sliding window of width 1: each query sees only its own key, so O_i = V_i
    and LSE_i = scale q_i . k_i, causal or not."""
    worst = 0.0
    for causal in (False, True):
        N, d = 9, 6
        q, k, v = (_rand(1, 1, N, d, seed=s) for s in (21, 22, 23))
        O, LSE = oracle.attn_fwd(q, k, v, 0.8, causal, None, 0.0, 0, window=1, _lib=L)
        worst = max(worst, np.abs(O - v).max())
        worst = max(worst, np.abs(LSE[0, 0] - 0.8 * np.einsum("nd,nd->n", q[0, 0], k[0, 0])).max())
    return worst


def pin_window_torch(L) -> float:
    """Sliding-window masks (causal and two-sided) against torch float64 for the
    forward and torch autograd for the backward, with key padding and dropout;
    a window of at least N gives exactly the unwindowed result."""
    worst = 0.0
    for N, d, causal, key_len, p, w in ((13, 4, True, 13, 0.0, 3), (16, 8, False, 12, 0.0, 4),
                                        (19, 4, True, 15, 0.3, 5), (11, 8, False, 11, 0.2, 2)):
        B, H = 1, 2
        q, k, v, do = (_rand(B, H, N, d) for _ in range(4))
        sc = 1 / math.sqrt(d)
        O, LSE = oracle.attn_fwd(q, k, v, sc, causal, [key_len], p, 7, window=w, _lib=L)
        dQ, dK, dV, _ = oracle.attn_bwd(q, k, v, do, sc, causal, [key_len], p, 7, window=w, _lib=L)
        for h in range(H):
            Z = oracle.dropout_mask(7, 0, h, N, N, p, _lib=L) if p > 0 else None
            tq, tk, tv = (torch.tensor(a[0, h], requires_grad=True) for a in (q, k, v))
            to, tl = _torch_chain(tq, tk, tv, sc, causal, key_len, p, Z, window=w)
            (to * torch.tensor(do[0, h])).sum().backward()
            worst = max(worst, np.abs(O[0, h] - to.detach().numpy()).max())
            fin = np.isfinite(LSE[0, h])
            worst = max(worst, np.abs(LSE[0, h][fin] - tl.detach().numpy()[fin]).max())
            for g, tg in ((dQ, tq), (dK, tk), (dV, tv)):
                worst = max(worst, np.abs(g[0, h] - tg.grad.numpy()).max())
        O2, LSE2 = oracle.attn_fwd(q, k, v, sc, causal, [key_len], p, 7, window=N, _lib=L)
        O3, LSE3 = oracle.attn_fwd(q, k, v, sc, causal, [key_len], p, 7, _lib=L)
        worst = max(worst, np.abs(O2 - O3).max(), np.abs(np.nan_to_num(LSE2 - LSE3)).max())
    return worst


def pin_cross_attention_torch(L) -> float:
    """Nq != Nk (queries aligned with the last keys: query i stands at key
    position i + Nk - Nq) against torch float64 with the rectangular mask
    written out, forward and autograd backward, with padding, dropout and a
    window; more queries than keys leaves the first Nq - Nk rows empty under
    the causal mask (O = 0, LSE = -inf, zero gradients)."""
    worst = 0.0
    for Nq, Nk, d, causal, key_len, p, w in ((5, 13, 4, True, 13, 0.0, 0), (13, 5, 8, True, 5, 0.0, 0),
                                              (7, 11, 4, False, 9, 0.25, 0), (9, 16, 8, True, 14, 0.0, 4),
                                              (1, 10, 4, True, 10, 0.0, 0)):
        B, H = 1, 2
        q, do = _rand(B, H, Nq, d), _rand(B, H, Nq, d)
        k, v = _rand(B, H, Nk, d), _rand(B, H, Nk, d)
        sc = 1 / math.sqrt(d)
        O, LSE, dQ, dK, dV = oracle.attn_fwd_bwd_qk(q, k, v, do, sc, causal, [key_len], p, 7,
                                                    window=w, _lib=L)
        i = np.arange(Nq)[:, None] + (Nk - Nq)
        j = np.arange(Nk)[None, :]
        valid = np.broadcast_to(j < key_len, (Nq, Nk)).copy()
        if causal:
            valid &= j <= i
        if w > 0:
            valid &= i - j < w
            if not causal:
                valid &= j - i < w
        for h in range(H):
            tq, tk, tv = (torch.tensor(a[0, h], requires_grad=True) for a in (q, k, v))
            s_ = (sc * tq @ tk.T).masked_fill(~torch.as_tensor(valid), float("-inf"))
            tl = torch.logsumexp(s_, dim=-1)
            P = torch.nan_to_num(torch.softmax(s_, dim=-1), nan=0.0)
            if p > 0:
                Z = oracle.dropout_mask(7, 0, h, Nq, Nk, p, _lib=L)
                P = P * torch.as_tensor(Z, dtype=torch.float64) / (1 - p)
            to = P @ tv
            (to * torch.tensor(do[0, h])).sum().backward()
            worst = max(worst, np.abs(O[0, h] - to.detach().numpy()).max())
            fin = np.isfinite(LSE[0, h])
            worst = max(worst, np.abs(LSE[0, h][fin] - tl.detach().numpy()[fin]).max())
            worst = max(worst, float((~fin != ~np.isfinite(tl.detach().numpy())).any()))
            for g, tg in ((dQ, tq), (dK, tk), (dV, tv)):
                worst = max(worst, np.abs(g[0, h] - tg.grad.numpy()).max())
    return worst


def pin_philox_vs_triton(L) -> float:
    """The oracle's Philox4x32-10 against Triton's implementation of the same
    generator (run by Triton's CPU interpreter in a child process).  Returns
    the number of mismatching words (NaN when Triton is unavailable)."""
    script = os.path.join(os.path.dirname(os.path.abspath(__file__)), "philox_triton_ref.py")
    rng = np.random.default_rng(7)
    ctrs = rng.integers(0, 2**32, size=(64, 4), dtype=np.uint64)
    ctrs[0] = 0
    ctrs[1] = 2**32 - 1
    ctrs[2] = [5, 1, 3, 2]
    seeds = [0, 1, 0x5EED0005, 0xFFFFFFFFFFFFFFFF, 0x123456789ABCDEF0]
    req = {"ctrs": ctrs.tolist(), "seeds": seeds}
    env = dict(os.environ, TRITON_INTERPRET="1")
    try:
        res = subprocess.run([sys.executable, script], input=json.dumps(req), text=True,
                             capture_output=True, env=env, timeout=600)
    except Exception:
        return float("nan")
    if res.returncode != 0:
        return float("nan")
    got = json.loads(res.stdout.strip().splitlines()[-1])
    bad = 0
    for si, seed in enumerate(seeds):
        key = [seed & 0xFFFFFFFF, seed >> 32]
        for ci, c in enumerate(ctrs):
            mine = oracle.philox4x32_10(c, key, _lib=L)
            bad += int(np.sum(mine != np.array(got[si][ci], dtype=np.uint32)))
    return float(bad)


# ---------------------------------------------------------------------------
# brute force and recurrence
# ---------------------------------------------------------------------------
def pin_varlen_equal_lengths(L) -> float:
    """Packed sequences of one common length (queries and keys) give the
    dense [B, H, N, d] result, dropout included (sequence b takes the dropout
    counters of batch entry b)."""
    worst = 0.0
    for B, H, Nq, Nk, d, causal, p, w in ((3, 2, 9, 9, 4, True, 0.3, 0), (2, 3, 6, 11, 8, False, 0.2, 0),
                                            (2, 2, 10, 7, 4, True, 0.0, 3)):
        q, do = _rand(B, H, Nq, d), _rand(B, H, Nq, d)
        k, v = _rand(B, H, Nk, d), _rand(B, H, Nk, d)
        dense = oracle.attn_fwd_bwd_qk(q, k, v, do, 0.4, causal, None, p, 31, window=w, _lib=L)
        pack = lambda x: np.ascontiguousarray(x.transpose(0, 2, 1, 3).reshape(-1, H, d))  # noqa: E731
        cu_q, cu_k = np.arange(B + 1) * Nq, np.arange(B + 1) * Nk
        O, LSE, dQ, dK, dV = oracle.attn_fwd_bwd_varlen(pack(q), pack(k), pack(v), pack(do), cu_q,
                                                        cu_k, 0.4, causal, p, 31, window=w, _lib=L)
        worst = max(worst, np.abs(O - pack(dense[0])).max(), np.abs(dQ - pack(dense[2])).max(),
                    np.abs(dK - pack(dense[3])).max(), np.abs(dV - pack(dense[4])).max())
        lse_dense = dense[1].transpose(1, 0, 2).reshape(H, -1)
        fin = np.isfinite(lse_dense)
        worst = max(worst, float((np.isfinite(LSE) != fin).any()),
                    np.abs(LSE[fin] - lse_dense[fin]).max())
    return worst


def pin_varlen_torch(L) -> float:
    """Packed sequences of different lengths (one without queries, one
    without keys, one with more queries than keys) against torch float64 run
    sequence by sequence with the mask written out, forward and autograd
    backward, with dropout and a window."""
    H, d, sc, seed = 2, 4, 0.5, 77
    lens_q = [5, 0, 7, 3, 4]
    lens_k = [9, 4, 3, 0, 6]
    cu_q, cu_k = np.concatenate([[0], np.cumsum(lens_q)]), np.concatenate([[0], np.cumsum(lens_k)])
    worst = 0.0
    for causal, p, w in ((True, 0.0, 0), (False, 0.25, 0), (True, 0.15, 3)):
        q, do = _rand(1, int(cu_q[-1]), H, d)[0], _rand(1, int(cu_q[-1]), H, d)[0]
        k, v = _rand(1, int(cu_k[-1]), H, d)[0], _rand(1, int(cu_k[-1]), H, d)[0]
        O, LSE, dQ, dK, dV = oracle.attn_fwd_bwd_varlen(q, k, v, do, cu_q, cu_k, sc, causal, p,
                                                        seed, window=w, _lib=L)
        for b in range(len(lens_q)):
            q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
            n, nk = q1 - q0, k1 - k0
            if n == 0:
                continue
            i = np.arange(n)[:, None] + (nk - n)
            j = np.arange(nk)[None, :]
            valid = np.ones((n, nk), dtype=bool)
            if causal:
                valid &= j <= i
            if w > 0:
                valid &= i - j < w
                if not causal:
                    valid &= j - i < w
            for h in range(H):
                tq = torch.tensor(q[q0:q1, h], requires_grad=True)
                tk = torch.tensor(k[k0:k1, h], requires_grad=True)
                tv = torch.tensor(v[k0:k1, h], requires_grad=True)
                s_ = (sc * tq @ tk.T).masked_fill(~torch.as_tensor(valid), float("-inf"))
                tl = torch.logsumexp(s_, dim=-1) if nk > 0 else torch.full((n,), float("-inf"))
                P = torch.nan_to_num(torch.softmax(s_, dim=-1), nan=0.0)
                if p > 0 and nk > 0:
                    Z = oracle.dropout_mask(seed, b, h, n, nk, p, _lib=L)
                    P = P * torch.as_tensor(Z, dtype=torch.float64) / (1 - p)
                to = P @ tv
                (to * torch.tensor(do[q0:q1, h])).sum().backward()
                worst = max(worst, np.abs(O[q0:q1, h] - to.detach().numpy()).max())
                tl = tl.detach().numpy()
                fin = np.isfinite(tl)
                worst = max(worst, float((np.isfinite(LSE[h, q0:q1]) != fin).any()))
                if fin.any():
                    worst = max(worst, np.abs(LSE[h, q0:q1][fin] - tl[fin]).max())
                worst = max(worst, np.abs(dQ[q0:q1, h] - tq.grad.numpy()).max())
                if nk > 0:
                    worst = max(worst, np.abs(dK[k0:k1, h] - tk.grad.numpy()).max(),
                                np.abs(dV[k0:k1, h] - tv.grad.numpy()).max())
        # keys of a sequence without queries get zero gradients
        worst = max(worst, np.abs(dK[cu_k[1]:cu_k[2]]).max(), np.abs(dV[cu_k[1]:cu_k[2]]).max())
    return worst


def pin_finite_differences(L, sizes=((1, 4), (5, 4), (17, 8))) -> float:
    """Central differences (h = 1e-6) of f = sum(O * dO) against the oracle's
    dQ, dK, dV; returns the worst max|g_fd - g| / max|g| over all cases."""
    worst = 0.0
    h = 1e-6
    for N, d in sizes:
        for causal in (False, True):
            for pad in (False, True):
                for p in (0.0, 0.3):
                    B, H = 1, 2
                    key_len = max(1, N - 2) if pad else N
                    q, k, v, do = (_rand(B, H, N, d) for _ in range(4))
                    sc = 1 / math.sqrt(d)
                    dQ, dK, dV, _ = oracle.attn_bwd(q, k, v, do, sc, causal, [key_len], p, 3,
                                                    _lib=L)

                    def f(qq, kk, vv):
                        O, _ = oracle.attn_fwd(qq, kk, vv, sc, causal, [key_len], p, 3, _lib=L)
                        return float((O * do).sum())

                    for which, g in ((0, dQ), (1, dK), (2, dV)):
                        args = [q, k, v]
                        fd = np.zeros_like(g)
                        base = args[which]
                        for idx in np.ndindex(base.shape):
                            old = base[idx]
                            base[idx] = old + h
                            fp = f(*args)
                            base[idx] = old - h
                            fm = f(*args)
                            base[idx] = old
                            fd[idx] = (fp - fm) / (2 * h)
                        denom = max(np.abs(g).max(), 1e-12)
                        worst = max(worst, np.abs(fd - g).max() / denom)
    return worst


def pin_dk_sums_to_zero(L) -> float:
    """sum_j dS_ij = 0 for every row with a valid key, hence sum_j dK_j = 0."""
    B, H, N, d = 2, 2, 15, 6
    q, k, v, do = (_rand(B, H, N, d) for _ in range(4))
    _, dK, _, _ = oracle.attn_bwd(q, k, v, do, 0.4, True, [15, 9], 0.2, 11, _lib=L)
    return float(np.abs(dK.sum(axis=2)).max())


def pin_D_equals_dO_dot_O(L) -> float:
    """D_i = sum_j P_ij dP_ij equals dO_i . O_i."""
    B, H, N, d = 1, 3, 14, 5
    q, k, v, do = (_rand(B, H, N, d) for _ in range(4))
    O, _ = oracle.attn_fwd(q, k, v, 0.45, False, [12], 0.3, 21, _lib=L)
    _, _, _, D = oracle.attn_bwd(q, k, v, do, 0.45, False, [12], 0.3, 21, _lib=L)
    return float(np.abs(D - (O * do).sum(-1)).max())


def pin_tile_invariance(L) -> float:
    """The online-softmax recurrence with tiles Br x Bc in {1, 3, 64, N} gives
    the materialised result (relative error)."""
    worst = 0.0
    N, d = 37, 8
    for causal in (False, True):
        for key_len, p in ((37, 0.0), (23, 0.0), (30, 0.35)):
            q, k, v = _rand(1, 1, N, d), _rand(1, 1, N, d), _rand(1, 1, N, d)
            O, LSE = oracle.attn_fwd(q, k, v, 0.35, causal, [key_len], p, 13, _lib=L)
            for Br in (1, 3, 64, N):
                for Bc in (1, 3, 64, N):
                    Ot, Lt = oracle.head_fwd_tiled(q[0, 0], k[0, 0], v[0, 0], 0.35, Br, Bc,
                                                   causal, key_len, p, 13, _lib=L)
                    worst = max(worst, np.abs(Ot - O[0, 0]).max() / np.abs(O).max())
                    worst = max(worst, np.abs(Lt - LSE[0, 0]).max() / np.abs(LSE).max())
    return worst


def pin_rows_variant(L) -> float:
    """The row-at-a-time evaluation equals the materialised one."""
    N, d = 40, 8
    q, k, v = _rand(1, 1, N, d), _rand(1, 1, N, d), _rand(1, 1, N, d)
    worst = 0.0
    for causal, key_len, p in ((False, 40, 0.0), (True, 31, 0.2)):
        O, LSE = oracle.attn_fwd(q, k, v, 0.3, causal, [key_len], p, 17, _lib=L)
        rows = np.array([0, 1, 17, 39])
        Or, Lr = oracle.head_fwd_rows(q[0, 0], k[0, 0], v[0, 0], rows, 0.3, causal, key_len, p,
                                      17, 0, 0, _lib=L)
        worst = max(worst, np.abs(Or - O[0, 0, rows]).max(), np.abs(Lr - LSE[0, 0, rows]).max())
    return worst


def pin_dropout_statistics(L) -> float:
    """Kept fraction of a 512 x 512 mask within 5 sigma of 1 - p, for several
    p; Philox words uniform (mean within 5 sigma of 2^31 - 0.5), and so their
    16-bit halves (mean within 5 sigma of 2^15 - 0.5).  Returns the largest
    deviation in units of sigma."""
    worst = 0.0
    n = 512 * 512
    for p in (0.1, 0.5, 0.9):
        Z = oracle.dropout_mask(0x5EED0005, 3, 7, 512, 512, p, _lib=L)
        sigma = math.sqrt(p * (1 - p) / n)
        worst = max(worst, abs(Z.mean() - (1 - p)) / sigma)
    words = np.array([oracle.philox4x32_10([i, 0, 0, 0], [1, 2], _lib=L) for i in range(2048)],
                     dtype=np.float64).ravel()
    sigma = (2.0**32) / math.sqrt(12 * words.size)
    worst = max(worst, abs(words.mean() - (2.0**31 - 0.5)) / sigma)
    halves = np.concatenate([np.floor(words / 65536.0), np.mod(words, 65536.0)])
    sigma = 65536.0 / math.sqrt(12 * halves.size)
    worst = max(worst, abs(halves.mean() - (2.0**15 - 0.5)) / sigma)
    return worst


def pin_dropout_threshold(L) -> float:
    """t = floor(p 2^16) clamped to 2^16 - 1; p = 0 keeps everything."""
    bad = 0
    bad += oracle.dropout_threshold(0.0, _lib=L) != 0
    bad += oracle.dropout_threshold(0.5, _lib=L) != 2**15
    bad += oracle.dropout_threshold(0.1, _lib=L) != 6553
    bad += oracle.dropout_threshold(1 - 2**-40, _lib=L) != 2**16 - 1
    Z = oracle.dropout_mask(1, 0, 0, 8, 8, 0.0, _lib=L)
    bad += int(Z.min() != 1)
    return float(bad)


def pin_dropout_counter_layout(L) -> float:
    """The keep bit of (i, j) is a 16-bit draw of Philox at counter
    (i, j>>3, h, b) under key (lo32(seed), hi32(seed)): word (j>>1)&3, its
    low half for even j and its high half for odd j, compared with t (drop
    iff draw < t).  Nine columns cross a counter boundary."""
    seed = 0x0000000A0000000B
    p = 0.5
    t = oracle.dropout_threshold(p, _lib=L)
    Z = oracle.dropout_mask(seed, 2, 5, 6, 9, p, _lib=L)
    bad = 0
    for i in range(6):
        for j in range(9):
            w = int(oracle.philox4x32_10([i, j >> 3, 5, 2], [0xB, 0xA], _lib=L)[(j >> 1) & 3])
            draw = (w >> 16) if j % 2 else (w & 0xFFFF)
            bad += int(Z[i, j] != (0 if draw < t else 1))
    return float(bad)


def pin_row_slices_partition(L) -> float:
    """Row slices: O, LSE, dQ of each slice equal the full evaluation's rows,
    and the slices' dK/dV contributions sum to the full dK/dV."""
    N, d = 29, 8
    worst = 0.0
    for causal, key_len, p in ((False, 29, 0.0), (True, 21, 0.3)):
        q, k, v, do = (_rand(1, 1, N, d) for _ in range(4))
        O, LSE = oracle.attn_fwd(q, k, v, 0.4, causal, [key_len], p, 9, _lib=L)
        dQ, dK, dV, _ = oracle.attn_bwd(q, k, v, do, 0.4, causal, [key_len], p, 9, _lib=L)
        sk, sv = np.zeros((N, d)), np.zeros((N, d))
        for r0, nr in ((0, 10), (10, 1), (11, 18)):
            Or, Lr, dQr, dKp, dVp = oracle.heads_rows_fwd_bwd(
                q[0], k[0], v[0], do[0], [0], [0], [key_len], 0.4, r0, nr, causal, p, 9, _lib=L)
            sk += dKp[0]
            sv += dVp[0]
            worst = max(worst, np.abs(Or[0] - O[0, 0, r0:r0 + nr]).max(),
                        np.abs(dQr[0] - dQ[0, 0, r0:r0 + nr]).max())
            fin = np.isfinite(LSE[0, 0, r0:r0 + nr])
            worst = max(worst, np.abs(Lr[0][fin] - LSE[0, 0, r0:r0 + nr][fin]).max())
        worst = max(worst, np.abs(sk - dK[0, 0]).max(), np.abs(sv - dV[0, 0]).max())
    return worst


PINS = {
    "zero_query": (pin_zero_query, 1e-12),
    "causal_row0": (pin_causal_row0, 1e-12),
    "single_key": (pin_single_key, 1e-12),
    "rows_are_distributions": (pin_rows_are_distributions, 1e-11),
    "two_keys_sigmoid": (pin_two_keys_sigmoid, 1e-13),
    "key_shift_invariance": (pin_key_shift_invariance, 1e-12),
    "torch_autograd": (pin_torch_autograd, 1e-12),
    "window_one": (pin_window_one, 1e-12),
    "window_torch": (pin_window_torch, 1e-12),
    "cross_attention_torch": (pin_cross_attention_torch, 1e-12),
    "varlen_equal_lengths": (pin_varlen_equal_lengths, 1e-12),
    "varlen_torch": (pin_varlen_torch, 1e-12),
    "finite_differences": (pin_finite_differences, 1e-6),
    "dk_sums_to_zero": (pin_dk_sums_to_zero, 1e-12),
    "D_equals_dO_dot_O": (pin_D_equals_dO_dot_O, 1e-12),
    "tile_invariance": (pin_tile_invariance, 1e-12),
    "rows_variant": (pin_rows_variant, 1e-12),
    "row_slices_partition": (pin_row_slices_partition, 1e-12),
    "dropout_statistics": (pin_dropout_statistics, 5.0),
    "dropout_threshold": (pin_dropout_threshold, 0.5),
    "dropout_counter_layout": (pin_dropout_counter_layout, 0.5),
}
