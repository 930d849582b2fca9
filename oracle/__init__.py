"""Float64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  Only the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py`` may import this package.  The CUDA
library never calls it, and it shares no code with the CUDA library: the
arithmetic lives in ``oracle.c`` (plain C, OpenMP over heads), built with gcc
into ``oracle/_build/liboracle.so``; this module only marshals numpy arrays.

What the oracle computes, and which page passage each function follows, is
described at the top of ``oracle.c``.  Every array is float64 and contiguous,
laid out [B, H, N, d] (LSE and D: [B, H, N]).
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build", platform.machine())
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_ip = ctypes.POINTER(ctypes.c_int32)
_up = ctypes.POINTER(ctypes.c_uint32)
_bp = ctypes.POINTER(ctypes.c_uint8)


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile ``oracle.c`` with gcc (OpenMP) if the library is missing or stale."""
    if (not force and os.path.exists(out)
            and os.path.getmtime(out) >= os.path.getmtime(src)):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-fPIC", "-shared", "-std=c11", "-Wall",
           "-o", tmp, src, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    lib.oracle_philox4x32_10.argtypes = [_up, _up, _up]
    lib.oracle_philox4x32_10.restype = None
    lib.oracle_dropout_threshold.argtypes = [ctypes.c_double]
    lib.oracle_dropout_threshold.restype = ctypes.c_uint32
    lib.oracle_dropout_mask.argtypes = [ctypes.c_uint64, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_double, _bp]
    lib.oracle_dropout_mask.restype = None
    # N, d, scale, causal, window, key_len, p, seed, b, h
    head_common = [ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_int, ctypes.c_int,
                   ctypes.c_int, ctypes.c_double, ctypes.c_uint64, ctypes.c_int, ctypes.c_int]
    lib.oracle_head_fwd.argtypes = [_dp, _dp, _dp, _dp, _dp] + head_common
    lib.oracle_head_fwd.restype = ctypes.c_int
    lib.oracle_head_bwd.argtypes = [_dp] * 8 + head_common
    lib.oracle_head_bwd.restype = ctypes.c_int
    lib.oracle_head_fwd_rows.argtypes = [_dp, _dp, _dp, _ip, ctypes.c_int, _dp, _dp] + head_common
    lib.oracle_head_fwd_rows.restype = ctypes.c_int
    lib.oracle_head_fwd_tiled.argtypes = [_dp] * 5 + head_common + [ctypes.c_int, ctypes.c_int]
    lib.oracle_head_fwd_tiled.restype = ctypes.c_int
    # nh, b_idx, h_idx, key_len, N, d, scale, causal, window, p, seed, nthreads
    heads_common = [ctypes.c_int, _ip, _ip, _ip, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                    ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_uint64, ctypes.c_int]
    lib.oracle_heads_fwd.argtypes = [_dp] * 5 + heads_common
    lib.oracle_heads_fwd.restype = ctypes.c_int
    lib.oracle_heads_bwd.argtypes = [_dp] * 8 + heads_common
    lib.oracle_heads_bwd.restype = ctypes.c_int
    lib.oracle_heads_rows_fwd_bwd.argtypes = (   # ..., key_len, Nq, Nk, d, scale, ...
        [_dp] * 4 + [ctypes.c_int, _ip, _ip, _ip, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                     ctypes.c_double,
                     ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_uint64, ctypes.c_int,
                     ctypes.c_int]
        + [_dp] * 5 + [ctypes.c_int])
    lib.oracle_heads_rows_fwd_bwd.restype = ctypes.c_int
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ctypes.c_int
    return lib


def lib():
    """The loaded oracle library (built on first use)."""
    global _lib
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
        return _lib


def load_variant(path: str):
    """Load another build of ``oracle.c`` (used by the mutation tests)."""
    return _bind(ctypes.CDLL(path))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray, t):
    return a.ctypes.data_as(t)


# --------------------------------------------------------------------------
# Philox / dropout bits
# --------------------------------------------------------------------------
def philox4x32_10(ctr, key, _lib=None) -> np.ndarray:
    """Philox4x32-10 of one 4-word counter under one 2-word key -> uint32[4]."""
    L = _lib or lib()
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32).reshape(4))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32).reshape(2))
    out = np.zeros(4, dtype=np.uint32)
    L.oracle_philox4x32_10(_ptr(c, _up), _ptr(k, _up), _ptr(out, _up))
    return out


def dropout_threshold(p: float, _lib=None) -> int:
    return int((_lib or lib()).oracle_dropout_threshold(float(p)))


def dropout_mask(seed: int, b: int, h: int, rows: int, cols: int, p: float,
                 _lib=None) -> np.ndarray:
    """Keep mask Z (uint8 0/1) of head (b, h), shape [rows, cols]."""
    L = _lib or lib()
    Z = np.zeros((rows, cols), dtype=np.uint8)
    L.oracle_dropout_mask(int(seed), int(b), int(h), int(rows), int(cols), float(p),
                          _ptr(Z, _bp))
    return Z


# --------------------------------------------------------------------------
# Attention
# --------------------------------------------------------------------------
def _key_lens(key_lens, B, N):
    if key_lens is None:
        return np.full(B, N, dtype=np.int32)
    kl = np.ascontiguousarray(np.asarray(key_lens, dtype=np.int32).reshape(B))
    return kl


def attn_fwd(Q, K, V, scale=None, causal=False, key_lens=None, dropout_p=0.0, seed=0,
             nthreads=0, window=0, _lib=None):
    """O, LSE of softmax(scale*Q K^T + mask) (dropout) V for [B,H,N,d] inputs."""
    L = _lib or lib()
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, N, d = Q.shape
    if K.shape != Q.shape or V.shape != Q.shape:
        raise ValueError("attn_fwd takes square problems (K, V shaped like Q); "
                         "use attn_fwd_bwd_qk for N_k != N")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kl = _key_lens(key_lens, B, N)
    nh = B * H
    b_idx = np.repeat(np.arange(B, dtype=np.int32), H)
    h_idx = np.tile(np.arange(H, dtype=np.int32), B)
    klh = np.repeat(kl, H).astype(np.int32)
    O = np.zeros_like(Q)
    LSE = np.zeros((B, H, N), dtype=np.float64)
    r = L.oracle_heads_fwd(_ptr(Q, _dp), _ptr(K, _dp), _ptr(V, _dp), _ptr(O, _dp),
                           _ptr(LSE, _dp), nh, _ptr(b_idx, _ip), _ptr(h_idx, _ip),
                           _ptr(klh, _ip), N, d, float(scale), int(bool(causal)), int(window),
                           float(dropout_p), int(seed), int(nthreads))
    if r != 0:
        raise ValueError("oracle_heads_fwd rejected its arguments")
    return O, LSE


def attn_bwd(Q, K, V, dO, scale=None, causal=False, key_lens=None, dropout_p=0.0, seed=0,
             nthreads=0, window=0, _lib=None):
    """dQ, dK, dV (and D = rowsum(dO*O)) of the same chain."""
    L = _lib or lib()
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, N, d = Q.shape
    if K.shape != Q.shape or V.shape != Q.shape or dO.shape != Q.shape:
        raise ValueError("attn_bwd takes square problems (K, V, dO shaped like Q); "
                         "use attn_fwd_bwd_qk for N_k != N")
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kl = _key_lens(key_lens, B, N)
    nh = B * H
    b_idx = np.repeat(np.arange(B, dtype=np.int32), H)
    h_idx = np.tile(np.arange(H, dtype=np.int32), B)
    klh = np.repeat(kl, H).astype(np.int32)
    dQ, dK, dV = np.zeros_like(Q), np.zeros_like(Q), np.zeros_like(Q)
    D = np.zeros((B, H, N), dtype=np.float64)
    r = L.oracle_heads_bwd(_ptr(Q, _dp), _ptr(K, _dp), _ptr(V, _dp), _ptr(dO, _dp),
                           _ptr(dQ, _dp), _ptr(dK, _dp), _ptr(dV, _dp), _ptr(D, _dp),
                           nh, _ptr(b_idx, _ip), _ptr(h_idx, _ip), _ptr(klh, _ip),
                           N, d, float(scale), int(bool(causal)), int(window), float(dropout_p),
                           int(seed), int(nthreads))
    if r != 0:
        raise ValueError("oracle_heads_bwd rejected its arguments")
    return dQ, dK, dV, D


def heads_fwd(Qh, Kh, Vh, b_idx, h_idx, key_len, scale, causal=False, dropout_p=0.0,
              seed=0, nthreads=0, window=0, _lib=None):
    """Forward of selected heads.  Qh..Vh: [nh, N, d]; b_idx/h_idx/key_len: [nh]."""
    L = _lib or lib()
    Qh, Kh, Vh = _f64(Qh), _f64(Kh), _f64(Vh)
    nh, N, d = Qh.shape
    b_idx = np.ascontiguousarray(b_idx, dtype=np.int32)
    h_idx = np.ascontiguousarray(h_idx, dtype=np.int32)
    key_len = np.ascontiguousarray(key_len, dtype=np.int32)
    O = np.zeros_like(Qh)
    LSE = np.zeros((nh, N), dtype=np.float64)
    r = L.oracle_heads_fwd(_ptr(Qh, _dp), _ptr(Kh, _dp), _ptr(Vh, _dp), _ptr(O, _dp),
                           _ptr(LSE, _dp), nh, _ptr(b_idx, _ip), _ptr(h_idx, _ip),
                           _ptr(key_len, _ip), N, d, float(scale), int(bool(causal)), int(window),
                           float(dropout_p), int(seed), int(nthreads))
    if r != 0:
        raise ValueError("oracle_heads_fwd rejected its arguments")
    return O, LSE


def heads_bwd(Qh, Kh, Vh, dOh, b_idx, h_idx, key_len, scale, causal=False, dropout_p=0.0,
              seed=0, nthreads=0, window=0, _lib=None):
    """Backward of selected heads.  Arrays [nh, N, d]; returns dQ, dK, dV, D."""
    L = _lib or lib()
    Qh, Kh, Vh, dOh = _f64(Qh), _f64(Kh), _f64(Vh), _f64(dOh)
    nh, N, d = Qh.shape
    b_idx = np.ascontiguousarray(b_idx, dtype=np.int32)
    h_idx = np.ascontiguousarray(h_idx, dtype=np.int32)
    key_len = np.ascontiguousarray(key_len, dtype=np.int32)
    dQ, dK, dV = np.zeros_like(Qh), np.zeros_like(Qh), np.zeros_like(Qh)
    D = np.zeros((nh, N), dtype=np.float64)
    r = L.oracle_heads_bwd(_ptr(Qh, _dp), _ptr(Kh, _dp), _ptr(Vh, _dp), _ptr(dOh, _dp),
                           _ptr(dQ, _dp), _ptr(dK, _dp), _ptr(dV, _dp), _ptr(D, _dp),
                           nh, _ptr(b_idx, _ip), _ptr(h_idx, _ip), _ptr(key_len, _ip),
                           N, d, float(scale), int(bool(causal)), int(window), float(dropout_p),
                           int(seed), int(nthreads))
    if r != 0:
        raise ValueError("oracle_heads_bwd rejected its arguments")
    return dQ, dK, dV, D


def head_fwd_rows(q, k, v, rows, scale, causal=False, key_len=None, dropout_p=0.0, seed=0,
                  b=0, h=0, window=0, _lib=None):
    """Selected rows of one head ([N, d] inputs) without an N x N array."""
    L = _lib or lib()
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, d = q.shape
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    kl = N if key_len is None else int(key_len)
    O = np.zeros((len(rows), d), dtype=np.float64)
    LSE = np.zeros(len(rows), dtype=np.float64)
    r = L.oracle_head_fwd_rows(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(rows, _ip),
                               len(rows), _ptr(O, _dp), _ptr(LSE, _dp), N, d, float(scale),
                               int(bool(causal)), int(window), kl, float(dropout_p), int(seed), int(b),
                               int(h))
    if r != 0:
        raise ValueError("oracle_head_fwd_rows rejected its arguments")
    return O, LSE


def head_fwd_tiled(q, k, v, scale, Br, Bc, causal=False, key_len=None, dropout_p=0.0,
                   seed=0, b=0, h=0, window=0, _lib=None):
    """One head through the online-softmax recurrence with tiles Br x Bc."""
    L = _lib or lib()
    q, k, v = _f64(q), _f64(k), _f64(v)
    N, d = q.shape
    kl = N if key_len is None else int(key_len)
    O = np.zeros((N, d), dtype=np.float64)
    LSE = np.zeros(N, dtype=np.float64)
    r = L.oracle_head_fwd_tiled(_ptr(q, _dp), _ptr(k, _dp), _ptr(v, _dp), _ptr(O, _dp),
                                _ptr(LSE, _dp), N, d, float(scale), int(bool(causal)), int(window), kl,
                                float(dropout_p), int(seed), int(b), int(h), int(Br), int(Bc))
    if r != 0:
        raise ValueError("oracle_head_fwd_tiled rejected its arguments")
    return O, LSE


def heads_rows_fwd_bwd(Qh, Kh, Vh, dOh, b_idx, h_idx, key_len, scale, row0, nrows,
                       causal=False, dropout_p=0.0, seed=0, nthreads=0, window=0, _lib=None):
    """Forward and backward of query rows [row0, row0+nrows) of selected heads.

    Qh, dOh are [nh, Nq, d] and Kh, Vh [nh, Nk, d]; Nq != Nk aligns the
    queries with the last keys (see oracle.c).  Returns O_rows, LSE_rows,
    dQ_rows ([nh, nrows, ...]) and the rows' contributions to dK and dV
    ([nh, Nk, d])."""
    L = _lib or lib()
    Qh, Kh, Vh, dOh = _f64(Qh), _f64(Kh), _f64(Vh), _f64(dOh)
    nh, N, d = Qh.shape
    Nk = Kh.shape[1]
    b_idx = np.ascontiguousarray(b_idx, dtype=np.int32)
    h_idx = np.ascontiguousarray(h_idx, dtype=np.int32)
    key_len = np.ascontiguousarray(key_len, dtype=np.int32)
    O = np.zeros((nh, nrows, d))
    LSE = np.zeros((nh, nrows))
    dQ = np.zeros((nh, nrows, d))
    dK = np.zeros((nh, Nk, d))
    dV = np.zeros((nh, Nk, d))
    r = L.oracle_heads_rows_fwd_bwd(_ptr(Qh, _dp), _ptr(Kh, _dp), _ptr(Vh, _dp), _ptr(dOh, _dp),
                                    nh, _ptr(b_idx, _ip), _ptr(h_idx, _ip), _ptr(key_len, _ip),
                                    N, Nk, d, float(scale), int(bool(causal)), int(window), float(dropout_p),
                                    int(seed), int(row0), int(nrows), _ptr(O, _dp),
                                    _ptr(LSE, _dp), _ptr(dQ, _dp), _ptr(dK, _dp), _ptr(dV, _dp),
                                    int(nthreads))
    if r != 0:
        raise ValueError("oracle_heads_rows_fwd_bwd rejected its arguments")
    return O, LSE, dQ, dK, dV


def attn_fwd_bwd_qk(Q, K, V, dO, scale=None, causal=False, key_lens=None, dropout_p=0.0,
                    seed=0, window=0, nthreads=0, _lib=None):
    """Forward and backward for Q, dO [B,H,Nq,d] and K, V [B,H,Nk,d], Nq and
    Nk free (cross-attention, queries aligned with the last keys).  Returns
    O, LSE, dQ, dK, dV."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    kl = _key_lens(key_lens, B, Nk)
    b_idx = np.repeat(np.arange(B, dtype=np.int32), H)
    h_idx = np.tile(np.arange(H, dtype=np.int32), B)
    klh = np.repeat(kl, H).astype(np.int32)
    O, LSE, dQ, dK, dV = heads_rows_fwd_bwd(
        Q.reshape(B * H, Nq, d), K.reshape(B * H, Nk, d), V.reshape(B * H, Nk, d),
        dO.reshape(B * H, Nq, d), b_idx, h_idx, klh, scale, 0, Nq, causal=causal,
        dropout_p=dropout_p, seed=seed, nthreads=nthreads, window=window, _lib=_lib)
    return (O.reshape(B, H, Nq, d), LSE.reshape(B, H, Nq), dQ.reshape(B, H, Nq, d),
            dK.reshape(B, H, Nk, d), dV.reshape(B, H, Nk, d))


def attn_fwd_bwd_varlen(Q, K, V, dO, cu_q, cu_k, scale=None, causal=False, dropout_p=0.0,
                        seed=0, window=0, nthreads=0, _lib=None):
    """Forward and backward over packed sequences: Q, dO [Tq, H, d], K, V
    [Tk, H, d]; sequence b holds query rows [cu_q[b], cu_q[b+1]) and key rows
    [cu_k[b], cu_k[b+1]) and is attended on its own (queries aligned with its
    last keys), with dropout counters (i, j>>3, h, b) counted within the
    sequence.  Returns O [Tq, H, d], LSE [H, Tq], dQ, dK, dV."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    Tq, H, d = Q.shape
    Tk = K.shape[0]
    cu_q = np.asarray(cu_q, dtype=np.int64)
    cu_k = np.asarray(cu_k, dtype=np.int64)
    if scale is None:
        scale = 1.0 / np.sqrt(d)
    O = np.zeros((Tq, H, d))
    LSE = np.full((H, Tq), -np.inf)
    dQ = np.zeros((Tq, H, d))
    dK = np.zeros((Tk, H, d))
    dV = np.zeros((Tk, H, d))
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        n, nk = q1 - q0, k1 - k0
        if n == 0 or nk == 0:   # no query, or no key: O = 0, LSE = -inf, zero gradients
            continue
        per_head = lambda x: np.ascontiguousarray(x.transpose(1, 0, 2))  # noqa: E731
        o, lse, dq, dk, dv = heads_rows_fwd_bwd(
            per_head(Q[q0:q1]), per_head(K[k0:k1]), per_head(V[k0:k1]), per_head(dO[q0:q1]),
            np.full(H, b), np.arange(H), np.full(H, nk), scale, 0, n, causal=causal,
            dropout_p=dropout_p, seed=seed, nthreads=nthreads, window=window, _lib=_lib)
        O[q0:q1] = o.transpose(1, 0, 2)
        LSE[:, q0:q1] = lse
        dQ[q0:q1] = dq.transpose(1, 0, 2)
        dK[k0:k1] = dk.transpose(1, 0, 2)
        dV[k0:k1] = dv.transpose(1, 0, 2)
    return O, LSE, dQ, dK, dV


def num_threads() -> int:
    return int(lib().oracle_num_threads())
