"""e4m3 (FP8) inputs: forward parity against the float64 oracle, with the
tolerance derived from the one rounding the fp8 path adds.

Q, K, V are e4m3 values; the oracle computes exact attention on those values
(upcast to float64).  S = scale Q K^T is then exact up to fp32 accumulation,
and the kernel's only coarse step is rounding P to e4m3 for the P V product
(l and LSE use the unrounded P).  With P_ij = exp(s_ij - m_i) <= 1 and
l_i = sum_j P_ij, a round-to-nearest e4m3 value is within 2^-4 P_ij of P_ij
for P_ij >= 2^-6 (3 mantissa bits) and within 2^-10 below (the subnormal
step is 2^-9).  The kernel rounds P relative to a reference max that is at
most the row max, i.e. on values at least as large, so these bounds hold a
fortiori.  Hence, per output element,

    |O_ic - O_ref_ic| <= (2^-4 sum_{P >= 2^-6} P_ij F_ij |V_jc|
                          + 2^-10 sum_{P < 2^-6} F_ij |V_jc|) / l_i
                         + 2^-8 |O_ref_ic| + 1e-3,

F_ij = Z_ij / (1 - p) under dropout (else 1); the last two terms cover the
bf16 rounding of O and fp32 accumulation."""
import math

import numpy as np
import pytest
import torch

import exact_attention_58_gb300 as ea
import oracle
from exact_attention_58_gb300.workloads import make_inputs
from gpu_helpers import O_ATOL, f64, gpu_fwd, lse_err

pytestmark = pytest.mark.gpu

FP8 = getattr(torch, "float8_e4m3fn", None)
if FP8 is None:   # pragma: no cover
    pytestmark = [pytest.mark.gpu, pytest.mark.skip(reason="torch without float8_e4m3fn")]


def rounding_bound(q, k, v, scale, causal, key_len, window, p, seed, b, h):
    """Per-element bound above for one head (float64 numpy, q [N, d], k, v [Nk, d])."""
    N, Nk = q.shape[0], k.shape[0]
    s = scale * q @ k.T
    i = np.arange(N)[:, None] + (Nk - N)
    j = np.arange(Nk)[None, :]
    valid = np.broadcast_to(j < key_len, (N, Nk)).copy()
    if causal:
        valid &= j <= i
    if window > 0:
        valid &= i - j < window
        if not causal:
            valid &= j - i < window
    s = np.where(valid, s, -np.inf)
    m = s.max(axis=1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    P = np.where(valid, np.exp(s - m), 0.0)
    l = P.sum(axis=1, keepdims=True)
    F = np.ones_like(P)
    if p > 0:
        F = oracle.dropout_mask(seed, b, h, N, Nk, p).astype(np.float64) / (1 - p)
    big = valid & (P >= 2.0**-6)
    small = valid & (P < 2.0**-6)
    av = np.abs(v)
    num = 2.0**-4 * (np.where(big, P * F, 0.0) @ av) + 2.0**-10 * (np.where(small, F, 0.0) @ av)
    return num / np.where(l > 0, l, 1.0)


def _inputs(B, H, N, d, seed, causal, **kw):
    inp = make_inputs(B, H, N, d, dtype=FP8, gen_seed=seed, causal=causal, with_do=False, **kw)
    return inp


def _check(inp, heads=None):
    o, lse = gpu_fwd(inp)
    assert o.dtype == torch.bfloat16
    B, H = inp.q.shape[:2]
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    kl = inp.key_lens.numpy() if inp.key_lens is not None else np.full(B, inp.k.shape[2])
    worst = 0.0
    for b, h in heads:
        q, k, v = (f64(t[b, h]) for t in (inp.q, inp.k, inp.v))
        O_ref, L_ref, _, _, _ = oracle.heads_rows_fwd_bwd(
            q[None], k[None], v[None], np.zeros_like(q)[None], [b], [h], [int(kl[b])], inp.scale,
            0, q.shape[0], causal=inp.causal, dropout_p=inp.dropout_p, seed=inp.seed,
            window=inp.window)
        bound = rounding_bound(q, k, v, inp.scale, inp.causal, int(kl[b]), inp.window,
                               inp.dropout_p, inp.seed, b, h)
        err = np.abs(f64(o[b, h]) - O_ref[0])
        tol = bound + 2.0**-8 * np.abs(O_ref[0]) + 1e-3
        assert (err <= tol).all(), float((err - tol).max())
        assert lse_err(f64(lse[b, h]), L_ref[0]) <= 4e-3
        worst = max(worst, float((err / tol).max()))
    return worst


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N", [1, 200, 513])
def test_fp8_shapes(causal, N):
    _check(_inputs(2, 2, N, 128, 900 + N + causal, causal))


@pytest.mark.parametrize("causal", [True, False])
def test_fp8_padding_dropout_window(causal):
    inp = _inputs(2, 2, 400, 128, 77 + causal, causal, key_len_range=(150, 400), dropout_p=0.1,
                  dropout_seed_value=0x5EED0F08)
    inp.window = 170
    _check(inp)


def test_fp8_cross_attention():
    inp = make_inputs(2, 2, 150, 128, dtype=FP8, gen_seed=5, causal=True, with_do=False, Nk=600)
    _check(inp)


def test_fp8_full_size_sampled_heads():
    """B = 4, H = 16, N = 4096, d = 128, causal e4m3: the full-size launch,
    two heads checked element by element against the bound."""
    inp = _inputs(4, 16, 4096, 128, 4243, True)
    _check(inp, heads=[(0, 0), (3, 15)])


def test_fp8_precision_study():
    """The e4m3 path against the bf16 path on the same (e4m3-representable)
    values: both against the float64 oracle.  The fp8 error is dominated by
    the rounding of P; it stays within a small multiple of the bf16 error's
    order and well inside the bound above."""
    inp8 = _inputs(1, 4, 1024, 128, 31337, True)
    o8, _ = gpu_fwd(inp8)
    inp16 = make_inputs(1, 4, 1024, 128, gen_seed=31337, causal=True, with_do=False)
    for name in ("q", "k", "v"):
        setattr(inp16, name, getattr(inp8, name).to(torch.float32).to(torch.bfloat16))
    o16, _ = gpu_fwd(inp16)
    O_ref, _ = oracle.attn_fwd(f64(inp8.q), f64(inp8.k), f64(inp8.v), inp8.scale, True)
    e8 = f64(o8) - O_ref
    e16 = f64(o16) - O_ref
    rms8, rms16 = math.sqrt(float((e8**2).mean())), math.sqrt(float((e16**2).mean()))
    print(f"\nfp8 vs oracle: rms {rms8:.3e} max {np.abs(e8).max():.3e}; "
          f"bf16 vs oracle: rms {rms16:.3e} max {np.abs(e16).max():.3e}")
    assert np.abs(e16).max() <= O_ATOL
    assert rms8 <= 2.0**-4 * math.sqrt(float((O_ref**2).mean())) + 1e-3


def test_fp8_packed_sequences():
    """e4m3 packed variable-length sequences, each sequence checked against
    the rounding bound on its own lengths."""
    from exact_attention_58_gb300.workloads import make_packed_inputs
    lens = [150, 33, 300]
    inp = make_packed_inputs(lens, lens, 2, 128, dtype=FP8, gen_seed=808, causal=True)
    q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
    cu = inp.cu_q.cuda()
    o, lse = ea.attn_fwd_varlen(q, k, v, cu, cu, inp.max_q, inp.max_k, causal=True,
                                scale=inp.scale)
    torch.cuda.synchronize()
    assert o.dtype == torch.bfloat16
    qd, kd, vd = f64(inp.q), f64(inp.k), f64(inp.v)
    O_ref, L_ref, _, _, _ = oracle.attn_fwd_bwd_varlen(qd, kd, vd, np.zeros_like(qd),
                                                       inp.cu_q.numpy(), inp.cu_k.numpy(),
                                                       inp.scale, True)
    cuq = inp.cu_q.numpy()
    for b in range(len(lens)):
        s0, s1 = int(cuq[b]), int(cuq[b + 1])
        for h in range(2):
            bound = rounding_bound(qd[s0:s1, h], kd[s0:s1, h], vd[s0:s1, h], inp.scale, True,
                                   s1 - s0, 0, 0.0, 0, b, h)
            err = np.abs(f64(o[s0:s1, h]) - O_ref[s0:s1, h])
            assert (err <= bound + 2.0**-8 * np.abs(O_ref[s0:s1, h]) + 1e-3).all()
            assert lse_err(f64(lse[h, s0:s1]), L_ref[h, s0:s1]) <= 4e-3


def test_fp8_spiky_keys_move_the_row_max():
    """The e4m3 path with keys of the last 32-key chunk of every block scaled
    up six-fold (the values stay in the e4m3 range): large jumps of the row
    max and its rescale of O and l."""
    inp = make_inputs(2, 2, 400, 128, dtype=torch.float32, gen_seed=77, causal=False,
                      with_do=False)
    j = np.arange(400)
    spike = torch.from_numpy(((j % 128) // 32) == 3)
    inp.k[:, :, spike] *= 6.0
    for name in ("q", "k", "v"):
        setattr(inp, name, getattr(inp, name).to(FP8))
    _check(inp)
