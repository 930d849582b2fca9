"""Shared helpers for the GPU parity tests: run the CUDA path through the C ABI
binding and the float64 oracle on the same seeded inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import exact_attention_58_gb300 as ea
import oracle

# Tolerances.  O: max |O - O_ref| <= 2e-2 (bf16 inputs, fp32 accumulation).
# LSE = ln 2 (m + log2 l): the row max m comes from fp32 scores, each the fp32
# sum of d exact products of 16-bit (or e4m3) inputs (absolute error about
# d 2^-24 sum_k |q_k k_k| scale log2e, below 1e-4 for unit-variance inputs at
# d <= 256); l is the fp32 sum of the unrounded exp2 values (ex2.approx, about
# 2^-22 relative each) over at most N keys, at most N 2^-24 relative (2.4e-4
# at N = 4096), which moves LSE by the same amount.  The budget is a few 1e-4;
# 4e-3 is the tolerance, with a margin of ten.
# Gradients: max |g - g_ref| / max |g_ref| <= 5e-2 per tensor.
O_ATOL = 2e-2
LSE_ATOL = 4e-3
GRAD_RTOL = 5e-2


def to_dev(inp):
    dev = "cuda"
    q, k, v = (t.to(dev) for t in (inp.q, inp.k, inp.v))
    do = inp.do.to(dev) if inp.do is not None else None
    kl = inp.key_lens.to(dev) if inp.key_lens is not None else None
    return q, k, v, do, kl


def gpu_fwd(inp):
    q, k, v, _, kl = to_dev(inp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = ea.attn_fwd(q, k, v, causal=inp.causal, key_lens=kl, dropout_p=inp.dropout_p,
                         seed=inp.seed, scale=inp.scale, dev_status=status, window=inp.window)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    return o, lse


def gpu_fwd_bwd(inp):
    q, k, v, do, kl = to_dev(inp)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = ea.attn_fwd(q, k, v, causal=inp.causal, key_lens=kl, dropout_p=inp.dropout_p,
                         seed=inp.seed, scale=inp.scale, dev_status=status, window=inp.window)
    dq, dk, dv = ea.attn_bwd(q, k, v, o, do, lse, causal=inp.causal, key_lens=kl,
                             dropout_p=inp.dropout_p, seed=inp.seed, scale=inp.scale,
                             dev_status=status, window=inp.window)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    return o, lse, dq, dk, dv


def f64(t):
    return t.double().cpu().numpy()


def oracle_fwd(inp):
    kl = None if inp.key_lens is None else inp.key_lens.numpy()
    return oracle.attn_fwd(f64(inp.q), f64(inp.k), f64(inp.v), inp.scale, inp.causal, kl,
                           inp.dropout_p, inp.seed, window=inp.window)


def oracle_bwd(inp):
    kl = None if inp.key_lens is None else inp.key_lens.numpy()
    return oracle.attn_bwd(f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.do), inp.scale,
                           inp.causal, kl, inp.dropout_p, inp.seed, window=inp.window)


def lse_err(lse, lse_ref):
    lse = np.asarray(lse, dtype=np.float64)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isfinite(lse), fin), "LSE -inf pattern differs"
    return float(np.abs(lse[fin] - lse_ref[fin]).max()) if fin.any() else 0.0


def grad_err(g, g_ref):
    g = np.asarray(g, dtype=np.float64)
    denom = np.abs(g_ref).max()
    if denom == 0:
        return float(np.abs(g).max())
    return float(np.abs(g - g_ref).max() / denom)


def sample_rows_check(inp, o, lse, heads, rows):
    """Compare selected (head, row) outputs with the oracle evaluated row by row."""
    B, H, N, d = inp.q.shape
    worst_o, worst_l = 0.0, 0.0
    o = o.float().cpu().numpy()
    lse = lse.cpu().numpy()
    for (b, h) in heads:
        kl = N if inp.key_lens is None else int(inp.key_lens[b])
        Or, Lr = oracle.head_fwd_rows(f64(inp.q[b, h]), f64(inp.k[b, h]), f64(inp.v[b, h]), rows,
                                      inp.scale, inp.causal, kl, inp.dropout_p, inp.seed, b, h)
        worst_o = max(worst_o, float(np.abs(o[b, h, rows] - Or).max()))
        worst_l = max(worst_l, lse_err(lse[b, h, rows], Lr))
    return worst_o, worst_l
