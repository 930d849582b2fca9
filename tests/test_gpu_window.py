"""Sliding-window attention: forward and backward parity against the float64
oracle.  Key blocks wholly outside the window are skipped by the kernels, so
these cases also check the block ranges (first and last block of every tile
and key block) and the masks of the boundary blocks."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_58_gb300.workloads import make_inputs
from gpu_helpers import (GRAD_RTOL, O_ATOL, f64, gpu_fwd_bwd, grad_err, lse_err, oracle_bwd,
                         oracle_fwd)

pytestmark = pytest.mark.gpu


def _check(inp):
    o, lse, dq, dk, dv = gpu_fwd_bwd(inp)
    O_ref, L_ref = oracle_fwd(inp)
    assert float(np.abs(f64(o) - O_ref).max()) <= O_ATOL
    assert lse_err(f64(lse), L_ref) <= 4e-3
    dQ, dK, dV, _ = oracle_bwd(inp)
    errs = {"dQ": grad_err(f64(dq), dQ), "dK": grad_err(f64(dk), dK), "dV": grad_err(f64(dv), dV)}
    for n in errs:
        assert errs[n] <= GRAD_RTOL, errs


@pytest.mark.parametrize("window", [1, 50, 128, 200, 700])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N,d", [(513, 64), (300, 128)])
def test_window_shapes(window, causal, N, d):
    inp = make_inputs(2, 2, N, d, gen_seed=7 * window + N + d + causal, causal=causal)
    inp.window = window
    _check(inp)


@pytest.mark.parametrize("causal", [True, False])
def test_window_padding_dropout(causal):
    inp = make_inputs(3, 2, 700, 64, gen_seed=123 + causal, causal=causal,
                      key_len_range=(200, 700), dropout_p=0.15, dropout_seed_value=0x5EED0777)
    inp.window = 160
    _check(inp)


def test_window_full_size_sampled_heads():
    """N = 4096, d = 128, causal, window 512: full-size launch, oracle on two heads."""
    inp = make_inputs(2, 4, 4096, 128, gen_seed=4242, causal=True)
    inp.window = 512
    o, lse, dq, dk, dv = gpu_fwd_bwd(inp)
    heads = [(0, 0), (1, 3)]
    sel = lambda t: np.stack([f64(t[b, h]) for b, h in heads])  # noqa: E731
    b_idx = np.array([b for b, _ in heads], dtype=np.int32)
    h_idx = np.array([h for _, h in heads], dtype=np.int32)
    kl = np.full(len(heads), 4096, dtype=np.int32)
    O_ref, _ = oracle.heads_fwd(sel(inp.q), sel(inp.k), sel(inp.v), b_idx, h_idx, kl, inp.scale,
                                True, window=512)
    assert float(np.abs(sel(o) - O_ref).max()) <= O_ATOL
    dQ, dK, dV, _ = oracle.heads_bwd(sel(inp.q), sel(inp.k), sel(inp.v), sel(inp.do), b_idx,
                                     h_idx, kl, inp.scale, True, window=512)
    for g, ref in ((dq, dQ), (dk, dK), (dv, dV)):
        for x in range(len(heads)):
            assert grad_err(sel(g)[x], ref[x]) <= GRAD_RTOL
