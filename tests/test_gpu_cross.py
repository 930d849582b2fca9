"""Cross-attention (N query rows, Nk keys, N != Nk): forward and backward
parity against the float64 oracle.

Queries are the last N positions of the key sequence: query i stands at key
position i + Nk - N in the causal and window tests.  With N > Nk and a causal
mask the first N - Nk queries see no key at all (O = 0, LSE = -inf, zero dQ),
which also exercises query tiles that are partly or wholly empty."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_58_gb300.workloads import make_inputs
from gpu_helpers import GRAD_RTOL, O_ATOL, f64, gpu_fwd_bwd, grad_err, lse_err

pytestmark = pytest.mark.gpu


def _oracle(inp):
    kl = None if inp.key_lens is None else inp.key_lens.numpy()
    return oracle.attn_fwd_bwd_qk(f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.do), inp.scale,
                                  inp.causal, kl, inp.dropout_p, inp.seed, window=inp.window)


def _check(inp):
    o, lse, dq, dk, dv = gpu_fwd_bwd(inp)
    assert dk.shape == inp.k.shape and dv.shape == inp.v.shape and dq.shape == inp.q.shape
    O_ref, L_ref, dQ, dK, dV = _oracle(inp)
    assert float(np.abs(f64(o) - O_ref).max()) <= O_ATOL
    assert lse_err(f64(lse), L_ref) <= 4e-3
    errs = {"dQ": grad_err(f64(dq), dQ), "dK": grad_err(f64(dk), dK), "dV": grad_err(f64(dv), dV)}
    for n in errs:
        assert errs[n] <= GRAD_RTOL, errs


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N,Nk,d", [
    (200, 700, 64),    # a chunk of queries continuing a longer key sequence
    (129, 1000, 128),
    (1, 900, 128),     # a single query (decode step)
    (600, 250, 64),    # more queries than keys: causal rows 0..349 see nothing
    (300, 1, 128),     # one key
    (384, 128, 128),   # whole tiles only
])
def test_cross_shapes(causal, N, Nk, d):
    inp = make_inputs(2, 2, N, d, gen_seed=31 * N + Nk + d + causal, causal=causal, Nk=Nk)
    _check(inp)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N,Nk,window", [(300, 800, 100), (700, 260, 90), (256, 640, 1)])
def test_cross_window(causal, N, Nk, window):
    inp = make_inputs(2, 2, N, 64, gen_seed=N + Nk + window + causal, causal=causal, Nk=Nk)
    inp.window = window
    _check(inp)


@pytest.mark.parametrize("causal", [True, False])
def test_cross_padding_dropout(causal):
    inp = make_inputs(3, 2, 333, 128, gen_seed=808 + causal, causal=causal, Nk=777,
                      key_len_range=(100, 777), dropout_p=0.2, dropout_seed_value=0x5EED0CC5)
    _check(inp)


def test_cross_fp16():
    inp = make_inputs(2, 2, 250, 128, dtype=torch.float16, gen_seed=99, causal=True, Nk=650)
    _check(inp)


def test_cross_full_size_sampled_heads():
    """N = 1024 queries against Nk = 8192 keys, d = 128, causal: a full-size
    launch, the oracle on two whole heads (every row, so dK and dV too).  No
    dropout, so the heads can be handed to the oracle as one batch."""
    inp = make_inputs(2, 4, 1024, 128, gen_seed=5150, causal=True, Nk=8192)
    o, lse, dq, dk, dv = gpu_fwd_bwd(inp)
    heads = ((0, 1), (1, 3))
    sel = lambda t: np.stack([f64(t[b, h]) for b, h in heads])[None]  # noqa: E731
    O_ref, L_ref, dQ, dK, dV = oracle.attn_fwd_bwd_qk(sel(inp.q), sel(inp.k), sel(inp.v),
                                                      sel(inp.do), inp.scale, True)
    assert float(np.abs(sel(o) - O_ref).max()) <= O_ATOL
    assert lse_err(sel(lse), L_ref) <= 4e-3
    for g, ref in ((dq, dQ), (dk, dK), (dv, dV)):
        for x in range(len(heads)):
            assert grad_err(sel(g)[0, x], ref[0, x]) <= GRAD_RTOL
