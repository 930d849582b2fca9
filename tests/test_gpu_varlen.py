"""Packed variable-length sequences (q [total_q, H, d], k, v [total_k, H, d],
cumulative offsets): forward and backward parity against the float64 oracle.

Tiles that cross from one sequence into the next are the case to get right:
the loads bring in the next sequence's rows, which the masks and the +inf
log-sum-exp of the backward must cancel, and the last key block of a
sequence must not write into its neighbour.  Sequences without queries or
without keys, and lengths that are not multiples of the tile, are included."""
import numpy as np
import pytest
import torch

import exact_attention_58_gb300 as ea
import oracle
from exact_attention_58_gb300.workloads import make_packed_inputs
from gpu_helpers import GRAD_RTOL, O_ATOL, f64, grad_err, lse_err

pytestmark = pytest.mark.gpu


def _gpu(inp):
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    cu_q, cu_k = inp.cu_q.cuda(), inp.cu_k.cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(causal=inp.causal, window=inp.window, dropout_p=inp.dropout_p, seed=inp.seed,
              scale=inp.scale, dev_status=status)
    o, lse = ea.attn_fwd_varlen(q, k, v, cu_q, cu_k, inp.max_q, inp.max_k, **kw)
    dq, dk, dv = ea.attn_bwd_varlen(q, k, v, o, do, lse, cu_q, cu_k, inp.max_q, inp.max_k, **kw)
    torch.cuda.synchronize()
    assert int(status.item()) == 0, f"device status {int(status.item())}"
    return o, lse, dq, dk, dv


def _oracle(inp):
    return oracle.attn_fwd_bwd_varlen(f64(inp.q), f64(inp.k), f64(inp.v), f64(inp.do),
                                      inp.cu_q.numpy(), inp.cu_k.numpy(), inp.scale, inp.causal,
                                      inp.dropout_p, inp.seed, window=inp.window)


def _check(inp):
    o, lse, dq, dk, dv = _gpu(inp)
    assert o.shape == inp.q.shape and lse.shape == (inp.q.shape[1], inp.q.shape[0])
    O_ref, L_ref, dQ, dK, dV = _oracle(inp)
    assert float(np.abs(f64(o) - O_ref).max()) <= O_ATOL
    assert lse_err(f64(lse), L_ref) <= 4e-3
    errs = {"dQ": grad_err(f64(dq), dQ), "dK": grad_err(f64(dk), dK), "dV": grad_err(f64(dv), dV)}
    for n in errs:
        assert errs[n] <= GRAD_RTOL, errs


SELF = [
    [128, 128],
    [1, 300, 77, 129, 256],
    [513, 5, 260],
    [0, 200, 0, 31],   # empty sequences
]


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("lens", SELF)
def test_varlen_self(causal, d, lens):
    inp = make_packed_inputs(lens, lens, 2, d, gen_seed=sum(lens) + d + causal, causal=causal)
    _check(inp)


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("lens_q,lens_k", [
    ([100, 7, 300], [400, 129, 50]),
    ([1, 1, 1], [700, 3, 129]),     # one query per sequence (decode)
    ([64, 0, 90], [0, 50, 200]),    # a sequence without keys, one without queries
])
def test_varlen_cross(causal, lens_q, lens_k):
    inp = make_packed_inputs(lens_q, lens_k, 3, 128, gen_seed=sum(lens_q) * 7 + sum(lens_k),
                             causal=causal)
    _check(inp)


@pytest.mark.parametrize("causal", [True, False])
def test_varlen_window_dropout(causal):
    lens_q, lens_k = [333, 90, 200], [333, 250, 140]
    inp = make_packed_inputs(lens_q, lens_k, 2, 64, gen_seed=4 + causal, causal=causal,
                             dropout_p=0.2, dropout_seed_value=0x5EED0F00, window=100)
    _check(inp)


def test_varlen_fp16():
    inp = make_packed_inputs([300, 45, 128], [300, 45, 128], 2, 128, dtype=torch.float16,
                             gen_seed=61, causal=True)
    _check(inp)


def test_varlen_max_seqlen_larger_than_needed():
    """max_seqlen is only a bound: a larger value gives the same results."""
    inp = make_packed_inputs([200, 70], [200, 70], 2, 64, gen_seed=3, causal=True)
    a = _gpu(inp)
    inp.max_q, inp.max_k = 1000, 700
    b = _gpu(inp)
    for x, y in zip(a, b):
        assert torch.equal(x, y)


def test_varlen_full_size_sampled_sequences():
    """24 causal sequences of 256 to 4096 tokens (about 50k tokens), H = 16,
    d = 128: a full-size launch, the oracle on two whole sequences."""
    rng = np.random.default_rng(2024)
    lens = [int(x) for x in rng.integers(256, 4097, size=24)]
    inp = make_packed_inputs(lens, lens, 16, 128, gen_seed=77, causal=True)
    o, lse, dq, dk, dv = _gpu(inp)
    cu = inp.cu_q.numpy()
    for b in (3, 17):
        s0, s1 = int(cu[b]), int(cu[b + 1])
        sl = lambda t: f64(t[s0:s1])  # noqa: E731
        one = np.array([0, s1 - s0])
        O_ref, L_ref, dQ, dK, dV = oracle.attn_fwd_bwd_varlen(
            sl(inp.q), sl(inp.k), sl(inp.v), sl(inp.do), one, one, inp.scale, True)
        assert float(np.abs(sl(o) - O_ref).max()) <= O_ATOL
        assert lse_err(f64(lse[:, s0:s1]), L_ref) <= 4e-3
        for g, ref in ((dq, dQ), (dk, dK), (dv, dV)):
            assert grad_err(sl(g), ref) <= GRAD_RTOL


def test_varlen_bad_offsets_are_clamped_and_reported():
    """Decreasing offsets and a sequence longer than max_seqlen: every access
    stays inside the tensors (the kernels clamp each sequence to [0, T] and
    to max_seqlen) and dev_status reports ATTN_ERR_INVALID_ARG."""
    H, d = 2, 64
    T = 400
    q, k, v = (torch.randn(T, H, d, dtype=torch.bfloat16, device="cuda") for _ in range(3))
    cu = torch.tensor([0, 300, 200, 400], dtype=torch.int32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = ea.attn_fwd_varlen(q, k, v, cu, cu, 256, 256, causal=True, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1   # ATTN_ERR_INVALID_ARG
    assert torch.isfinite(o[:256].float()).all()
    do = torch.randn(T, H, d, dtype=torch.bfloat16, device="cuda")
    status2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    dq, dk, dv = ea.attn_bwd_varlen(q, k, v, o, do, lse, cu, cu, 256, 256, causal=True,
                                    dev_status=status2)
    torch.cuda.synchronize()
    assert int(status2.item()) == 1
    for g in (dq, dk, dv):
        assert torch.isfinite(g[:256].float()).all()
