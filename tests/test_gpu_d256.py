"""Head dimension 256 (bf16 and fp16): parity against the float64 oracle.

Forward: one 128-row query tile per CTA (its fp32 O takes 256 tensor-memory
columns), tiles of 512-byte rows in four 128-byte swizzled column blocks, and
the P V product as one N = 256 MMA per 16 keys.  Backward: one CTA per (head,
128-key block, half of d) walking 64-row query blocks, S and dP recomputed
over the whole head dim in each half."""
import numpy as np
import pytest
import torch

import exact_attention_58_gb300 as ea
import oracle
from exact_attention_58_gb300.workloads import make_inputs, make_packed_inputs
from gpu_helpers import (GRAD_RTOL, LSE_ATOL, O_ATOL, f64, gpu_fwd, gpu_fwd_bwd, grad_err, lse_err,
                         oracle_bwd, oracle_fwd)

pytestmark = pytest.mark.gpu


def _check(inp):
    o, lse = gpu_fwd(inp)
    O_ref, L_ref = oracle_fwd(inp)
    assert float(np.abs(f64(o) - O_ref).max()) <= O_ATOL
    assert lse_err(f64(lse), L_ref) <= LSE_ATOL


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N", [1, 128, 300, 700])
def test_d256_shapes(causal, N):
    _check(make_inputs(2, 2, N, 256, gen_seed=256 + N + causal, causal=causal, with_do=False))


@pytest.mark.parametrize("causal", [True, False])
def test_d256_padding_dropout_window(causal):
    inp = make_inputs(3, 2, 500, 256, gen_seed=41 + causal, causal=causal, key_len_range=(100, 500),
                      dropout_p=0.15, dropout_seed_value=0x5EED0256, with_do=False)
    inp.window = 200
    _check(inp)


def test_d256_fp16():
    _check(make_inputs(2, 2, 333, 256, dtype=torch.float16, gen_seed=12, causal=True,
                       with_do=False))


def test_d256_cross_attention():
    inp = make_inputs(2, 2, 200, 256, gen_seed=13, causal=True, Nk=640)
    q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
    o, lse = ea.attn_fwd(q, k, v, causal=True, scale=inp.scale)
    O_ref, L_ref, _, _, _ = oracle.attn_fwd_bwd_qk(f64(inp.q), f64(inp.k), f64(inp.v),
                                                   f64(inp.do), inp.scale, True)
    assert float(np.abs(f64(o) - O_ref).max()) <= O_ATOL
    assert lse_err(f64(lse), L_ref) <= LSE_ATOL


def test_d256_packed():
    inp = make_packed_inputs([130, 7, 400], [130, 7, 400], 2, 256, gen_seed=14, causal=True)
    q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
    cu = inp.cu_q.cuda()
    o, lse = ea.attn_fwd_varlen(q, k, v, cu, cu, inp.max_q, inp.max_k, causal=True,
                                scale=inp.scale)
    O_ref, L_ref, _, _, _ = oracle.attn_fwd_bwd_varlen(f64(inp.q), f64(inp.k), f64(inp.v),
                                                       f64(inp.do), inp.cu_q.numpy(),
                                                       inp.cu_k.numpy(), inp.scale, True)
    assert float(np.abs(f64(o) - O_ref).max()) <= O_ATOL
    assert lse_err(f64(lse), L_ref) <= LSE_ATOL


def test_d256_full_size_sampled_heads():
    """B = 4, H = 16, N = 4096, d = 256, causal: the full-size launch, the
    oracle on two heads."""
    inp = make_inputs(4, 16, 4096, 256, gen_seed=2560, causal=True, with_do=False)
    o, lse = gpu_fwd(inp)
    heads = [(0, 3), (3, 12)]
    sel = lambda t: np.stack([f64(t[b, h]) for b, h in heads])  # noqa: E731
    O_ref, L_ref = oracle.heads_fwd(sel(inp.q), sel(inp.k), sel(inp.v),
                                    np.array([b for b, _ in heads], np.int32),
                                    np.array([h for _, h in heads], np.int32),
                                    np.full(2, 4096, np.int32), inp.scale, True)
    assert float(np.abs(sel(o) - O_ref).max()) <= O_ATOL
    assert lse_err(sel(lse), L_ref) <= LSE_ATOL



# ---------------------------------------------------------------------------
# backward
# ---------------------------------------------------------------------------
def _check_bwd(inp):
    o, lse, dq, dk, dv = gpu_fwd_bwd(inp)
    O_ref, L_ref = oracle_fwd(inp)
    assert float(np.abs(f64(o) - O_ref).max()) <= O_ATOL
    dQ, dK, dV, _ = oracle_bwd(inp)
    errs = {"dQ": grad_err(f64(dq), dQ), "dK": grad_err(f64(dk), dK), "dV": grad_err(f64(dv), dV)}
    for n in errs:
        assert errs[n] <= GRAD_RTOL, errs


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("N", [1, 64, 128, 333, 700])
def test_d256_backward_shapes(causal, N):
    _check_bwd(make_inputs(2, 2, N, 256, gen_seed=2560 + N + causal, causal=causal))


@pytest.mark.parametrize("causal", [True, False])
def test_d256_backward_padding_dropout_window(causal):
    inp = make_inputs(3, 2, 500, 256, gen_seed=43 + causal, causal=causal, key_len_range=(100, 500),
                      dropout_p=0.15, dropout_seed_value=0x5EED1256)
    inp.window = 200
    _check_bwd(inp)


@pytest.mark.parametrize("causal", [True, False])
def test_d256_backward_padding_dropout(causal):
    inp = make_inputs(2, 3, 400, 256, gen_seed=47 + causal, causal=causal, key_len_range=(0, 400),
                      dropout_p=0.1, dropout_seed_value=0x5EED2256)
    _check_bwd(inp)


def test_d256_backward_fp16():
    _check_bwd(make_inputs(2, 2, 333, 256, dtype=torch.float16, gen_seed=15, causal=True))


@pytest.mark.parametrize("causal", [True, False])
def test_d256_backward_cross_attention(causal):
    inp = make_inputs(2, 2, 200, 256, gen_seed=16 + causal, causal=causal, Nk=640)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = ea.attn_fwd(q, k, v, causal=causal, scale=inp.scale, dev_status=st)
    dq, dk, dv = ea.attn_bwd(q, k, v, o, do, lse, causal=causal, scale=inp.scale, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O_ref, L_ref, dQ, dK, dV = oracle.attn_fwd_bwd_qk(f64(inp.q), f64(inp.k), f64(inp.v),
                                                      f64(inp.do), inp.scale, causal)
    assert float(np.abs(f64(o) - O_ref).max()) <= O_ATOL
    for g, ref in ((dq, dQ), (dk, dK), (dv, dV)):
        assert grad_err(f64(g), ref) <= GRAD_RTOL


def test_d256_backward_packed():
    lens = [130, 7, 0, 400, 65]
    inp = make_packed_inputs(lens, lens, 2, 256, gen_seed=17, causal=True, dropout_p=0.1,
                             dropout_seed_value=0x5EED3256)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    cu = inp.cu_q.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    kw = dict(causal=True, dropout_p=inp.dropout_p, seed=inp.seed, scale=inp.scale, dev_status=st)
    o, lse = ea.attn_fwd_varlen(q, k, v, cu, cu, inp.max_q, inp.max_k, **kw)
    dq, dk, dv = ea.attn_bwd_varlen(q, k, v, o, do, lse, cu, cu, inp.max_q, inp.max_k, **kw)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    O_ref, L_ref, dQ, dK, dV = oracle.attn_fwd_bwd_varlen(f64(inp.q), f64(inp.k), f64(inp.v),
                                                          f64(inp.do), inp.cu_q.numpy(),
                                                          inp.cu_k.numpy(), inp.scale, True,
                                                          inp.dropout_p, inp.seed)
    assert float(np.abs(f64(o) - O_ref).max()) <= O_ATOL
    for g, ref in ((dq, dQ), (dk, dK), (dv, dV)):
        assert grad_err(f64(g), ref) <= GRAD_RTOL


def test_d256_backward_noalloc_and_guard_bands():
    """The backward writes nothing outside dQ, dK, dV (bands of NaN around
    each output stay NaN), and attn_bwd_noalloc gives the same result."""
    inp = make_inputs(1, 2, 300, 256, gen_seed=18, causal=True)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    o, lse = ea.attn_fwd(q, k, v, causal=True, scale=inp.scale)
    n = q.numel()
    bufs = [torch.full((n + 2 * 4096,), float("nan"), dtype=q.dtype, device="cuda") for _ in range(3)]
    views = [b[4096:4096 + n].view(q.shape) for b in bufs]
    ea.attn_bwd(q, k, v, o, do, lse, causal=True, scale=inp.scale, dq=views[0], dk=views[1],
                dv=views[2])
    torch.cuda.synchronize()
    for b in bufs:
        assert torch.isnan(b[:4096].float()).all() and torch.isnan(b[4096 + n:].float()).all()
    ref = ea.attn_bwd_noalloc(q, k, v, o, do, lse, causal=True, scale=inp.scale)
    torch.cuda.synchronize()
    dQ, dK, dV, _ = oracle_bwd(inp)
    for g, r in zip(views, (dQ, dK, dV)):
        assert grad_err(f64(g), r) <= GRAD_RTOL
    for g, r in zip(ref, (dQ, dK, dV)):
        assert grad_err(f64(g), r) <= GRAD_RTOL
