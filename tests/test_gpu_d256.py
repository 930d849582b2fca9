"""Head dimension 256 (forward, bf16 and fp16): parity against the float64
oracle.  One 128-row query tile per CTA (its fp32 O takes 256 tensor-memory
columns), tiles of 512-byte rows in four 128-byte swizzled column blocks, and
the P V product as one N = 256 MMA per 16 keys."""
import numpy as np
import pytest
import torch

import exact_attention_58_gb300 as ea
import oracle
from exact_attention_58_gb300.workloads import make_inputs, make_packed_inputs
from gpu_helpers import LSE_ATOL, O_ATOL, f64, gpu_fwd, lse_err, oracle_fwd

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


def test_d256_backward_is_refused():
    inp = make_inputs(1, 1, 128, 256, gen_seed=15)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    o, lse = ea.attn_fwd(q, k, v)
    with pytest.raises(ea.AttnError):
        ea.attn_bwd(q, k, v, o, do, lse)


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
