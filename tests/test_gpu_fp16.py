"""fp16 (IEEE half) storage: forward and backward parity against the float64
oracle, on the same seeded inputs as the bf16 tests but rounded to half."""
import numpy as np
import pytest
import torch

from exact_attention_58_gb300.workloads import make_inputs
from gpu_helpers import (GRAD_RTOL, LSE_ATOL, O_ATOL, f64, gpu_fwd, gpu_fwd_bwd, grad_err,
                         oracle_bwd, oracle_fwd)

pytestmark = pytest.mark.gpu


def _check(inp, backward=True):
    if backward:
        o, lse, dq, dk, dv = gpu_fwd_bwd(inp)
    else:
        o, lse = gpu_fwd(inp)
    assert o.dtype == torch.float16
    O_ref, L_ref = oracle_fwd(inp)
    err_o = float(np.abs(f64(o) - O_ref).max())
    fin = np.isfinite(L_ref)
    err_l = float(np.abs(f64(lse)[fin] - L_ref[fin]).max()) if fin.any() else 0.0
    assert err_o <= O_ATOL, err_o
    assert err_l <= LSE_ATOL, err_l
    if backward:
        dQ, dK, dV, _ = oracle_bwd(inp)
        errs = {"dQ": grad_err(f64(dq), dQ), "dK": grad_err(f64(dk), dK), "dV": grad_err(f64(dv), dV)}
        for n in errs:
            assert errs[n] <= GRAD_RTOL, errs


@pytest.mark.parametrize("B,H,N,d", [(1, 2, 256, 64), (2, 1, 300, 128), (1, 1, 130, 64),
                                     (1, 1, 1, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp16_shapes(B, H, N, d, causal):
    _check(make_inputs(B, H, N, d, dtype=torch.float16, gen_seed=5 * N + d + causal,
                       causal=causal))


@pytest.mark.parametrize("d", [64, 128])
def test_fp16_padding_dropout(d):
    inp = make_inputs(3, 2, 260, d, dtype=torch.float16, gen_seed=77 + d, causal=True,
                      key_len_range=(1, 260), dropout_p=0.2, dropout_seed_value=0x5EED0042)
    _check(inp)


def test_fp16_long_forward():
    """A longer non-causal forward (several key blocks per CTA) at d = 64."""
    _check(make_inputs(1, 4, 1024, 64, dtype=torch.float16, gen_seed=9, sigma=0.5),
           backward=False)
