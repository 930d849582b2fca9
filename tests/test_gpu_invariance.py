"""Key-shift invariance of exact attention, checked on the GPU's own outputs.

Adding one vector c to every key adds scale * (q_i . c) to every score of
row i, so each softmax row is unchanged ("Why FlashAttention Is a Kernel
Story", section "Tiling: fitting the work inside SRAM": the tiled result is
the full softmax, and a softmax row depends on its scores only up to a common
shift).  Hence O, dV and dK (built from P and dS) are unchanged, dQ is
unchanged because sum_j dS_ij = 0 cancels scale * sum_j dS_ij c, and the
log-sum-exp of row i moves by exactly scale * (q_i . c).

Inputs are put on a 1/16 grid in [-4, 4] so that K + c is exactly
representable in bf16 and both launches see exact inputs.
"""
import numpy as np
import pytest
import torch

import exact_attention_58_gb300 as ea
from exact_attention_58_gb300.workloads import make_inputs
from gpu_helpers import GRAD_RTOL, LSE_ATOL, O_ATOL, f64, grad_err, lse_err, oracle_bwd, oracle_fwd

pytestmark = pytest.mark.gpu


def _grid(t):
    return (t.float() * 16).round().clamp(-64, 64).div(16).to(t.dtype)


def _run(inp, q, k, v, do, kl):
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    o, lse = ea.attn_fwd(q, k, v, causal=inp.causal, key_lens=kl, dropout_p=inp.dropout_p,
                         seed=inp.seed, scale=inp.scale, dev_status=st)
    dq, dk, dv = ea.attn_bwd(q, k, v, o, do, lse, causal=inp.causal, key_lens=kl,
                             dropout_p=inp.dropout_p, seed=inp.seed, scale=inp.scale,
                             dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return o, lse, dq, dk, dv


@pytest.mark.parametrize("d,causal,pad,p", [
    (64, False, False, 0.0),
    (128, True, False, 0.0),
    (64, True, True, 0.1),
    (128, False, True, 0.2),
])
def test_key_shift_leaves_o_and_gradients_and_moves_lse(d, causal, pad, p):
    B, H, N = 2, 2, 333   # several 128-row tiles and a ragged tail
    inp = make_inputs(B, H, N, d, gen_seed=700 + d + 7 * causal + 3 * pad, causal=causal,
                      key_len_range=(150, N) if pad else None, dropout_p=p,
                      dropout_seed_value=0x5EED7000 + d)
    inp.q, inp.k, inp.v = _grid(inp.q), _grid(inp.k), _grid(inp.v)
    g = torch.Generator().manual_seed(9)
    c = (torch.randint(-32, 33, (B, H, 1, d), generator=g).float() / 16)   # exact shift in bf16
    k2 = (inp.k.float() + c).to(inp.k.dtype)
    assert torch.equal(k2.float(), inp.k.float() + c), "the shifted keys must be exact"
    dev = lambda t: t.cuda()  # noqa: E731
    kl = None if inp.key_lens is None else dev(inp.key_lens)
    r1 = _run(inp, dev(inp.q), dev(inp.k), dev(inp.v), dev(inp.do), kl)
    r2 = _run(inp, dev(inp.q), dev(k2), dev(inp.v), dev(inp.do), kl)
    # both launches against the oracle of the unshifted keys (O and the gradients
    # are invariant)
    O_ref, L_ref = oracle_fwd(inp)
    dQ_ref, dK_ref, dV_ref, _ = oracle_bwd(inp)
    for o, lse, dq, dk, dv in (r1, r2):
        assert np.abs(f64(o) - O_ref).max() <= O_ATOL
        for g_, ref in ((dq, dQ_ref), (dk, dK_ref), (dv, dV_ref)):
            assert grad_err(f64(g_), ref) <= GRAD_RTOL
    # the invariance between the two GPU results
    o1, l1, dq1, dk1, dv1 = r1
    o2, l2, dq2, dk2, dv2 = r2
    assert float((o1.float() - o2.float()).abs().max()) <= O_ATOL
    shift = inp.scale * torch.einsum("bhnd,bhd->bhn", inp.q.double(), c[:, :, 0].double())
    lse_shifted = f64(l1) + shift.numpy()
    assert lse_err(f64(l2), lse_shifted) <= 2 * LSE_ATOL
    assert lse_err(f64(l2), L_ref + shift.numpy()) <= LSE_ATOL
    for a, b_ in ((dq1, dq2), (dk1, dk2), (dv1, dv2)):
        assert grad_err(f64(b_), f64(a)) <= GRAD_RTOL
