"""Invariances of exact attention checked on the GPU's own outputs: key shift
and tile size.

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
import oracle
from exact_attention_58_gb300.workloads import make_inputs, make_packed_inputs
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


# ---------------------------------------------------------------------------
# Tile-size invariance on the GPU: the forward run with one and with two
# 128-row query tiles per CTA (GBATTN_FWD_TILES, read at each call).  The
# pages' tiled result is the full softmax whatever the tiling ("Tiling:
# fitting the work inside SRAM"): each layout must meet the tolerance against
# the oracle, and the two must agree to 1e-2.
# ---------------------------------------------------------------------------
def _with_tiles(monkeypatch, tiles, fn):
    monkeypatch.setenv("GBATTN_FWD_TILES", str(tiles))
    try:
        return fn()
    finally:
        monkeypatch.delenv("GBATTN_FWD_TILES")


@pytest.mark.parametrize("d,causal,pad,p,window", [
    (64, True, False, 0.0, 0),
    (128, True, False, 0.0, 0),
    (64, False, True, 0.1, 0),
    (128, False, True, 0.0, 0),
    (128, True, False, 0.0, 200),
    (64, False, False, 0.1, 150),
])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_one_and_two_query_tiles_per_cta_agree(monkeypatch, d, causal, pad, p, window, dtype):
    B, H, N = 2, 3, 645   # 5 tiles of 128 rows and a ragged 5-row tail: odd tile counts
    inp = make_inputs(B, H, N, d, dtype=dtype, gen_seed=900 + d + 5 * causal + 3 * pad,
                      causal=causal, key_len_range=(300, N) if pad else None, dropout_p=p,
                      dropout_seed_value=0x5EED9000 + d, with_do=False)
    inp.window = window
    q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
    kl = None if inp.key_lens is None else inp.key_lens.cuda()

    def run():
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        o, lse = ea.attn_fwd(q, k, v, causal=causal, key_lens=kl, dropout_p=p, seed=inp.seed,
                             scale=inp.scale, window=window, dev_status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == 0
        return o, lse

    o1, l1 = _with_tiles(monkeypatch, 1, run)
    o2, l2 = _with_tiles(monkeypatch, 2, run)
    O_ref, L_ref = oracle_fwd(inp)
    for o, lse in ((o1, l1), (o2, l2)):
        assert np.abs(f64(o) - O_ref).max() <= O_ATOL
        assert lse_err(f64(lse), L_ref) <= LSE_ATOL
    assert float((o1.float() - o2.float()).abs().max()) <= 1e-2
    assert lse_err(f64(l1), f64(l2)) <= 1e-2


@pytest.mark.parametrize("d", [64, 128])
def test_one_and_two_query_tiles_per_cta_agree_packed(monkeypatch, d):
    lens = [1, 300, 77, 129, 256, 0, 513]
    inp = make_packed_inputs(lens, lens, 2, d, gen_seed=950 + d, causal=True)
    q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
    cu = inp.cu_q.cuda()

    def run():
        o, lse = ea.attn_fwd_varlen(q, k, v, cu, cu, inp.max_q, inp.max_k, causal=True,
                                    scale=inp.scale)
        torch.cuda.synchronize()
        return o, lse

    o1, l1 = _with_tiles(monkeypatch, 1, run)
    o2, l2 = _with_tiles(monkeypatch, 2, run)
    O_ref, L_ref, *_ = oracle.attn_fwd_bwd_varlen(f64(inp.q), f64(inp.k), f64(inp.v),
                                                  f64(inp.do), inp.cu_q.numpy(), inp.cu_k.numpy(),
                                                  inp.scale, True, 0.0, 0)
    for o, lse in ((o1, l1), (o2, l2)):
        assert np.abs(f64(o) - O_ref).max() <= O_ATOL
        assert lse_err(f64(lse), L_ref) <= LSE_ATOL
    assert float((o1.float() - o2.float()).abs().max()) <= 1e-2
