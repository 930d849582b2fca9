"""Guard bands: every output is a view into a larger buffer whose margins are
filled with a sentinel, and no kernel writes outside its output (ragged
lengths, causal and windowed masks, cross-attention, packed sequences, the
backward's row-by-row tail stores)."""
import pytest
import torch

import exact_attention_58_gb300 as ea
from exact_attention_58_gb300.workloads import make_inputs, make_packed_inputs

pytestmark = pytest.mark.gpu

GUARD = 4096          # elements on each side (a multiple of 8: keeps 16-byte alignment)
SENTINEL = 0x7FC1     # a NaN bf16 bit pattern no kernel writes


def _guarded(shape, dtype):
    n = 1
    for s in shape:
        n *= s
    buf = torch.full((n + 2 * GUARD,), SENTINEL, dtype=torch.int16, device="cuda")
    view = buf[GUARD:GUARD + n].view(dtype).view(shape)
    return buf, view


def _intact(buf, n):
    return bool((buf[:GUARD] == SENTINEL).all()) and bool((buf[GUARD + n:] == SENTINEL).all())


def _lse_guarded(shape):
    n = 1
    for s in shape:
        n *= s
    buf = torch.full((n + 2 * GUARD,), float("nan"), dtype=torch.float32, device="cuda")
    return buf, buf[GUARD:GUARD + n].view(shape)


@pytest.mark.parametrize("N,Nk,causal,window", [(130, 130, True, 0), (300, 77, True, 0),
                                                (77, 300, False, 50), (1, 513, True, 0)])
def test_dense_outputs_stay_inside(N, Nk, causal, window):
    inp = make_inputs(2, 3, N, 64, gen_seed=N + Nk, causal=causal, Nk=Nk)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    bo, o = _guarded(q.shape, q.dtype)
    bl, lse = _lse_guarded(q.shape[:3])
    ea.attn_fwd(q, k, v, causal=causal, window=window, out=o, lse=lse)
    bq, dq = _guarded(q.shape, q.dtype)
    bk, dk = _guarded(k.shape, k.dtype)
    bv, dv = _guarded(k.shape, k.dtype)
    ea.attn_bwd(q, k, v, o, do, lse, causal=causal, window=window, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    for buf, t in ((bo, o), (bq, dq), (bk, dk), (bv, dv)):
        assert _intact(buf, t.numel())
    assert bool(torch.isnan(bl[:GUARD]).all()) and bool(torch.isnan(bl[GUARD + lse.numel():]).all())


def test_packed_outputs_stay_inside():
    lens_q, lens_k = [200, 1, 129, 60], [260, 7, 129, 300]
    inp = make_packed_inputs(lens_q, lens_k, 2, 128, gen_seed=5, causal=True)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    cq, ck = inp.cu_q.cuda(), inp.cu_k.cuda()
    bo, o = _guarded(q.shape, q.dtype)
    o2, lse = ea.attn_fwd_varlen(q, k, v, cq, ck, inp.max_q, inp.max_k, causal=True, out=o)
    bq, dq = _guarded(q.shape, q.dtype)
    bk, dk = _guarded(k.shape, k.dtype)
    bv, dv = _guarded(k.shape, k.dtype)
    ea.attn_bwd_varlen(q, k, v, o, do, lse, cq, ck, inp.max_q, inp.max_k, causal=True, dq=dq,
                       dk=dk, dv=dv)
    torch.cuda.synchronize()
    for buf, t in ((bo, o), (bq, dq), (bk, dk), (bv, dv)):
        assert _intact(buf, t.numel())
