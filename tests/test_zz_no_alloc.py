"""attn_bwd_noalloc: the backward with the library's built-in scratch buffer.

It exists for callers that cannot allocate device memory where they run the
backward (a plugin inside a framework that owns all device memory, or
latency-critical code that must not call cudaMalloc).  This file is named so
that pytest collects it last; it must pass on its own in a fresh process and
after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import exact_attention_58_gb300 as ea
from exact_attention_58_gb300.workloads import make_inputs
from gpu_helpers import GRAD_RTOL, grad_err

pytestmark = pytest.mark.gpu


def _call_noalloc(lib, q, k, v, o, do, lse, dq, dk, dv, inp, status):
    """Straight through the C ABI: no workspace argument at all."""
    B, H, N, d = q.shape
    Nk = k.shape[2]
    p = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    kl = None if inp.key_lens is None else ctypes.c_void_p(inp.key_lens.cuda().data_ptr())
    return lib.attn_bwd_noalloc(p(q), p(k), p(v), p(o), p(do), p(lse), p(dq), p(dk), p(dv),
                                B, H, N, Nk, d, 0, inp.scale, int(inp.causal), 0, kl, inp.dropout_p,
                                inp.seed, p(status),
                                ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("d,causal", [(128, True), (64, False)])
def test_noalloc_matches_workspace_backward_twice(d, causal):
    lib = ea.library()
    inp = make_inputs(2, 3, 300, d, gen_seed=55 + d, causal=causal, key_len_range=(200, 300),
                      dropout_p=0.1, dropout_seed_value=0x5EED0099)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    kl = inp.key_lens.cuda()
    o, lse = ea.attn_fwd(q, k, v, causal=causal, key_lens=kl, dropout_p=inp.dropout_p,
                         seed=inp.seed, scale=inp.scale)
    ref = ea.attn_bwd(q, k, v, o, do, lse, causal=causal, key_lens=kl,
                      dropout_p=inp.dropout_p, seed=inp.seed, scale=inp.scale)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    outs = [tuple(torch.full_like(q, float("nan")) for _ in range(3)) for _ in range(2)]
    torch.cuda.synchronize()
    for call in range(2):   # the buffer keeps the last call's contents: both must be right
        dq, dk, dv = outs[call]
        if call == 1:   # device memory in use, seen by the driver and by torch's allocator
            free0, _ = torch.cuda.mem_get_info()
            alloc0 = torch.cuda.memory_allocated()
        st = _call_noalloc(lib, q, k, v, o, do, lse, dq, dk, dv, inp, status)
        torch.cuda.synchronize()
        if call == 1:   # the call itself allocated nothing (kernels were loaded by call 0)
            assert torch.cuda.mem_get_info()[0] == free0
            assert torch.cuda.memory_allocated() == alloc0
        assert st == 0, ea.attn_status_string(st)
        assert int(status.item()) == 0
        for got, want, name in zip((dq, dk, dv), ref, ("dQ", "dK", "dV")):
            err = grad_err(got.double().cpu().numpy(), want.double().cpu().numpy())
            assert err <= GRAD_RTOL, (call, name, err)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = ea.library()
    fake = ctypes.c_void_p(0x10000)
    # 64 heads x 4096 rows x (2 + 128) floats = 136 MB > 32 MiB
    st = lib.attn_bwd_noalloc(*([fake] * 9), 4, 16, 4096, 4096, 128, 0, 0.088, 1, 0, None, 0.0, 0,
                              None, None)
    assert st == 4   # ATTN_ERR_WORKSPACE, before anything is enqueued
