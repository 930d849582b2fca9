"""Backward parity: dQ, dK, dV from the CUDA path against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
from exact_attention_58_gb300.workloads import make_inputs, make_workload_inputs, workload
from gpu_helpers import (GRAD_RTOL, O_ATOL, f64, gpu_fwd_bwd, grad_err, oracle_bwd,
                         oracle_fwd)

pytestmark = pytest.mark.gpu


def _check(inp):
    o, lse, dq, dk, dv = gpu_fwd_bwd(inp)
    O_ref, _ = oracle_fwd(inp)
    dQ, dK, dV, _ = oracle_bwd(inp)
    errs = {"O": float(np.abs(f64(o) - O_ref).max()), "dQ": grad_err(f64(dq), dQ),
            "dK": grad_err(f64(dk), dK), "dV": grad_err(f64(dv), dV)}
    assert errs["O"] <= O_ATOL, errs
    for n in ("dQ", "dK", "dV"):
        assert errs[n] <= GRAD_RTOL, errs
    return errs


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 128, 64), (2, 3, 130, 64), (1, 2, 300, 128),
                                     (1, 1, 1, 64), (2, 1, 7, 128), (1, 1, 513, 64),
                                     (1, 2, 256, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_shapes(B, H, N, d, causal):
    _check(make_inputs(B, H, N, d, gen_seed=3 * N + d + causal, causal=causal))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_key_padding(d, causal):
    inp = make_inputs(4, 2, 300, d, gen_seed=17 + d, causal=causal)
    inp.key_lens = torch.tensor([0, 1, 129, 300], dtype=torch.int32)
    _check(inp)


@pytest.mark.parametrize("p", [0.1, 0.5])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_dropout(p, d, causal):
    inp = make_inputs(2, 2, 260, d, gen_seed=41, causal=causal, key_len_range=(130, 260),
                      dropout_p=p, dropout_seed_value=0x5EED0005)
    _check(inp)


@pytest.mark.parametrize("p", [1e-6, 0.9])
@pytest.mark.parametrize("d", [64, 128])
def test_dropout_extreme_p(p, d):
    """p below 2^-16 (threshold 0: nothing dropped, kept values still scaled
    by 1/(1-p)) and p = 0.9 (nine scores in ten dropped), with key lengths
    that end inside a group of eight keys (one Philox block).  Not causal:
    the first causal rows attend one key, whose kept value is scaled tenfold,
    beyond what the bf16 rounding of O allows for under the O tolerance."""
    inp = make_inputs(2, 2, 203, d, gen_seed=43 + d, causal=False, key_len_range=(61, 203),
                      dropout_p=p, dropout_seed_value=0x5EED0011)
    _check(inp)


def _sampled_heads_check(index, heads):
    inp = make_workload_inputs(index)
    w = workload(index)
    o, lse, dq, dk, dv = gpu_fwd_bwd(inp)
    b_idx = np.array([b for b, _ in heads], dtype=np.int32)
    h_idx = np.array([h for _, h in heads], dtype=np.int32)
    sel = lambda t: np.stack([f64(t[b, h]) for b, h in heads])  # noqa: E731
    kl = np.array([w.N if inp.key_lens is None else int(inp.key_lens[b]) for b, _ in heads],
                  dtype=np.int32)
    dQ, dK, dV, _ = oracle.heads_bwd(sel(inp.q), sel(inp.k), sel(inp.v), sel(inp.do), b_idx,
                                     h_idx, kl, inp.scale, inp.causal, inp.dropout_p, inp.seed)
    errs = {n: max(grad_err(sel(g)[x], ref[x]) for x in range(len(heads)))
            for n, g, ref in (("dQ", dq, dQ), ("dK", dk, dK), ("dV", dv, dV))}
    for n in errs:
        assert errs[n] <= GRAD_RTOL, errs
    # a property that holds at any size: sum_j dK_j = 0 per head (rows of dS sum to 0)
    dk_sum = dk.float().sum(dim=2).abs().max().item()
    assert dk_sum <= 0.05 * dk.float().abs().max().item() * np.sqrt(w.N), dk_sum
    return errs


def test_workload2_full_size_sampled_heads():
    """GPT-2-small shape, causal, full size; oracle backward on three heads."""
    _sampled_heads_check(2, [(0, 0), (7, 11), (3, 5)])


def test_workload5_full_size_sampled_heads():
    """BERT-large shape with key padding and dropout, full size."""
    _sampled_heads_check(5, [(0, 0), (31, 15), (12, 7)])


@pytest.mark.slow
def test_workload3_full_size_sampled_heads():
    """Headline shape (N = 4096, d = 128, causal), full size; two heads."""
    _sampled_heads_check(3, [(0, 0), (3, 15)])


def test_stage_entry_points_equal_attn_bwd():
    """attn_bwd_preprocess + attn_bwd_main + attn_bwd_dq_convert == attn_bwd."""
    import exact_attention_58_gb300 as ea
    inp = make_inputs(2, 2, 200, 64, gen_seed=8, causal=True)
    q, k, v, do = (t.cuda() for t in (inp.q, inp.k, inp.v, inp.do))
    o, lse = ea.attn_fwd(q, k, v, causal=True)
    dq1, dk1, dv1 = ea.attn_bwd(q, k, v, o, do, lse, causal=True)
    ws = torch.empty(ea.attn_bwd_workspace_size(2, 2, 200, 64), dtype=torch.uint8, device="cuda")
    dq2, dk2, dv2 = (torch.empty_like(q) for _ in range(3))
    ea.attn_bwd_preprocess(o, do, lse, ws)
    ea.attn_bwd_main(q, k, v, do, dk2, dv2, ws, causal=True)
    ea.attn_bwd_dq_convert(dq2, ws)
    torch.cuda.synchronize()
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert (dq1.float() - dq2.float()).abs().max().item() <= 1e-2  # atomic order may differ
