"""Forward parity: the CUDA path (through the C ABI) against the float64 oracle."""
import numpy as np
import pytest
import torch

from exact_attention_58_gb300.workloads import make_inputs, make_workload_inputs, workload
from gpu_helpers import (LSE_ATOL, O_ATOL, gpu_fwd, lse_err, oracle_fwd, sample_rows_check)

pytestmark = pytest.mark.gpu


def _check(inp):
    o, lse = gpu_fwd(inp)
    O_ref, L_ref = oracle_fwd(inp)
    err_o = float(np.abs(o.double().cpu().numpy() - O_ref).max())
    err_l = lse_err(lse.cpu().numpy(), L_ref)
    assert err_o <= O_ATOL, f"max|O - O_ref| = {err_o}"
    assert err_l <= LSE_ATOL, f"max|LSE - LSE_ref| = {err_l}"
    return err_o, err_l


def test_workload1_fp32_tf32():
    """B=1, H=1, N=128, d=64, fp32 inputs, non-causal (TF32 products)."""
    _check(make_workload_inputs(1))


@pytest.mark.parametrize("B,H,N,d", [(1, 1, 128, 64), (2, 3, 130, 64), (1, 2, 300, 128),
                                     (1, 1, 1, 64), (1, 1, 1, 128), (2, 1, 7, 64),
                                     (1, 2, 256, 128), (1, 1, 513, 64)])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_shapes(B, H, N, d, causal):
    _check(make_inputs(B, H, N, d, gen_seed=N * 7 + d + causal, causal=causal, with_do=False))


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_key_padding(d, causal):
    inp = make_inputs(4, 2, 257, d, gen_seed=11 + d, causal=causal, with_do=False)
    inp.key_lens = torch.tensor([1, 128, 200, 257], dtype=torch.int32)
    _check(inp)


def test_fully_masked_rows():
    """key_len = 0: O = 0 and LSE = -inf for every row of that sequence."""
    inp = make_inputs(2, 2, 140, 64, gen_seed=5, with_do=False)
    inp.key_lens = torch.tensor([0, 140], dtype=torch.int32)
    o, lse = gpu_fwd(inp)
    assert torch.all(o[0] == 0)
    assert torch.all(torch.isneginf(lse[0]))
    _check(inp)


@pytest.mark.parametrize("p", [0.1, 0.5])
@pytest.mark.parametrize("d", [64, 128])
def test_dropout(p, d):
    inp = make_inputs(2, 2, 200, d, gen_seed=21, causal=False, key_len_range=(100, 200),
                      dropout_p=p, dropout_seed_value=0x5EED0005, with_do=False)
    _check(inp)


def test_dropout_fp32():
    inp = make_inputs(1, 2, 128, 64, dtype=torch.float32, gen_seed=3, dropout_p=0.2,
                      dropout_seed_value=77, with_do=False)
    _check(inp)


def test_dropout_mask_bit_exact():
    """Read the fused kernel's own keep mask: with Q = 0 every valid score is
    equal, so O_i = sum_j Z_ij V_j / ((1-p) #valid); with V_j one-hot on
    column j - 64 kb for the keys of block kb (zero elsewhere), output column c
    of row i is nonzero iff Z[i, 64 kb + c] = 1.  Compared bit for bit with the
    oracle's Philox mask."""
    import oracle
    B, H, N, d, p, seed = 2, 2, 320, 64, 0.3, 0x5EED0005
    kl = torch.tensor([320, 250], dtype=torch.int32)
    q = torch.zeros(B, H, N, d, dtype=torch.bfloat16, device="cuda")
    k = torch.randn(B, H, N, d, generator=torch.Generator().manual_seed(1)).to(torch.bfloat16).cuda()
    import exact_attention_58_gb300 as ea
    got = np.zeros((B, H, N, N), dtype=np.uint8)
    for kb in range((N + d - 1) // d):
        v = torch.zeros(B, H, N, d, dtype=torch.bfloat16)
        for c in range(d):
            j = kb * d + c
            if j < N:
                v[:, :, j, c] = 1.0
        o, _ = ea.attn_fwd(q, k, v.cuda(), key_lens=kl.cuda(), dropout_p=p, seed=seed)
        torch.cuda.synchronize()
        nz = (o.float().cpu().numpy() != 0)
        cols = min(d, N - kb * d)
        got[:, :, :, kb * d: kb * d + cols] = nz[:, :, :, :cols]
    for b in range(B):
        for h in range(H):
            Z = oracle.dropout_mask(seed, b, h, N, N, p)
            L = int(kl[b])
            assert np.array_equal(got[b, h, :, :L], Z[:, :L]), f"mask differs at b={b} h={h}"
            assert not got[b, h, :, L:].any()


@pytest.mark.parametrize("index", [2, 3, 4])
def test_full_size_workload_sampled(index):
    """Full-size workloads 2-4 in the benchmark's launch configuration, checked
    on sampled heads and rows against the row-at-a-time oracle."""
    inp = make_workload_inputs(index)
    w = workload(index)
    o, lse = gpu_fwd(inp)
    rng = np.random.default_rng(index)
    heads = [(0, 0), (w.B - 1, w.H - 1), (int(rng.integers(w.B)), int(rng.integers(w.H)))]
    rows = np.unique(np.concatenate([[0, 1, 127, 128, 255, 256, w.N - 1],
                                     rng.integers(0, w.N, 25)])).astype(np.int32)
    err_o, err_l = sample_rows_check(inp, o, lse, heads, rows)
    assert err_o <= O_ATOL and err_l <= LSE_ATOL, (err_o, err_l)


def test_workload5_forward_sampled():
    """BERT-large shape with key padding and dropout (full size), sampled."""
    inp = make_workload_inputs(5)
    o, lse = gpu_fwd(inp)
    heads = [(0, 0), (31, 15), (7, 3)]
    rows = np.array([0, 5, 100, 255, 256, 400, 511], dtype=np.int32)
    err_o, err_l = sample_rows_check(inp, o, lse, heads, rows)
    assert err_o <= O_ATOL and err_l <= LSE_ATOL, (err_o, err_l)


def test_invalid_key_len_reported_on_device():
    inp = make_inputs(2, 1, 130, 64, gen_seed=2, with_do=False)
    inp.key_lens = torch.tensor([500, -3], dtype=torch.int32)
    import exact_attention_58_gb300 as ea
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    ea.attn_fwd(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), key_lens=inp.key_lens.cuda(),
                dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 1   # ATTN_ERR_INVALID_ARG


def test_no_nxn_buffer_long_sequence():
    """Workload 4 (N = 16384): peak device memory beyond inputs and outputs stays
    far below one N x N bf16 matrix per head (537 MB)."""
    inp = make_workload_inputs(4)
    q, k, v = (t.cuda() for t in (inp.q, inp.k, inp.v))
    import exact_attention_58_gb300 as ea
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    ea.attn_fwd(q, k, v, out=o, lse=lse)
    torch.cuda.synchronize()
    extra = torch.cuda.max_memory_allocated() - base
    assert extra < 64 * 2**20, extra


@pytest.mark.parametrize("chunk", [1, 2, 3])
@pytest.mark.parametrize("d,causal", [(64, False), (128, True)])
def test_spiky_keys_move_the_row_max(chunk, d, causal):
    """Keys of one 32-key chunk of every 128-key block scaled up six-fold, so
    that a row's maximum jumps by far more than the lazy-rescale threshold
    from one block to the next (the rescale of O and l) and varies strongly
    inside a block."""
    inp = make_inputs(2, 2, 520, d, gen_seed=7000 + 10 * chunk + d, causal=causal, with_do=False)
    j = np.arange(inp.k.shape[2])
    spike = torch.from_numpy(((j % 128) // 32) == chunk)
    k = inp.k.float()
    k[:, :, spike] *= 6.0
    inp.k = k.to(inp.q.dtype)
    _check(inp)
