"""Seeded synthetic workloads shared by the tests, the smoke check and the benchmark.

This module draws inputs only; it holds none of the attention arithmetic, so
both the CUDA path and the float64 oracle can be fed from it.

The five workloads stand in for the shapes the pages measure on (GPT-2 small,
BERT-large, long sequences) with iid Gaussian data; no dataset or trained
weight is used.  Recipe for workload c (1-based):
  * a CPU ``torch.Generator`` seeded with 1000 + c;
  * float32 N(0, sigma^2) drawn in the order Q, K, V, dO (Q and dO [B, H, N, d],
    K and V [B, H, Nk, d] with Nk = N unless a key length is given), then the
    per-sequence key lengths (uniform integers in [lo, hi], at most Nk);
  * Q, K, V, dO cast to the workload dtype (bf16 rounds to nearest even);
  * the dropout seed is 0x5EED0000 + c.
"""
from __future__ import annotations

import dataclasses
import itertools
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    dtype: str            # "bf16" or "fp32"
    sigma: float
    causal: bool
    key_len_range: Optional[tuple]   # (lo, hi) inclusive, or None = all keys valid
    dropout_p: float
    backward: bool

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    def flops_fwd(self) -> float:
        """4 B H N^2 d, halved for causal (the convention the metric states)."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    def flops_bwd(self) -> float:
        """Backward counted as 2.5 x the forward."""
        return 2.5 * self.flops_fwd()


WORKLOADS = [
    Workload("c1_b1h1n128d64_fp32", 1, 1, 128, 64, "fp32", 1.0, False, None, 0.0, False),
    Workload("c2_gpt2s_b8h12n1024d64_causal", 8, 12, 1024, 64, "bf16", 1.0, True, None, 0.0, True),
    Workload("c3_b4h16n4096d128_causal", 4, 16, 4096, 128, "bf16", 1.0, True, None, 0.0, True),
    Workload("c4_long_b1h16n16384d64", 1, 16, 16384, 64, "bf16", 0.5, False, None, 0.0, False),
    Workload("c5_bertl_b32h16n512d64_pad_drop", 32, 16, 512, 64, "bf16", 1.0, False, (128, 512),
             0.1, True),
]


def workload(index: int) -> Workload:
    """Workload by 1-based index."""
    return WORKLOADS[index - 1]


def dropout_seed(index: int) -> int:
    return 0x5EED0000 + index


@dataclasses.dataclass
class Inputs:
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    do: Optional[torch.Tensor]
    key_lens: Optional[torch.Tensor]   # int32 [B] or None
    scale: float
    causal: bool
    dropout_p: float
    seed: int
    window: int = 0   # > 0: sliding window of this many keys


def make_inputs(B: int, H: int, N: int, d: int, *, dtype=torch.bfloat16, sigma: float = 1.0,
                gen_seed: int = 0, causal: bool = False, key_len_range=None,
                dropout_p: float = 0.0, dropout_seed_value: int = 0, with_do: bool = True,
                scale: Optional[float] = None, Nk: Optional[int] = None) -> Inputs:
    """Draw one seeded input set on the CPU (see the module docstring for the
    order).  ``Nk`` (default N) keys: cross-attention when it differs from N."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(gen_seed))
    shape = (B, H, N, d)
    Nk = N if Nk is None else int(Nk)
    kshape = (B, H, Nk, d)
    q = (torch.randn(shape, generator=g, dtype=torch.float32) * sigma).to(dtype)
    k = (torch.randn(kshape, generator=g, dtype=torch.float32) * sigma).to(dtype)
    v = (torch.randn(kshape, generator=g, dtype=torch.float32) * sigma).to(dtype)
    do = (torch.randn(shape, generator=g, dtype=torch.float32)).to(dtype) if with_do else None
    kl = None
    if key_len_range is not None:
        lo, hi = key_len_range
        kl = torch.randint(int(lo), int(hi) + 1, (B,), generator=g, dtype=torch.int64)
        kl = kl.clamp(max=Nk).to(torch.int32)
    return Inputs(q, k, v, do, kl, (1.0 / math.sqrt(d)) if scale is None else float(scale),
                  causal, float(dropout_p), int(dropout_seed_value))


def make_workload_inputs(index: int, B: Optional[int] = None, H: Optional[int] = None,
                         N: Optional[int] = None, Nk: Optional[int] = None,
                         d: Optional[int] = None) -> Inputs:
    """Inputs of workload ``index`` (1-based), optionally with B/H/N cut down,
    with ``Nk`` keys (cross-attention) instead of N, or another head dim."""
    w = workload(index)
    return make_inputs(B or w.B, H or w.H, N or w.N, d or w.d, dtype=w.torch_dtype, sigma=w.sigma,
                       gen_seed=1000 + index, causal=w.causal, key_len_range=w.key_len_range,
                       dropout_p=w.dropout_p, dropout_seed_value=dropout_seed(index),
                       with_do=w.backward, Nk=Nk)


@dataclasses.dataclass
class PackedInputs:
    q: torch.Tensor           # [total_q, H, d]
    k: torch.Tensor           # [total_k, H, d]
    v: torch.Tensor
    do: torch.Tensor          # [total_q, H, d]
    cu_q: torch.Tensor        # int32 [B + 1]
    cu_k: torch.Tensor
    max_q: int
    max_k: int
    scale: float
    causal: bool
    dropout_p: float
    seed: int
    window: int = 0


def make_packed_inputs(lens_q, lens_k, H: int, d: int, *, dtype=torch.bfloat16,
                       sigma: float = 1.0, gen_seed: int = 0, causal: bool = False,
                       dropout_p: float = 0.0, dropout_seed_value: int = 0,
                       window: int = 0) -> PackedInputs:
    """Packed variable-length sequences: sequence b has lens_q[b] queries and
    lens_k[b] keys.  Drawn in the order Q, K, V, dO as float32 N(0, sigma^2)
    (dO unit variance) on a CPU generator seeded with ``gen_seed``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(gen_seed))
    tq, tk = int(sum(lens_q)), int(sum(lens_k))
    q = (torch.randn((tq, H, d), generator=g, dtype=torch.float32) * sigma).to(dtype)
    k = (torch.randn((tk, H, d), generator=g, dtype=torch.float32) * sigma).to(dtype)
    v = (torch.randn((tk, H, d), generator=g, dtype=torch.float32) * sigma).to(dtype)
    do = torch.randn((tq, H, d), generator=g, dtype=torch.float32).to(dtype)
    cu = lambda lens: torch.tensor([0] + list(itertools.accumulate(int(x) for x in lens)),  # noqa: E731
                                   dtype=torch.int32)
    return PackedInputs(q, k, v, do, cu(lens_q), cu(lens_k), max(1, max(lens_q)),
                        max(1, max(lens_k)), 1.0 / math.sqrt(d), causal, float(dropout_p),
                        int(dropout_seed_value), int(window))
