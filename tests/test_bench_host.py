"""Host-side arithmetic of bench.py (CPU): the exact FLOP count of masked,
cross-attention and windowed problems against a brute-force count of the
attended (query, key) pairs, and the packed-sequence length draw."""
import dataclasses
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402
from exact_attention_58_gb300.workloads import workload  # noqa: E402


def _pairs_brute(N, Nk, causal, window):
    n = 0
    for i in range(N):
        t = i + Nk - N
        for j in range(Nk):
            ok = True
            if causal and j > t:
                ok = False
            if window > 0 and (t - j >= window or (not causal and j - t >= window)):
                ok = False
            n += ok
    return n


@pytest.mark.parametrize("N,Nk", [(37, 37), (20, 53), (53, 20), (1, 9), (64, 64)])
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("window", [0, 1, 5, 100])
def test_pairs_flops_match_a_brute_force_count(N, Nk, causal, window):
    w = dataclasses.replace(workload(3), B=2, H=3, N=N, d=8, causal=causal)
    flops = bench.pairs_flops_fwd(w, window, Nk)
    assert flops == 4.0 * 2 * 3 * 8 * _pairs_brute(N, Nk, causal, window)


def test_square_causal_count_is_the_halved_convention_plus_the_diagonal():
    w = workload(3)
    exact = bench.pairs_flops_fwd(w, 0, w.N)
    # N (N + 1) / 2 pairs against the N^2 / 2 of the convention
    assert exact == pytest.approx(w.flops_fwd() * (w.N + 1) / w.N)


@pytest.mark.parametrize("index", [2, 3, 5])
def test_packed_lengths_use_the_token_budget(index):
    w = workload(index)
    lens = bench.varlen_lengths(w)
    assert sum(lens) == w.B * w.N
    assert all(1 <= n <= w.N for n in lens)
    assert all(n >= max(1, w.N // 8) for n in lens[:-1])   # only the last one is cut
    assert lens == bench.varlen_lengths(w)                  # seeded
