"""The float64 oracle against its pins (CPU only)."""
import math
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from oracle_pins import PINS, pin_philox_vs_triton


@pytest.mark.parametrize("name", sorted(PINS))
def test_pin(name):
    fn, bound = PINS[name]
    err = fn(oracle.lib())
    assert err <= bound, f"{name}: {err} > {bound}"


def test_philox_matches_triton():
    pytest.importorskip("triton")
    bad = pin_philox_vs_triton(oracle.lib())
    if math.isnan(bad):
        pytest.skip("Triton's CPU interpreter is not usable here")
    assert bad == 0


def test_fully_masked_rows():
    """key_len = 0: every row is empty -> O = 0, LSE = -inf, zero gradients."""
    rng = np.random.default_rng(0)
    q, k, v, do = (rng.standard_normal((1, 2, 6, 4)) for _ in range(4))
    O, LSE = oracle.attn_fwd(q, k, v, 0.5, False, [0])
    assert np.all(O == 0) and np.all(LSE == -np.inf)
    dQ, dK, dV, D = oracle.attn_bwd(q, k, v, do, 0.5, False, [0])
    assert np.all(dQ == 0) and np.all(dK == 0) and np.all(dV == 0) and np.all(D == 0)


def test_rejects_bad_arguments():
    q = np.zeros((1, 1, 4, 2))
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, q, q, 1.0, False, [5])       # key_len > N
    with pytest.raises(ValueError):
        oracle.attn_fwd(q, q, q, 1.0, False, None, 1.0)  # p outside [0, 1)


# ---------------------------------------------------------------------------
# mutation test: plausible mistakes planted in a copy of the oracle must each
# fail at least one pin (the copy is built on the CPU, in a temporary folder)
# ---------------------------------------------------------------------------
MUTATIONS = {
    "drop_D_term": ("* (dS[(size_t)i * N + j] - Di);", "* (dS[(size_t)i * N + j]);"),
    "dK_sign": ("for (size_t x = 0; x < (size_t)N * d; ++x) dk[x] *= scale;",
                "for (size_t x = 0; x < (size_t)N * d; ++x) dk[x] *= -scale;"),
    "dQ_missing_scale": ("dq[(size_t)i * d + c] = scale * acc;", "dq[(size_t)i * d + c] = acc;"),
    "dV_transposed": ("dv[(size_t)j * d + c] += w * dout[(size_t)i * d + c];",
                      "dv[(size_t)i * d + c] += w * dout[(size_t)j * d + c];"),
    "causal_off_by_one": ("if (causal && j > i) return 0;", "if (causal && j >= i) return 0;"),
    "window_off_by_one": ("if (i - j >= window) return 0;", "if (i - j > window) return 0;"),
    "window_one_sided": ("if (!causal && j - i >= window) return 0;", "if (0) return 0;"),
    "cross_offset_sign": ("if (valid_pair(i + off, j, causal, window, key_len)) {",
                          "if (valid_pair(i - off, j, causal, window, key_len)) {"),
    "scores_unscaled": ("                s = scale * acc;\n", "                s = acc;\n"),
    "dropout_no_rescale": ("oracle_dropout_keep(seed, b, h, i, j, t) ? inv : 0.0;",
                           "oracle_dropout_keep(seed, b, h, i, j, t) ? 1.0 : 0.0;"),
    "lse_missing_max": ("        lse[i] = m + log(l);\n", "        lse[i] = log(l);\n"),
    "philox_swapped_words": ("uint32_t n0 = hi1 ^ c1 ^ k0;", "uint32_t n0 = hi0 ^ c1 ^ k0;"),
    "dropout_counter_swapped": ("{(uint32_t)i, (uint32_t)j >> 3, (uint32_t)h, (uint32_t)b}",
                                "{(uint32_t)j >> 3, (uint32_t)i, (uint32_t)h, (uint32_t)b}"),
    "dropout_counter_stride": ("{(uint32_t)i, (uint32_t)j >> 3, (uint32_t)h, (uint32_t)b}",
                               "{(uint32_t)i, (uint32_t)j >> 2, (uint32_t)h, (uint32_t)b}"),
    "dropout_word_index": ("uint32_t word = r[(j >> 1) & 3];", "uint32_t word = r[j & 3];"),
    "dropout_halves_swapped": ("(j & 1) ? (word >> 16) : (word & 0xFFFFu);",
                               "(j & 1) ? (word & 0xFFFFu) : (word >> 16);"),
    "keep_compare_flipped": ("return draw < threshold ? 0 : 1;",
                             "return draw < threshold ? 1 : 0;"),
    "tiled_no_rescale": ("for (int c = 0; c < d; ++c) acc[(size_t)r * d + c] *= alpha;",
                         "for (int c = 0; c < d; ++c) acc[(size_t)r * d + c] *= 1.0;"),
}

# the cheap pins run on every mutant; finite differences use smaller sizes
_FAST = {k: v for k, v in PINS.items() if k != "finite_differences"}


def _pins_fail(lib) -> list:
    failed = []
    for name, (fn, bound) in _FAST.items():
        try:
            err = fn(lib)
        except Exception:
            failed.append(name)
            continue
        if not err <= bound:
            failed.append(name)
    from oracle_pins import pin_finite_differences
    if not pin_finite_differences(lib, sizes=((5, 4),)) <= 1e-6:
        failed.append("finite_differences")
    return failed


@pytest.mark.parametrize("mutation", sorted(MUTATIONS))
def test_mutation_is_caught(mutation, tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = open(oracle._SRC).read()
    old, new = MUTATIONS[mutation]
    assert src.count(old) >= 1, f"mutation anchor not found: {old!r}"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    so = tmp_path / "liboracle_mut.so"
    oracle.build(force=True, src=str(mutated), out=str(so))
    lib = oracle.load_variant(str(so))
    failed = _pins_fail(lib)
    if mutation.startswith("philox") and not failed:
        bad = pin_philox_vs_triton(lib)
        if not math.isnan(bad) and bad > 0:
            failed.append("philox_vs_triton")
    assert failed, f"mutation {mutation} slipped through every pin"
