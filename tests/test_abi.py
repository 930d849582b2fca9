"""The C ABI library loads, exports what include/gbattn.h declares, and rejects
bad arguments before touching the GPU (CPU only: every call here returns
before any CUDA call, so fake pointers are safe)."""
import ctypes
import os
import re

import pytest

import exact_attention_58_gb300 as ea
from exact_attention_58_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gbattn.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ea.LIB_PATH):
        _build.build()
    return ea.library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_[a-z_0-9]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_status_string",
                     "attn_version"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"libgbattn.so does not export {name}"
    # and nothing in the shared object is a C++-only stand-in
    assert lib.attn_version() == 200


def test_status_strings(lib):
    for code in range(7):
        assert ea.attn_status_string(code) != "unknown status"
    assert ea.attn_status_string(99) == "unknown status"


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every case fails validation first


def _fwd(lib, **kw):
    a = dict(Q=FAKE, K=FAKE, V=FAKE, O=FAKE, LSE=FAKE, B=1, H=1, N=128, d=64, dtype=0,
             scale=0.125, causal=0, window=0, key_lens=None, p=0.0, seed=0, dev_status=None,
             stream=None)
    a.update(kw)
    a.setdefault("Nk", a["N"])
    return lib.attn_fwd(a["Q"], a["K"], a["V"], a["O"], a["LSE"], a["B"], a["H"], a["N"],
                        a["Nk"], a["d"], a["dtype"], a["scale"], a["causal"], a["window"], a["key_lens"],
                        a["p"], a["seed"], a["dev_status"], a["stream"])


@pytest.mark.parametrize("kw,expected", [
    (dict(Q=None), 1),
    (dict(LSE=None), 1),
    (dict(N=0), 1),
    (dict(Nk=0), 1),
    (dict(N=128, Nk=-5), 1),
    (dict(B=-1), 1),
    (dict(d=96), 2),
    (dict(d=256, dtype=1), 2),     # head dim 256: 16-bit types only
    (dict(d=256, dtype=3), 2),
    (dict(d=512), 2),
    (dict(dtype=1, d=128), 2),
    (dict(dtype=2, d=96), 2),
    (dict(dtype=3), 2),            # e4m3 needs d = 128
    (dict(dtype=4), 1),
    (dict(dtype=7), 1),
    (dict(scale=0.0), 1),
    (dict(scale=float("nan")), 1),
    (dict(scale=-1.0), 1),
    (dict(p=1.0), 1),
    (dict(p=-0.1), 1),
    (dict(K=FAKE + 8), 3),
    (dict(O=FAKE + 2), 3),
    (dict(B=65536, H=65536), 2),
    (dict(B=64, H=64, N=128, Nk=1 << 20), 2),
])
def test_fwd_validation(lib, kw, expected):
    assert _fwd(lib, **kw) == expected


def _bwd(lib, **kw):
    a = dict(B=1, H=1, N=128, d=64, dtype=0, scale=0.125, p=0.0, ws=FAKE, ws_bytes=1 << 20,
             ptrs=[FAKE] * 9)
    a.update(kw)
    a.setdefault("Nk", a["N"])
    return lib.attn_bwd(*a["ptrs"], a["B"], a["H"], a["N"], a["Nk"], a["d"], a["dtype"], a["scale"], 0,
                        0, None, a["p"], 0, a["ws"], a["ws_bytes"], None, None)


@pytest.mark.parametrize("kw,expected", [
    (dict(ptrs=[FAKE] * 8 + [None]), 1),
    (dict(dtype=1), 2),
    (dict(dtype=2, d=96), 2),
    (dict(dtype=3), 2),            # e4m3: forward only
    (dict(dtype=3, d=128), 2),
    (dict(d=256, dtype=1), 2),     # head dim 256: 16-bit types only
    (dict(d=512), 2),
    (dict(dtype=4), 1),
    (dict(d=80), 2),
    (dict(ws=None), 4),
    (dict(ws_bytes=16), 4),
    (dict(ws=FAKE + 4), 3),
    (dict(ptrs=[FAKE] * 5 + [FAKE + 4] + [FAKE] * 3), 3),
    (dict(p=1.5), 1),
    (dict(Nk=0), 1),
    (dict(B=64, H=64, Nk=1 << 20), 2),
])
def test_bwd_validation(lib, kw, expected):
    assert _bwd(lib, **kw) == expected


def _fwd_varlen(lib, **kw):
    a = dict(ptrs=[FAKE] * 5, cu_q=FAKE, cu_k=FAKE, B=2, H=1, tq=300, tk=300, mq=200, mk=200,
             d=64, dtype=0, scale=0.125, p=0.0)
    a.update(kw)
    return lib.attn_fwd_varlen(*a["ptrs"], a["cu_q"], a["cu_k"], a["B"], a["H"], a["tq"], a["tk"],
                               a["mq"], a["mk"], a["d"], a["dtype"], a["scale"], 0, 0, a["p"], 0,
                               None, None)


def _bwd_varlen(lib, **kw):
    a = dict(ptrs=[FAKE] * 9, cu_q=FAKE, cu_k=FAKE, B=2, H=1, tq=300, tk=300, mq=200, mk=200,
             d=64, dtype=0, scale=0.125, p=0.0, ws=FAKE, ws_bytes=1 << 20)
    a.update(kw)
    return lib.attn_bwd_varlen(*a["ptrs"], a["cu_q"], a["cu_k"], a["B"], a["H"], a["tq"], a["tk"],
                               a["mq"], a["mk"], a["d"], a["dtype"], a["scale"], 0, 0, a["p"], 0,
                               a["ws"], a["ws_bytes"], None, None)


VARLEN_CASES = [
    (dict(cu_q=None), 1),
    (dict(cu_k=None), 1),
    (dict(cu_q=FAKE + 2), 3),
    (dict(tq=0), 1),
    (dict(tk=-1), 1),
    (dict(mq=0), 1),
    (dict(mk=0), 1),
    (dict(B=0), 1),
    (dict(d=96), 2),
    (dict(dtype=1), 2),
    (dict(dtype=5), 1),
    (dict(scale=0.0), 1),
    (dict(p=1.0), 1),
    (dict(H=64, tq=1 << 20), 2),
    (dict(B=4096, H=64, mq=1 << 14), 2),
]


@pytest.mark.parametrize("kw,expected", VARLEN_CASES + [(dict(ptrs=[FAKE] * 4 + [None]), 1),
                                                        (dict(ptrs=[FAKE + 8] + [FAKE] * 4), 3)])
def test_fwd_varlen_validation(lib, kw, expected):
    assert _fwd_varlen(lib, **kw) == expected


@pytest.mark.parametrize("kw,expected", VARLEN_CASES + [(dict(ptrs=[FAKE] * 8 + [None]), 1),
                                                        (dict(ws=None), 4),
                                                        (dict(ws_bytes=64), 4)])
def test_bwd_varlen_validation(lib, kw, expected):
    assert _bwd_varlen(lib, **kw) == expected


def test_workspace_size(lib):
    # D and log-sum-exp (2 floats per padded row) plus the fp32 dQ accumulator
    assert ea.attn_bwd_workspace_size(2, 3, 130, 64) == 2 * 3 * 256 * (2 + 64) * 4
    assert ea.attn_bwd_workspace_size(1, 1, 128, 128) == 128 * 130 * 4
    assert ea.attn_bwd_workspace_size(1, 1, 128, 96) == 0


def test_product_path_fails_loudly_without_the_library(tmp_path, monkeypatch):
    """The binding has no fallback: a missing library is an error, not a CPU path."""
    import importlib
    monkeypatch.setattr(ea, "_lib", None)
    monkeypatch.setattr(ea, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="no fallback"):
        ea.library()
    monkeypatch.setattr(ea, "_lib", None)
    importlib.reload(ea)


def test_product_code_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "exact_attention_58_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", text, re.M), f
                assert "liboracle" not in text and "oracle.c" not in text, f


def test_binding_rejects_bad_packed_arguments_before_any_call():
    """The Python binding checks packed-sequence tensors before it reaches the
    library (CPU tensors: any call into the library would fail differently)."""
    import torch
    q = torch.zeros(10, 2, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 4, 10], dtype=torch.int32)
    with pytest.raises(ValueError, match="k must be"):
        ea.attn_fwd_varlen(q, torch.zeros(10, 3, 64, dtype=torch.bfloat16), q, cu, cu, 6, 6)
    with pytest.raises(ValueError, match="v must match"):
        ea.attn_fwd_varlen(q, q, torch.zeros(9, 2, 64, dtype=torch.bfloat16), cu, cu, 6, 6)
    with pytest.raises(ValueError, match="cu_seqlens_q"):
        ea.attn_fwd_varlen(q, q, q, cu.to(torch.int64), cu, 6, 6)
    with pytest.raises(ValueError, match="same length"):
        ea.attn_fwd_varlen(q, q, q, cu, torch.tensor([0, 10], dtype=torch.int32), 6, 6)
    with pytest.raises(ValueError, match="expected q"):
        ea.attn_fwd_varlen(q[None], q, q, cu, cu, 6, 6)


def test_binding_rejects_mismatched_dense_keys():
    import torch
    q = torch.zeros(1, 2, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="k must be"):
        ea.attn_fwd(q, torch.zeros(1, 3, 8, 64, dtype=torch.bfloat16), q)
    with pytest.raises(ValueError, match="k must be"):
        ea.attn_fwd(q, torch.zeros(1, 2, 8, 32, dtype=torch.bfloat16), q)


def _noalloc(lib, **kw):
    a = dict(B=4, H=16, N=4096, d=128, dtype=0, scale=0.088, p=0.0, ptrs=[FAKE] * 9)
    a.update(kw)
    a.setdefault("Nk", a["N"])
    return lib.attn_bwd_noalloc(*a["ptrs"], a["B"], a["H"], a["N"], a["Nk"], a["d"], a["dtype"],
                                a["scale"], 1, 0, None, a["p"], 0, None, None)


@pytest.mark.parametrize("kw,expected", [
    (dict(), 4),                                   # valid, but 136 MB of scratch > 32 MiB
    (dict(dtype=1), 2),                            # fp32 backward: unsupported, whatever the size
    (dict(scale=float("nan")), 1),
    (dict(p=1.0), 1),
    (dict(Nk=0), 1),
    (dict(ptrs=[FAKE] * 8 + [FAKE + 8]), 3),      # misaligned dV
    (dict(ptrs=[FAKE] * 8 + [None]), 1),
])
def test_noalloc_reports_attn_bwd_errors_before_its_size_limit(lib, kw, expected):
    """attn_bwd_noalloc returns the same argument errors as attn_bwd; only a
    shape that passes them and needs more than the built-in scratch gets
    ATTN_ERR_WORKSPACE."""
    assert _noalloc(lib, **kw) == expected


def test_binding_rejects_views_and_foreign_buffers():
    """Malformed tensors are refused by the binding before the library sees
    them: a transposed (non-contiguous) q, an lse of the wrong type or shape,
    a dev_status that is not int32, and tensors that are not on a GPU."""
    import torch
    B, H, N, d = 1, 2, 8, 64
    x = torch.zeros(B, H, N, d, dtype=torch.bfloat16)
    qt = torch.zeros(B, N, H, d, dtype=torch.bfloat16).transpose(1, 2)   # [B, H, N, d] view
    lse = torch.zeros(B, H, N, dtype=torch.float32)
    with pytest.raises(ValueError, match="q must be contiguous"):
        ea.attn_bwd(qt, x, x, x, x, lse)
    with pytest.raises(ValueError, match="q must be contiguous"):
        ea.attn_bwd_noalloc(qt, x, x, x, x, lse)
    with pytest.raises(ValueError, match="q must be contiguous"):
        ea.attn_fwd(qt, x, x)
    with pytest.raises(ValueError, match="lse must be"):
        ea.attn_bwd(x, x, x, x, x, lse.to(torch.float16))
    with pytest.raises(ValueError, match="lse must be"):
        ea.attn_bwd(x, x, x, x, x, lse[:, :, :4])
    with pytest.raises(ValueError, match="lse must be"):
        ea.attn_fwd(x, x, x, lse=lse.double())
    with pytest.raises(ValueError, match="dev_status must be"):
        ea.attn_fwd(x, x, x, dev_status=torch.zeros(1, dtype=torch.int64))
    with pytest.raises(ValueError, match="dev_status must be"):
        ea.attn_bwd(x, x, x, x, x, lse, dev_status=torch.zeros(0, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA device"):
        ea.attn_fwd(x, x, x)
    with pytest.raises(ValueError, match="CUDA device"):
        ea.attn_bwd(x, x, x, x, x, lse, workspace=torch.zeros(1 << 16, dtype=torch.uint8))
    pq = torch.zeros(10, H, d, dtype=torch.bfloat16)
    cu = torch.tensor([0, 4, 10], dtype=torch.int32)
    with pytest.raises(ValueError, match="q must be"):
        ea.attn_bwd_varlen(torch.zeros(10, d, H, dtype=torch.bfloat16).transpose(1, 2), pq, pq,
                           pq, pq, torch.zeros(H, 10), cu, cu, 6, 6)
    with pytest.raises(ValueError, match="lse must be"):
        ea.attn_bwd_varlen(pq, pq, pq, pq, pq, torch.zeros(H, 9), cu, cu, 6, 6)
