"""Fused exact attention for GB300 (sm_103a): Python binding of libgbattn.so.

The functions here carry the names of the C ABI in ``include/gbattn.h`` and
do argument marshalling only: every step of the computation runs in the CUDA
kernels of ``libgbattn.so``.  PyTorch supplies device memory and streams.
There is no fallback: if the library has not been built, or an argument is
unsupported, the call raises.

    import exact_attention_58_gb300 as ea
    o, lse = ea.attn_fwd(q, k, v, causal=True)
    dq, dk, dv = ea.attn_bwd(q, k, v, o, do, lse, causal=True)

q, o, do, dq are [B, H, N, d] and k, v, dk, dv [B, H, Nk, d] (Nk = N for
self-attention), contiguous, on one CUDA device; bf16 or fp16 (d = 64 or 128;
the forward also d = 256), or, forward only, fp32 with d = 64 and e4m3
(torch.float8_e4m3fn, O in bf16) with d = 128.  attn_fwd_varlen and
attn_bwd_varlen take packed sequences: [total, H, d] tensors and cumulative
offsets.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading
from typing import Optional

import torch

from . import _build

__all__ = [
    "AttnError", "attn_fwd", "attn_bwd", "attn_bwd_workspace_size", "attn_bwd_preprocess",
    "attn_bwd_main", "attn_bwd_dq_convert", "attn_bwd_noalloc", "attn_fwd_varlen",
    "attn_bwd_varlen", "attn_selftest_wait", "attn_selftest_fwd_withheld", "attn_status_string",
    "attn_version", "library",
    "LIB_PATH", "STATUS",
]

LIB_PATH = _build.LIB_PATH

STATUS = {
    0: "ATTN_OK",
    1: "ATTN_ERR_INVALID_ARG",
    2: "ATTN_ERR_UNSUPPORTED",
    3: "ATTN_ERR_MISALIGNED",
    4: "ATTN_ERR_WORKSPACE",
    5: "ATTN_ERR_CUDA",
    6: "ATTN_ERR_DEVICE_TIMEOUT",
}
_DTYPE = {torch.bfloat16: 0, torch.float32: 1, torch.float16: 2}
if hasattr(torch, "float8_e4m3fn"):
    _DTYPE[torch.float8_e4m3fn] = 3


def _out_dtype(q: torch.Tensor):
    """O takes q's dtype, except bf16 for e4m3 inputs."""
    return torch.bfloat16 if _DTYPE.get(q.dtype) == 3 else q.dtype

_lock = threading.Lock()
_lib = None


class AttnError(RuntimeError):
    """A non-zero attn_status from the library."""

    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {STATUS.get(self.status, self.status)} "
                         f"({attn_status_string(self.status)})")


def library():
    """The loaded libgbattn.so.  Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with exact_attention_58_gb300._build.build() "
                    "(there is no fallback implementation)")
            lib = ctypes.CDLL(LIB_PATH)
            vp, ip, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
            f, u64 = ctypes.c_float, ctypes.c_uint64
            lib.attn_fwd.argtypes = [vp] * 5 + [ip] * 6 + [f, ip, ip, vp, f, u64, vp, vp]
            lib.attn_bwd.argtypes = [vp] * 9 + [ip] * 6 + [f, ip, ip, vp, f, u64, vp, sz, vp, vp]
            lib.attn_bwd_noalloc.argtypes = [vp] * 9 + [ip] * 6 + [f, ip, ip, vp, f, u64, vp, vp]
            lib.attn_bwd_workspace_size.argtypes = [ip, ip, ip, ip]
            lib.attn_bwd_workspace_size.restype = sz
            lib.attn_bwd_preprocess.argtypes = [vp, vp, vp, ip, ip, ip, ip, ip, vp, sz, vp]
            lib.attn_bwd_main.argtypes = [vp] * 6 + [ip] * 6 + [f, ip, ip, vp, f, u64, vp, sz, vp,
                                                              vp]
            lib.attn_bwd_dq_convert.argtypes = [vp, ip, ip, ip, ip, ip, f, vp, sz, vp]
            lib.attn_fwd_varlen.argtypes = [vp] * 7 + [ip] * 8 + [f, ip, ip, f, u64, vp, vp]
            lib.attn_selftest_wait.argtypes = [vp, ip, vp]
            lib.attn_selftest_wait.restype = ctypes.c_int
            lib.attn_selftest_fwd_withheld.argtypes = [vp] * 5 + [ip] * 6 + [vp, vp]
            lib.attn_selftest_fwd_withheld.restype = ctypes.c_int
            lib.attn_bwd_varlen.argtypes = ([vp] * 11 + [ip] * 8 +
                                            [f, ip, ip, f, u64, vp, sz, vp, vp])
            for fn in ("attn_fwd", "attn_bwd", "attn_bwd_preprocess", "attn_bwd_main",
                       "attn_bwd_dq_convert", "attn_bwd_noalloc", "attn_fwd_varlen",
                       "attn_bwd_varlen"):
                getattr(lib, fn).restype = ctypes.c_int
            lib.attn_status_string.argtypes = [ctypes.c_int]
            lib.attn_status_string.restype = ctypes.c_char_p
            lib.attn_version.argtypes = []
            lib.attn_version.restype = ctypes.c_int
            _lib = lib
        return _lib


def attn_status_string(status: int) -> str:
    return library().attn_status_string(int(status)).decode()


def attn_version() -> int:
    return int(library().attn_version())


def attn_bwd_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(library().attn_bwd_workspace_size(B, H, N, d))


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------
def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _shape(q: torch.Tensor):
    if not isinstance(q, torch.Tensor) or q.dim() != 4:
        raise ValueError("expected a [B, H, N, d] tensor")
    _check_like("q", q, q)
    return tuple(int(x) for x in q.shape)


def _check_like(name: str, t: torch.Tensor, ref: torch.Tensor):
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a tensor")
    if t.shape != ref.shape or t.dtype != ref.dtype or t.device != ref.device:
        raise ValueError(f"{name} must match q in shape, dtype and device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _on_gpu(q: torch.Tensor):
    """Every tensor argument has been checked to be on q's device; that device
    must be a CUDA one (a host pointer handed to a kernel would be read or
    written as if it were device memory)."""
    if not q.is_cuda:
        raise ValueError("the tensors must be on a CUDA device")


def _check_lse(lse, shape, q: torch.Tensor):
    """The log-sum-exp buffer: contiguous float32 of `shape` on q's device."""
    if (not isinstance(lse, torch.Tensor) or lse.dtype != torch.float32
            or tuple(lse.shape) != tuple(shape) or lse.device != q.device
            or not lse.is_contiguous()):
        raise ValueError(f"lse must be a contiguous float32 tensor of shape {tuple(shape)} "
                         "on q's device")
    return lse


def _check_status(dev_status, q: torch.Tensor):
    """dev_status: None, or an int32 tensor (at least one element) on q's device."""
    if dev_status is None:
        return None
    if (not isinstance(dev_status, torch.Tensor) or dev_status.dtype != torch.int32
            or dev_status.numel() < 1 or dev_status.device != q.device
            or not dev_status.is_contiguous()):
        raise ValueError("dev_status must be a contiguous int32 tensor with at least one "
                         "element on q's device")
    return dev_status


def _check_workspace(workspace, q: torch.Tensor):
    if (not isinstance(workspace, torch.Tensor) or workspace.device != q.device
            or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous tensor on q's device")
    return workspace


def _keys(q: torch.Tensor, k: torch.Tensor) -> int:
    """Nk of k, which must be [B, H, Nk, d] like q apart from its length."""
    if (not isinstance(k, torch.Tensor) or k.dim() != 4 or k.shape[:2] != q.shape[:2]
            or k.shape[3] != q.shape[3] or k.dtype != q.dtype or k.device != q.device):
        raise ValueError("k must be [B, H, Nk, d] with q's B, H, d, dtype and device")
    if not k.is_contiguous():
        raise ValueError("k must be contiguous")
    return int(k.shape[2])


def _dtype_code(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPE:
        raise ValueError(f"unsupported dtype {t.dtype}")
    return _DTYPE[t.dtype]


def _key_lens(key_lens, q):
    if key_lens is None:
        return None
    if (key_lens.dtype != torch.int32 or key_lens.device != q.device or key_lens.dim() != 1
            or key_lens.shape[0] != q.shape[0] or not key_lens.is_contiguous()):
        raise ValueError("key_lens must be a contiguous int32 [B] tensor on q's device")
    return key_lens


def _raise(st: int, where: str):
    if st != 0:
        raise AttnError(st, where)


# ---------------------------------------------------------------------------
# entry points
# ---------------------------------------------------------------------------
def attn_fwd(q, k, v, *, causal: bool = False, window: int = 0, key_lens=None,
             dropout_p: float = 0.0,
             seed: int = 0, scale: Optional[float] = None, out=None, lse=None,
             dev_status=None, stream=None):
    """O, LSE = attention(q, k, v); see include/gbattn.h for the exact contract."""
    B, H, N, d = _shape(q)
    _check_like("q", q, q)
    Nk = _keys(q, k)
    _check_like("v", v, k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=_out_dtype(q), device=q.device)
    if out.shape != q.shape or out.dtype != _out_dtype(q) or out.device != q.device \
            or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of q's shape (bf16 for e4m3 q)")
    if lse is None:
        lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    _check_lse(lse, (B, H, N), q)
    _check_status(dev_status, q)
    kl = _key_lens(key_lens, q)
    _on_gpu(q)
    st = library().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B, H, N, Nk, d,
                            _dtype_code(q), float(scale), int(bool(causal)), int(window), _ptr(kl),
                            float(dropout_p), int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(dev_status),
                            _stream(stream))
    _raise(st, "attn_fwd")
    return out, lse


def _workspace(B, H, N, d, workspace, q):
    need = attn_bwd_workspace_size(B, H, N, d)
    if workspace is None:
        workspace = torch.empty(max(need, 16), dtype=torch.uint8, device=q.device)
    _check_workspace(workspace, q)
    return workspace, int(workspace.numel() * workspace.element_size())


def attn_bwd(q, k, v, o, do, lse, *, causal: bool = False, window: int = 0, key_lens=None,
             dropout_p: float = 0.0, seed: int = 0, scale: Optional[float] = None, dq=None,
             dk=None, dv=None, workspace=None, dev_status=None, stream=None):
    """dQ, dK, dV of attention given the forward's o and lse and the gradient do."""
    B, H, N, d = _shape(q)
    Nk = _keys(q, k)
    for name, t in (("o", o), ("do", do)):
        _check_like(name, t, q)
    _check_like("v", v, k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(k) if dv is None else dv
    _check_like("dq", dq, q)
    _check_like("dk", dk, k)
    _check_like("dv", dv, k)
    _check_lse(lse, (B, H, N), q)
    _check_status(dev_status, q)
    ws, ws_bytes = _workspace(B, H, N, d, workspace, q)
    kl = _key_lens(key_lens, q)
    _on_gpu(q)
    st = library().attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                            _ptr(dk), _ptr(dv), B, H, N, Nk, d, _dtype_code(q), float(scale),
                            int(bool(causal)), int(window), _ptr(kl), float(dropout_p),
                            int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(ws), ws_bytes, _ptr(dev_status),
                            _stream(stream))
    _raise(st, "attn_bwd")
    return dq, dk, dv


def attn_bwd_noalloc(q, k, v, o, do, lse, *, causal: bool = False, window: int = 0,
                     key_lens=None,
                     dropout_p: float = 0.0, seed: int = 0, scale: Optional[float] = None,
                     dq=None, dk=None, dv=None, dev_status=None, stream=None):
    """attn_bwd using the library's built-in 32 MiB scratch instead of a
    workspace, for callers that cannot allocate device memory.  Outputs must be
    passed in (dq, dk, dv) by such callers; see include/gbattn.h."""
    B, H, N, d = _shape(q)
    Nk = _keys(q, k)
    for name, t in (("o", o), ("do", do)):
        _check_like(name, t, q)
    _check_like("v", v, k)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(k) if dv is None else dv
    _check_like("dq", dq, q)
    _check_like("dk", dk, k)
    _check_like("dv", dv, k)
    _check_lse(lse, (B, H, N), q)
    _check_status(dev_status, q)
    kl = _key_lens(key_lens, q)
    _on_gpu(q)
    st = library().attn_bwd_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                    _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, Nk, d, _dtype_code(q),
                                    float(scale), int(bool(causal)), int(window), _ptr(kl),
                                    float(dropout_p),
                                    int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(dev_status),
                                    _stream(stream))
    _raise(st, "attn_bwd_noalloc")
    return dq, dk, dv


def attn_bwd_preprocess(o, do, lse, workspace, *, stream=None):
    B, H, N, d = _shape(o)
    _check_like("do", do, o)
    _check_lse(lse, (B, H, N), o)
    _check_workspace(workspace, o)
    _on_gpu(o)
    st = library().attn_bwd_preprocess(_ptr(o), _ptr(do), _ptr(lse), B, H, N, d,
                                       _dtype_code(o), _ptr(workspace),
                                       workspace.numel() * workspace.element_size(),
                                       _stream(stream))
    _raise(st, "attn_bwd_preprocess")


def attn_bwd_main(q, k, v, do, dk, dv, workspace, *, causal=False, window=0, key_lens=None,
                  dropout_p=0.0, seed=0, scale=None, dev_status=None, stream=None):
    B, H, N, d = _shape(q)
    Nk = _keys(q, k)
    _check_like("v", v, k)
    _check_like("do", do, q)
    _check_like("dk", dk, k)
    _check_like("dv", dv, k)
    _check_workspace(workspace, q)
    _check_status(dev_status, q)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    kl = _key_lens(key_lens, q)
    _on_gpu(q)
    st = library().attn_bwd_main(_ptr(q), _ptr(k), _ptr(v), _ptr(do), _ptr(dk), _ptr(dv), B, H,
                                 N, Nk, d, _dtype_code(q), float(scale), int(bool(causal)),
                                 int(window), _ptr(kl),
                                 float(dropout_p), int(seed) & 0xFFFFFFFFFFFFFFFF,
                                 _ptr(workspace), workspace.numel() * workspace.element_size(),
                                 _ptr(dev_status), _stream(stream))
    _raise(st, "attn_bwd_main")


def attn_bwd_dq_convert(dq, workspace, *, scale=None, stream=None):
    B, H, N, d = _shape(dq)
    _check_workspace(workspace, dq)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    _on_gpu(dq)
    st = library().attn_bwd_dq_convert(_ptr(dq), B, H, N, d, _dtype_code(dq), float(scale),
                                       _ptr(workspace), workspace.numel() * workspace.element_size(),
                                       _stream(stream))
    _raise(st, "attn_bwd_dq_convert")


# ---------------------------------------------------------------------------
# packed variable-length sequences
# ---------------------------------------------------------------------------
def _packed(name: str, t: torch.Tensor, H: int, d: int, ref: torch.Tensor):
    if not isinstance(t, torch.Tensor):
        raise ValueError(f"{name} must be a tensor")
    if (t.dim() != 3 or t.shape[1] != H or t.shape[2] != d or t.dtype != ref.dtype
            or t.device != ref.device):
        raise ValueError(f"{name} must be [total, H, d] with q's H, d, dtype and device")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return int(t.shape[0])


def _cu(name: str, cu, q: torch.Tensor) -> int:
    if (not isinstance(cu, torch.Tensor) or cu.dtype != torch.int32 or cu.device != q.device
            or cu.dim() != 1 or cu.numel() < 2 or not cu.is_contiguous()):
        raise ValueError(f"{name} must be a contiguous int32 [B + 1] tensor on q's device")
    return int(cu.numel()) - 1


def attn_fwd_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, max_seqlen_k: int, *,
                    causal: bool = False, window: int = 0, dropout_p: float = 0.0, seed: int = 0,
                    scale: Optional[float] = None, out=None, lse=None, dev_status=None,
                    stream=None):
    """Attention over packed sequences: q [total_q, H, d], k, v [total_k, H, d],
    sequence b at rows [cu[b], cu[b+1]).  Returns O [total_q, H, d] and LSE
    [H, total_q]; see include/gbattn.h."""
    if q.dim() != 3:
        raise ValueError("expected q as [total_q, H, d]")
    total_q, H, d = (int(x) for x in q.shape)
    _packed("q", q, H, d, q)
    total_k = _packed("k", k, H, d, q)
    if _packed("v", v, H, d, q) != total_k:
        raise ValueError("v must match k")
    B = _cu("cu_seqlens_q", cu_seqlens_q, q)
    if _cu("cu_seqlens_k", cu_seqlens_k, q) != B:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty(q.shape, dtype=_out_dtype(q), device=q.device)
    if out.shape != q.shape or out.dtype != _out_dtype(q) or out.device != q.device \
            or not out.is_contiguous():
        raise ValueError("out must be a contiguous tensor of q's shape (bf16 for e4m3 q)")
    if lse is None:
        lse = torch.empty((H, total_q), dtype=torch.float32, device=q.device)
    _check_lse(lse, (H, total_q), q)
    _check_status(dev_status, q)
    _on_gpu(q)
    st = library().attn_fwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse),
                                   _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), B, H, total_q, total_k,
                                   int(max_seqlen_q), int(max_seqlen_k), d, _dtype_code(q),
                                   float(scale), int(bool(causal)), int(window), float(dropout_p),
                                   int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(dev_status),
                                   _stream(stream))
    _raise(st, "attn_fwd_varlen")
    return out, lse


def attn_bwd_varlen(q, k, v, o, do, lse, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int,
                    max_seqlen_k: int, *, causal: bool = False, window: int = 0,
                    dropout_p: float = 0.0, seed: int = 0, scale: Optional[float] = None,
                    dq=None, dk=None, dv=None, workspace=None, dev_status=None, stream=None):
    """dQ, dK, dV of attn_fwd_varlen (same packed layouts)."""
    if q.dim() != 3:
        raise ValueError("expected q as [total_q, H, d]")
    total_q, H, d = (int(x) for x in q.shape)
    _packed("q", q, H, d, q)
    total_k = _packed("k", k, H, d, q)
    if _packed("v", v, H, d, q) != total_k:
        raise ValueError("v must match k")
    for name, t in (("o", o), ("do", do)):
        _check_like(name, t, q)
    B = _cu("cu_seqlens_q", cu_seqlens_q, q)
    if _cu("cu_seqlens_k", cu_seqlens_k, q) != B:
        raise ValueError("cu_seqlens_q and cu_seqlens_k must have the same length")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(k) if dv is None else dv
    _check_like("dq", dq, q)
    _check_like("dk", dk, k)
    _check_like("dv", dv, k)
    _check_lse(lse, (H, total_q), q)
    _check_status(dev_status, q)
    ws, ws_bytes = _workspace(B, H, int(max_seqlen_q), d, workspace, q)
    _on_gpu(q)
    st = library().attn_bwd_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                   _ptr(dq), _ptr(dk), _ptr(dv), _ptr(cu_seqlens_q),
                                   _ptr(cu_seqlens_k), B, H, total_q, total_k, int(max_seqlen_q),
                                   int(max_seqlen_k), d, _dtype_code(q), float(scale),
                                   int(bool(causal)), int(window), float(dropout_p),
                                   int(seed) & 0xFFFFFFFFFFFFFFFF, _ptr(ws), ws_bytes,
                                   _ptr(dev_status), _stream(stream))
    _raise(st, "attn_bwd_varlen")
    return dq, dk, dv


def attn_selftest_wait(dev_status, *, arrive: bool, stream=None):
    """Device self-test of the bounded waits (see include/gbattn.h): with
    arrive=False the wait expires and ATTN_ERR_DEVICE_TIMEOUT lands in
    dev_status (a CUDA int32 tensor, 0 on entry)."""
    st = library().attn_selftest_wait(_ptr(dev_status), int(bool(arrive)), _stream(stream))
    _raise(st, "attn_selftest_wait")


def attn_selftest_fwd_withheld(q, k, v, dev_status, *, withhold_block: int, wait_ms: int = 20,
                               out=None, lse=None, stream=None):
    """Device self-test of the forward kernel's abort path (see
    include/gbattn.h): bf16 [B, H, N, 128] q and [B, H, Nk, 128] k, v; the K
    tile of key block `withhold_block` is never loaded (< 0: nothing withheld)
    and waits give up after `wait_ms`.  dev_status: a CUDA int32 tensor, 0 on
    entry."""
    B, H, N, d = _shape(q)
    Nk = _keys(q, k)
    _check_like("v", v, k)
    if q.dtype != torch.bfloat16 or d != 128:
        raise ValueError("the self test runs bf16 with d = 128")
    out = torch.empty_like(q) if out is None else out
    _check_like("out", out, q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    _check_lse(lse, (B, H, N), q)
    if _check_status(dev_status, q) is None:
        raise ValueError("dev_status is required")
    _on_gpu(q)
    st = library().attn_selftest_fwd_withheld(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), B,
                                              H, N, Nk, int(withhold_block), int(wait_ms),
                                              _ptr(dev_status), _stream(stream))
    _raise(st, "attn_selftest_fwd_withheld")
    return out, lse
