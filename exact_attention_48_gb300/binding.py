"""Thin ctypes binding of libfa.so (argument marshalling only).

The functions carry the C-ABI names.  They take torch CUDA tensors, check
dtype/shape/contiguity, allocate outputs with torch when none are given and
pass raw device pointers and the current torch stream to the library.  Every
step of the computation runs in the library's kernels; there is no fallback:
if ``libfa.so`` is missing or cannot be loaded, every call raises.
"""
from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

from .build import LIB

_lock = threading.Lock()
_lib = None

FA_OK = 0
STATUS_NAMES = {
    0: "FA_OK",
    1: "FA_ERR_INVALID_ARGUMENT",
    2: "FA_ERR_UNSUPPORTED",
    3: "FA_ERR_WORKSPACE",
    4: "FA_ERR_CUDA",
    5: "FA_ERR_DEVICE_TIMEOUT",
}


class FaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)} ({status_string(code)})")


def library(path: str | None = None):
    """Load (once) and return the ctypes handle of libfa.so."""
    global _lib
    with _lock:
        if _lib is None:
            p = path or LIB
            if not os.path.exists(p):
                raise RuntimeError(
                    f"libfa.so not found at {p}; build it with "
                    "`python -m exact_attention_48_gb300.build` (there is no CPU fallback)")
            lib = ctypes.CDLL(p)
            vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
            lib.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
            lib.fa_fwd.restype = i
            lib.fa_bwd_workspace_bytes.argtypes = [i, i, i, i]
            lib.fa_bwd_workspace_bytes.restype = sz
            lib.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, sz, vp]
            lib.fa_bwd.restype = i
            lib.fa_bwd_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, vp]
            lib.fa_bwd_noalloc.restype = i
            lib.fa_device_status.argtypes = [vp]
            lib.fa_device_status.restype = i
            lib.fa_debug_last_wait_site.argtypes = []
            lib.fa_debug_last_wait_site.restype = i
            lib.fa_debug_time_next_bwd.argtypes = [vp, vp, vp]
            lib.fa_debug_time_next_bwd.restype = i
            p64 = ctypes.POINTER(ctypes.c_int64)
            lib.fa_fwd_strided.argtypes = [vp, p64, vp, p64, vp, p64, vp, p64, vp, i, i, i, i, i, f, vp]
            lib.fa_fwd_strided.restype = i
            lib.fa_bwd_strided.argtypes = [vp, p64, vp, p64, vp, p64, vp, p64, vp, p64, vp, vp, p64, vp, p64,
                                           vp, p64, i, i, i, i, i, f, vp, sz, vp]
            lib.fa_bwd_strided.restype = i
            lib.fa_fwd_varlen.argtypes = [vp, p64, vp, p64, vp, p64, vp, p64, vp, vp, i, i, i, i, i, i, f, vp]
            lib.fa_fwd_varlen.restype = i
            lib.fa_bwd_varlen.argtypes = [vp, p64, vp, p64, vp, p64, vp, p64, vp, p64, vp, vp, p64, vp, p64,
                                          vp, p64, vp, i, i, i, i, i, i, f, vp, sz, vp]
            lib.fa_bwd_varlen.restype = i
            lib.fa_fwd_fp8.argtypes = [vp, vp, vp, f, f, f, vp, vp, i, i, i, i, i, f, vp]
            lib.fa_fwd_fp8.restype = i
            lib.fa_decode_workspace_bytes.argtypes = [i, i, i, i, i]
            lib.fa_decode_workspace_bytes.restype = sz
            lib.fa_fwd_decode.argtypes = [vp, p64, vp, p64, vp, p64, vp, p64, vp, vp, i, i, i, i, i, i, f, vp, sz,
                                          vp]
            lib.fa_fwd_decode.restype = i
            lib.fa_status_string.argtypes = [i]
            lib.fa_status_string.restype = ctypes.c_char_p
            _lib = lib
    return _lib


def status_string(code: int) -> str:
    return library().fa_status_string(int(code)).decode()


def _stream_handle(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _check_qkv(name, t, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _check_view(name, t, shape=None):
    """A [B, H, N, d] bf16 CUDA view with contiguous d (any other strides)."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != 4 or t.stride(-1) != 1:
        raise ValueError(f"{name} must be a [B, H, N, d] view with contiguous d")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _strides(t):
    return (ctypes.c_int64 * 3)(*t.stride()[:3])


def fa_fwd_strided(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None, stream=None):
    """fa_fwd on [B, H, N, d] views of any layout whose d is contiguous
    (e.g. ``x.transpose(1, 2)`` of a [B, N, H, d] tensor, or the q, k, v
    slices of a packed projection).  ``o`` defaults to a contiguous tensor."""
    _check_view("q", q)
    B, H, N, d = q.shape
    _check_view("k", k, q.shape)
    _check_view("v", v, q.shape)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty(q.shape, device=q.device, dtype=q.dtype)
    else:
        _check_view("o", o, q.shape)
    if lse is None:
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    elif lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    rc = library().fa_fwd_strided(q.data_ptr(), _strides(q), k.data_ptr(), _strides(k), v.data_ptr(), _strides(v),
                                  o.data_ptr(), _strides(o), lse.data_ptr(), B, H, N, d, int(bool(causal)),
                                  float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_strided")
    return o, lse


def fa_bwd_strided(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None,
                   dq=None, dk=None, dv=None, workspace=None, stream=None):
    """fa_bwd on [B, H, N, d] views of any layout whose d is contiguous;
    dq, dk, dv default to contiguous tensors."""
    _check_view("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_view(name, t, q.shape)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous() or not lse.is_cuda:
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [B, H, N]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    new = lambda: torch.empty(q.shape, device=q.device, dtype=q.dtype)  # noqa: E731
    dq = new() if dq is None else dq
    dk = new() if dk is None else dk
    dv = new() if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_view(name, t, q.shape)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    rc = library().fa_bwd_strided(q.data_ptr(), _strides(q), k.data_ptr(), _strides(k), v.data_ptr(), _strides(v),
                                  o.data_ptr(), _strides(o), dout.data_ptr(), _strides(dout), lse.data_ptr(),
                                  dq.data_ptr(), _strides(dq), dk.data_ptr(), _strides(dk), dv.data_ptr(),
                                  _strides(dv), B, H, N, d, int(bool(causal)), float(scale), ws_ptr, ws_bytes,
                                  _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_strided")
    return dq, dk, dv


def _check_packed(name, t, shape=None):
    """A [T, H, d] bf16 CUDA view with contiguous d."""
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != torch.bfloat16:
        raise TypeError(f"{name} must be bfloat16, got {t.dtype}")
    if t.dim() != 3 or t.stride(-1) != 1:
        raise ValueError(f"{name} must be a [T, H, d] view with contiguous d")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _strides2(t):
    return (ctypes.c_int64 * 2)(t.stride(0), t.stride(1))


def _check_cu(cu_seqlens):
    if not isinstance(cu_seqlens, torch.Tensor) or not cu_seqlens.is_cuda or cu_seqlens.dtype != torch.int32 \
            or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous() or cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens must be a contiguous int32 CUDA tensor of B + 1 row offsets")
    return cu_seqlens.numel() - 1


def fa_fwd_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False, scale: float | None = None,
                  o=None, lse=None, stream=None):
    """Attention over B packed sequences: q, k, v are [T, H, d] (rows of all
    sequences back to back), sequence b is rows cu_seqlens[b]:cu_seqlens[b+1].
    Returns (o [T, H, d] bf16, lse [H, T] fp32)."""
    _check_packed("q", q)
    T, H, d = q.shape
    _check_packed("k", k, q.shape)
    _check_packed("v", v, q.shape)
    B = _check_cu(cu_seqlens)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    o = torch.empty(q.shape, device=q.device, dtype=q.dtype) if o is None else o
    _check_packed("o", o, q.shape)
    if lse is None:
        lse = torch.empty((H, T), device=q.device, dtype=torch.float32)
    elif lse.dtype != torch.float32 or tuple(lse.shape) != (H, T) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [H, T] tensor")
    rc = library().fa_fwd_varlen(q.data_ptr(), _strides2(q), k.data_ptr(), _strides2(k), v.data_ptr(), _strides2(v),
                                 o.data_ptr(), _strides2(o), lse.data_ptr(), cu_seqlens.data_ptr(), B, H, T,
                                 int(max_seqlen), d, int(bool(causal)), float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_varlen")
    return o, lse


def fa_bwd_varlen(q, k, v, o, dout, lse, cu_seqlens, max_seqlen: int, causal: bool = False,
                  scale: float | None = None, dq=None, dk=None, dv=None, workspace=None, stream=None):
    """Gradients of fa_fwd_varlen; dq, dk, dv default to contiguous [T, H, d]."""
    _check_packed("q", q)
    T, H, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_packed(name, t, q.shape)
    B = _check_cu(cu_seqlens)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, T) or not lse.is_contiguous() or not lse.is_cuda:
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [H, T]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    new = lambda: torch.empty(q.shape, device=q.device, dtype=q.dtype)  # noqa: E731
    dq = new() if dq is None else dq
    dk = new() if dk is None else dk
    dv = new() if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_packed(name, t, q.shape)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    rc = library().fa_bwd_varlen(q.data_ptr(), _strides2(q), k.data_ptr(), _strides2(k), v.data_ptr(), _strides2(v),
                                 o.data_ptr(), _strides2(o), dout.data_ptr(), _strides2(dout), lse.data_ptr(),
                                 dq.data_ptr(), _strides2(dq), dk.data_ptr(), _strides2(dk), dv.data_ptr(),
                                 _strides2(dv), cu_seqlens.data_ptr(), B, H, T, int(max_seqlen), d,
                                 int(bool(causal)), float(scale), ws_ptr, ws_bytes, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_varlen")
    return dq, dk, dv


def _check_e4m3(name, t, shape=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype not in (torch.float8_e4m3fn, torch.uint8):
        raise TypeError(f"{name} must hold e4m3 codes (float8_e4m3fn or uint8), got {t.dtype}")
    if t.dim() != 4 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous [B, H, N, d] tensor")
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def fa_fwd_fp8(q8, k8, v8, q_scale: float, k_scale: float, v_scale: float, causal: bool = False,
               scale: float | None = None, o=None, lse=None, stream=None):
    """FP8 forward: q8, k8, v8 contiguous [B, H, N, d] e4m3 codes
    (torch.float8_e4m3fn or uint8) with one scale per tensor (value = code *
    scale); d = 128.  Returns (o [B, H, N, d] bf16, lse [B, H, N] fp32)."""
    _check_e4m3("q8", q8)
    B, H, N, d = q8.shape
    _check_e4m3("k8", k8, q8.shape)
    _check_e4m3("v8", v8, q8.shape)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty(q8.shape, device=q8.device, dtype=torch.bfloat16)
    else:
        _check_qkv("o", o, q8.shape)
    if lse is None:
        lse = torch.empty((B, H, N), device=q8.device, dtype=torch.float32)
    elif lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    rc = library().fa_fwd_fp8(q8.data_ptr(), k8.data_ptr(), v8.data_ptr(), float(q_scale), float(k_scale),
                              float(v_scale), o.data_ptr(), lse.data_ptr(), B, H, N, d, int(bool(causal)),
                              float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_fp8")
    return o, lse


def fa_decode_workspace_bytes(B: int, H: int, Nq: int, Nk: int, d: int) -> int:
    return int(library().fa_decode_workspace_bytes(B, H, Nq, Nk, d))


def fa_fwd_decode(q, k, v, cache_seqlens=None, causal: bool = False, scale: float | None = None, o=None, lse=None,
                  workspace=None, stream=None):
    """Decode forward: q [B, H, Nq, d] (Nq <= 8, the last Nq positions)
    against a key/value cache k, v [B, H, Nk, d] (views with contiguous d,
    e.g. ``cache.transpose(1, 2)`` of a [B, Nk, H, d] cache), of which the
    first cache_seqlens[b] rows are valid (int32 CUDA tensor [B], or None
    for all Nk).  Returns (o [B, H, Nq, d] bf16, lse [B, H, Nq] fp32)."""
    _check_view("q", q)
    B, H, Nq, d = q.shape
    _check_view("k", k)
    Nk = k.shape[2]
    if tuple(k.shape) != (B, H, Nk, d):
        raise ValueError(f"k has shape {tuple(k.shape)}, expected ({B}, {H}, Nk, {d})")
    _check_view("v", v, k.shape)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty(q.shape, device=q.device, dtype=q.dtype)
    else:
        _check_view("o", o, q.shape)
    if lse is None:
        lse = torch.empty((B, H, Nq), device=q.device, dtype=torch.float32)
    elif lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Nq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, Nq] tensor")
    cl = None
    if cache_seqlens is not None:
        if not isinstance(cache_seqlens, torch.Tensor) or not cache_seqlens.is_cuda \
                or cache_seqlens.dtype != torch.int32 or tuple(cache_seqlens.shape) != (B,) \
                or not cache_seqlens.is_contiguous():
            raise ValueError("cache_seqlens must be a contiguous int32 CUDA tensor [B]")
        cl = cache_seqlens.data_ptr()
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    rc = library().fa_fwd_decode(q.data_ptr(), _strides(q), k.data_ptr(), _strides(k), v.data_ptr(), _strides(v),
                                 o.data_ptr(), _strides(o), lse.data_ptr(), cl, B, H, Nq, Nk, d, int(bool(causal)),
                                 float(scale), ws_ptr, ws_bytes, _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd_decode")
    return o, lse


def fa_fwd(q, k, v, causal: bool = False, scale: float | None = None, o=None, lse=None, stream=None):
    """o, lse = softmax(q k^T * scale) v and its natural-log logsumexp.

    q, k, v: contiguous bf16 CUDA tensors [B, H, N, d] (d = 64 or 128).
    Returns (o [B, H, N, d] bf16, lse [B, H, N] fp32).
    """
    _check_qkv("q", q)
    B, H, N, d = q.shape
    _check_qkv("k", k, q.shape)
    _check_qkv("v", v, q.shape)
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if o is None:
        o = torch.empty_like(q)
    else:
        _check_qkv("o", o, q.shape)
    if lse is None:
        lse = torch.empty((B, H, N), device=q.device, dtype=torch.float32)
    elif lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, N] tensor")
    rc = library().fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                          B, H, N, d, int(bool(causal)), float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_fwd")
    return o, lse


def fa_bwd_workspace_bytes(B: int, H: int, N: int, d: int) -> int:
    return int(library().fa_bwd_workspace_bytes(B, H, N, d))


def fa_bwd(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None,
           dq=None, dk=None, dv=None, workspace=None, stream=None):
    """dq, dk, dv of a loss through o = attention(q, k, v), given dout and the saved lse.

    ``workspace`` may be a CUDA uint8 tensor of at least
    ``fa_bwd_workspace_bytes(B, H, N, d)`` bytes (256-byte aligned); if None
    the library allocates it on the stream.
    """
    _check_qkv("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_qkv(name, t, q.shape)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous() or not lse.is_cuda:
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [B, H, N]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, q.shape)
    ws_ptr, ws_bytes = None, 0
    if workspace is not None:
        if not workspace.is_cuda or not workspace.is_contiguous():
            raise ValueError("workspace must be a contiguous CUDA tensor")
        ws_ptr, ws_bytes = workspace.data_ptr(), workspace.numel() * workspace.element_size()
    rc = library().fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                          lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                          B, H, N, d, int(bool(causal)), float(scale), ws_ptr, ws_bytes,
                          _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd")
    return dq, dk, dv


def fa_bwd_noalloc(q, k, v, o, dout, lse, causal: bool = False, scale: float | None = None,
                   dq=None, dk=None, dv=None, stream=None):
    """fa_bwd for callers that cannot allocate device memory: the library's
    fixed scratch array replaces the workspace (see include/fa.h)."""
    _check_qkv("q", q)
    B, H, N, d = q.shape
    for name, t in (("k", k), ("v", v), ("o", o), ("dout", dout)):
        _check_qkv(name, t, q.shape)
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N) or not lse.is_contiguous() or not lse.is_cuda:
        raise ValueError("lse must be a contiguous fp32 CUDA tensor [B, H, N]")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        _check_qkv(name, t, q.shape)
    rc = library().fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), dout.data_ptr(),
                                  lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                  B, H, N, d, int(bool(causal)), float(scale), _stream_handle(stream))
    if rc != FA_OK:
        raise FaError(rc, "fa_bwd_noalloc")
    return dq, dk, dv


def fa_debug_time_next_bwd(start, mid, stop) -> None:
    """Have the next fa_bwd of this thread record three torch.cuda.Events:
    before its dK/dV kernel, between it and its dQ kernel, after the dQ kernel."""
    for e in (start, mid, stop):
        e.record()  # make sure torch has created the underlying CUDA events
    rc = library().fa_debug_time_next_bwd(start.cuda_event, mid.cuda_event, stop.cuda_event)
    if rc != FA_OK:
        raise FaError(rc, "fa_debug_time_next_bwd")


def fa_device_status(stream=None) -> int:
    """Synchronise the stream and return (and clear) the device status word."""
    return int(library().fa_device_status(_stream_handle(stream)))
