"""GB300 (sm_103a) scaled dot-product attention forward: Python binding.

This module only marshals arguments to the C ABI declared in include/attn.h
(``libattn.so`` next to this file): every step of the computation runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.  There is
no CPU path: when the library is missing, every call raises.

    attn_fwd(q, k, v, out=None, scale=None, causal=False, kv_len=None, stream=None)
    attn_decode(q, kcache, vcache, out=None, kv_len=None, stream=None)
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional

ATTN_F32 = 0
ATTN_BF16 = 1

ATTN_OK = 0
ATTN_EINVAL = -1
ATTN_EUNSUPPORTED = -2
ATTN_ECUDA = -3
ATTN_ENOMEM = -4
ATTN_ETIMEOUT = -5
ATTN_ECONFLICT = -6

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libattn.so")

# The exported functions, as declared in include/attn.h: name -> (restype, argtypes)
_vp, _i, _f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
SIGNATURES = {
    "attn_fwd": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _f, _i, _vp, _i, _vp]),
    "attn_fwd_gqa": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _i, _vp]),
    "attn_fwd_chunked": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _vp, _i, _vp]),
    "attn_fwd_host": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _i, _vp]),
    "attn_fwd_debug": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _f, _i, _vp, _i, _vp]),
    "attn_decode": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _i, _vp]),
    "attn_decode_gqa": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp, _i, _vp]),
    "attn_decode_noalloc": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _vp, _i, _vp]),
    "attn_decode_splits": (_i, [_i, _i, _i, _i]),
    "attn_device_status": (_i, [_vp]),
    "attn_last_error": (ctypes.c_char_p, []),
    "attn_release": (None, []),
    "attn_selftest_wait_timeout": (_i, [ctypes.c_longlong, _vp]),
}

_lib = None


class AttnError(RuntimeError):
    """A non-zero status from the library; ``code`` is the ATTN_E* value."""

    def __init__(self, code: int, message: str):
        super().__init__(f"[{code}] {message}")
        self.code = code


def lib(path: Optional[str] = None):
    """The loaded C library (ctypes handle with typed signatures)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"{LIB_PATH} is not built; run `python -m transformer_scaled_dot_fwd_gb300.build`")
        _lib = _bind(ctypes.CDLL(LIB_PATH))
    return _lib


def _bind(handle):
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(handle, name)
        fn.restype = res
        fn.argtypes = args
    return handle


def attn_last_error() -> str:
    return (lib().attn_last_error() or b"").decode(errors="replace")


def _check(rc: int):
    if rc != ATTN_OK:
        raise AttnError(rc, attn_last_error())


def _torch():
    import torch
    return torch


def _dtype_code(t):
    torch = _torch()
    if t.dtype == torch.bfloat16:
        return ATTN_BF16
    if t.dtype == torch.float32:
        return ATTN_F32
    raise TypeError(f"unsupported dtype {t.dtype} (bfloat16 or float32)")


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _stream_handle(stream):
    torch = _torch()
    if stream is None:
        stream = torch.cuda.current_stream()
    if isinstance(stream, torch.cuda.Stream):
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _check_tensor(name, t, ndim):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dim() != ndim:
        raise ValueError(f"{name} must be {ndim}-D")


def _kv_len_arg(kv_len, B, device):
    torch = _torch()
    if kv_len is None:
        return None
    if not (kv_len.is_cuda and kv_len.dtype == torch.int32 and kv_len.shape == (B,)
            and kv_len.is_contiguous() and kv_len.device == device):
        raise ValueError("kv_len must be a contiguous int32 CUDA tensor of shape (B,) on q's device")
    return kv_len


def attn_fwd(q, k, v, out=None, scale: Optional[float] = None, causal: bool = False,
             kv_len=None, stream=None):
    """Prefill attention of (B, H, Sq, D) queries against (B, H_kv, Skv, D)
    keys/values, H_kv dividing H (H_kv < H: grouped-query attention, calls
    attn_fwd_gqa).

    Returns ``out`` (allocated like q when not given).  See include/attn.h.
    """
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(name, t, 4)
    B, H, Sq, D = q.shape
    H_kv, Skv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, H_kv, Skv, D) or tuple(v.shape) != (B, H_kv, Skv, D) or H % H_kv:
        raise ValueError("k and v must be (B, H_kv, Skv, D) matching q, with H_kv dividing H")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    if out is None:
        out = _torch().empty_like(q)
    _check_tensor("out", out, 4)
    if tuple(out.shape) != tuple(q.shape) or out.dtype != q.dtype:
        raise ValueError("out must match q's shape and dtype")
    kl = _kv_len_arg(kv_len, B, q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    if H_kv == H:
        rc = lib().attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, Sq, Skv, D, float(scale),
                            int(bool(causal)), _ptr(kl), _dtype_code(q), _stream_handle(stream))
    else:
        rc = lib().attn_fwd_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, H_kv, Sq, Skv, D,
                                float(scale), int(bool(causal)), _ptr(kl), _dtype_code(q),
                                _stream_handle(stream))
    _check(rc)
    return out


def attn_fwd_host(q, k, v, out=None, scale: Optional[float] = None, causal: bool = False,
                  kv_len=None, stream=None):
    """attn_fwd with q, k, v, out in host memory (contiguous CPU tensors; pinned
    ones copy fastest): the library copies each chunk of heads in, computes it
    and copies it out, overlapping the three.  kv_len is a CPU int32 tensor of
    shape (B,) or a sequence of B ints.  Returns ``out`` (allocated like q,
    pinned if q is, when not given) once it holds the result.  See
    include/attn.h.
    """
    torch = _torch()
    for name, t in (("q", q), ("k", k), ("v", v)):
        if t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D CPU tensor")
    B, H, Sq, D = q.shape
    H_kv, Skv = k.shape[1], k.shape[2]
    if tuple(k.shape) != (B, H_kv, Skv, D) or tuple(v.shape) != (B, H_kv, Skv, D) or H % H_kv:
        raise ValueError("k and v must be (B, H_kv, Skv, D) matching q, with H_kv dividing H")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    if out is None:
        out = torch.empty(q.shape, dtype=q.dtype, pin_memory=q.is_pinned())
    if out.is_cuda or not out.is_contiguous() or tuple(out.shape) != tuple(q.shape) or out.dtype != q.dtype:
        raise ValueError("out must be a contiguous CPU tensor matching q")
    kl = None
    if kv_len is not None:
        kl = torch.as_tensor(kv_len, dtype=torch.int32).contiguous()
        if kl.is_cuda or tuple(kl.shape) != (B,):
            raise ValueError("kv_len must be B ints on the host")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib().attn_fwd_host(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, H, H_kv, Sq, Skv, D, float(scale),
                             int(bool(causal)), _ptr(kl), _dtype_code(q), _stream_handle(stream))
    _check(rc)
    return out


def attn_fwd_chunked(q, kcache, vcache, out=None, lse=None, scale: Optional[float] = None,
                     cache_len=None, return_lse: bool = False, stream=None):
    """Prefill of a chunk of (B, H, Sq, D) queries against a (B, H_kv, Skv, D)
    KV cache whose last positions hold the chunk's own keys/values: query i
    of sequence b sits at position cache_len[b] - Sq + i (causal).  Returns
    ``out``, or ``(out, lse)`` with the (B, H, Sq) fp32 log-sum-exp when
    ``return_lse`` (or an ``lse`` tensor) is given.  See include/attn.h.
    """
    for name, t in (("q", q), ("kcache", kcache), ("vcache", vcache)):
        _check_tensor(name, t, 4)
    B, H, Sq, D = q.shape
    H_kv, Skv = kcache.shape[1], kcache.shape[2]
    if (tuple(kcache.shape) != (B, H_kv, Skv, D) or tuple(vcache.shape) != (B, H_kv, Skv, D)
            or H % H_kv):
        raise ValueError("kcache and vcache must be (B, H_kv, Skv, D) matching q, with H_kv dividing H")
    if not (q.dtype == kcache.dtype == vcache.dtype):
        raise TypeError("q, kcache, vcache must share one dtype")
    torch = _torch()
    if out is None:
        out = torch.empty_like(q)
    _check_tensor("out", out, 4)
    if lse is None and return_lse:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if lse is not None:
        _check_tensor("lse", lse, 3)
        if tuple(lse.shape) != (B, H, Sq) or lse.dtype != torch.float32:
            raise ValueError("lse must be a float32 (B, H, Sq) tensor")
    cl = _kv_len_arg(cache_len, B, q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rc = lib().attn_fwd_chunked(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(out), _ptr(lse), B, H, H_kv,
                                Sq, Skv, D, float(scale), _ptr(cl), _dtype_code(q), _stream_handle(stream))
    _check(rc)
    return (out, lse) if lse is not None else out


def attn_fwd_debug(q, k, v, out=None, weights=None, scale: Optional[float] = None, causal: bool = False,
                   kv_len=None, return_weights: bool = False, stream=None):
    """General attention for inspection: q (B, H, Sq, Dk), k (B, H_kv, Skv, Dk),
    v (B, H_kv, Skv, Dv); returns out (B, H, Sq, Dv), or (out, weights) with
    the (B, H, Sq, Skv) fp32 attention weights.  See include/attn.h."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        _check_tensor(name, t, 4)
    B, H, Sq, Dk = q.shape
    H_kv, Skv, Dv = k.shape[1], k.shape[2], v.shape[3]
    if tuple(k.shape) != (B, H_kv, Skv, Dk) or tuple(v.shape[:3]) != (B, H_kv, Skv) or H % H_kv:
        raise ValueError("k must be (B, H_kv, Skv, Dk) and v (B, H_kv, Skv, Dv), with H_kv dividing H")
    if not (q.dtype == k.dtype == v.dtype):
        raise TypeError("q, k, v must share one dtype")
    torch = _torch()
    if out is None:
        out = torch.empty((B, H, Sq, Dv), dtype=q.dtype, device=q.device)
    _check_tensor("out", out, 4)
    if weights is None and return_weights:
        weights = torch.empty((B, H, Sq, Skv), dtype=torch.float32, device=q.device)
    if weights is not None:
        _check_tensor("weights", weights, 4)
    kl = _kv_len_arg(kv_len, B, q.device)
    if scale is None:
        scale = 1.0 / math.sqrt(Dk)
    rc = lib().attn_fwd_debug(_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(weights), B, H, H_kv, Sq, Skv,
                              Dk, Dv, float(scale), int(bool(causal)), _ptr(kl), _dtype_code(q),
                              _stream_handle(stream))
    _check(rc)
    return (out, weights) if weights is not None else out


def attn_decode(q, kcache, vcache, out=None, kv_len=None, stream=None):
    """One query per (batch, head): q (B, H, D) against a (B, H_kv, Skv, D)
    cache, H_kv dividing H (H_kv < H: grouped-query decode, attn_decode_gqa).

    Returns ``out`` (B, H, D).  See include/attn.h.
    """
    _check_tensor("q", q, 3)
    _check_tensor("kcache", kcache, 4)
    _check_tensor("vcache", vcache, 4)
    B, H, D = q.shape
    H_kv, Skv = kcache.shape[1], kcache.shape[2]
    if (tuple(kcache.shape) != (B, H_kv, Skv, D) or tuple(vcache.shape) != (B, H_kv, Skv, D)
            or H % H_kv):
        raise ValueError("kcache and vcache must be (B, H_kv, Skv, D) matching q, with H_kv dividing H")
    if not (q.dtype == kcache.dtype == vcache.dtype):
        raise TypeError("q, kcache, vcache must share one dtype")
    if out is None:
        out = _torch().empty_like(q)
    _check_tensor("out", out, 3)
    kl = _kv_len_arg(kv_len, B, q.device)
    if H_kv == H:
        rc = lib().attn_decode(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(out), B, H, Skv, D, _ptr(kl),
                               _dtype_code(q), _stream_handle(stream))
    else:
        rc = lib().attn_decode_gqa(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(out), B, H, H_kv, Skv, D,
                                   _ptr(kl), _dtype_code(q), _stream_handle(stream))
    _check(rc)
    return out


def attn_decode_noalloc(q, kcache, vcache, out, kv_len=None, stream=None):
    """attn_decode without any device allocation (see include/attn.h): the
    caller supplies ``out``; the scratch is a fixed array inside the library."""
    _check_tensor("q", q, 3)
    _check_tensor("kcache", kcache, 4)
    _check_tensor("vcache", vcache, 4)
    _check_tensor("out", out, 3)
    B, H, D = q.shape
    Skv = kcache.shape[2]
    if tuple(kcache.shape) != (B, H, Skv, D) or tuple(vcache.shape) != (B, H, Skv, D):
        raise ValueError("kcache and vcache must be (B, H, Skv, D) matching q")
    if tuple(out.shape) != (B, H, D) or not (q.dtype == kcache.dtype == vcache.dtype == out.dtype):
        raise ValueError("out must be (B, H, D) and every tensor must share q's dtype")
    kl = _kv_len_arg(kv_len, B, q.device)
    rc = lib().attn_decode_noalloc(_ptr(q), _ptr(kcache), _ptr(vcache), _ptr(out), B, H, Skv, D, _ptr(kl),
                                   _dtype_code(q), _stream_handle(stream))
    _check(rc)
    return out


def attn_decode_splits(B: int, H: int, Skv: int, D: int) -> int:
    return lib().attn_decode_splits(B, H, Skv, D)


def attn_device_status(stream=None) -> None:
    """Synchronise the stream and raise AttnError if a kernel reported a timed-out
    wait (ATTN_ETIMEOUT) or a shared prefill work counter (ATTN_ECONFLICT)."""
    _check(lib().attn_device_status(_stream_handle(stream)))


def attn_selftest_wait_timeout(limit_cycles: int = 1_000_000, stream=None) -> None:
    """Enqueue the diagnostic kernel whose wait runs out (see include/attn.h)."""
    _check(lib().attn_selftest_wait_timeout(int(limit_cycles), _stream_handle(stream)))


def attn_release() -> None:
    lib().attn_release()


__all__ = [
    "attn_fwd", "attn_fwd_chunked", "attn_fwd_debug", "attn_fwd_host", "attn_decode", "attn_decode_noalloc", "attn_decode_splits", "attn_device_status", "attn_release",
    "attn_last_error", "attn_selftest_wait_timeout", "lib", "AttnError", "SIGNATURES", "LIB_PATH",
    "ATTN_F32", "ATTN_BF16", "ATTN_OK", "ATTN_EINVAL", "ATTN_EUNSUPPORTED", "ATTN_ECUDA",
    "ATTN_ENOMEM", "ATTN_ETIMEOUT", "ATTN_ECONFLICT",
]
