"""fp64 CPU oracle for scaled dot-product attention (test infrastructure only).

This package is the checker, not the product: only the tests, the smoke check
and the benchmark's CPU-baseline leg load it.  It shares no code with the CUDA
library and imports nothing from it.

The arithmetic lives in ``oracle.c`` (plain C, double precision, one score row
materialised per query); this module only builds that file with gcc and
marshals numpy / torch-CPU arrays into it.  Definition and the readings taken
where the pages are silent are stated at the top of ``oracle.c``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F32 = 0
BF16 = 1

_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB) -> str:
    """Compile oracle.c into a shared library with gcc (OpenMP over (b, h))."""
    if force or not os.path.exists(out) or os.path.getmtime(out) < os.path.getmtime(src):
        tmp = out + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c99", src, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, out)
    return out


def load(path: Optional[str] = None):
    """Load (building if needed) the oracle library; returns the ctypes handle."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _bind(lib):
    vp, dp, i32p = ctypes.c_void_p, ctypes.POINTER(ctypes.c_double), ctypes.c_void_p
    lib.oracle_attention_gqa.restype = ctypes.c_int
    lib.oracle_attention_gqa.argtypes = [vp, vp, vp, ctypes.c_int, dp, dp] + [ctypes.c_int] * 7 + [
        ctypes.c_double, ctypes.c_int, i32p, ctypes.c_int, ctypes.c_int]
    lib.oracle_attention_cache.restype = ctypes.c_int
    lib.oracle_attention_cache.argtypes = [vp, vp, vp, ctypes.c_int, dp, dp] + [ctypes.c_int] * 7 + [
        ctypes.c_double, i32p, ctypes.c_int]
    lib.oracle_attention_rows_gqa.restype = ctypes.c_int
    lib.oracle_attention_rows_gqa.argtypes = [vp, vp, vp, ctypes.c_int, dp] + [ctypes.c_int] * 7 + [
        ctypes.c_double, ctypes.c_int, i32p, ctypes.c_int, vp, ctypes.c_longlong, ctypes.c_int]
    return lib


def _threads(nthreads: Optional[int]) -> int:
    if nthreads is not None and nthreads > 0:
        return int(nthreads)
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _as_storage(x):
    """Return (contiguous numpy array, dtype code) holding the exact stored values.

    Accepts numpy float32/float64 arrays and torch CPU tensors (float32,
    bfloat16, float64).  bfloat16 is passed as its raw 16-bit patterns; float64
    is narrowed to float32 only if that is exact.
    """
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    if torch is not None and isinstance(x, torch.Tensor):
        x = x.detach().cpu().contiguous()
        if x.dtype == torch.bfloat16:
            return x.view(torch.int16).numpy().view(np.uint16), BF16
        x = x.numpy()
    x = np.ascontiguousarray(x)
    if x.dtype == np.float32:
        return x, F32
    if x.dtype == np.float64:
        x32 = x.astype(np.float32)
        if not np.array_equal(x32.astype(np.float64), x):
            raise ValueError("float64 input is not exactly representable in float32")
        return x32, F32
    raise TypeError(f"unsupported oracle input dtype {x.dtype}")


def _kv_len_array(kv_len, B):
    if kv_len is None:
        return None
    a = np.ascontiguousarray(np.asarray(
        kv_len.cpu().numpy() if hasattr(kv_len, "cpu") else kv_len, dtype=np.int32))
    if a.shape != (B,):
        raise ValueError("kv_len must have shape (B,)")
    return a


def attention(q, k, v, scale=None, causal=False, kv_len=None, query_padding=None,
              need_weights=False, nthreads=None, lib=None, cache_len=None, need_lse=False):
    """Attention of (B, H, Sq, Dk) queries against (B, Hkv, Skv, Dk) keys and
    (B, Hkv, Skv, Dv) values, Hkv dividing H: query head h uses key/value head
    h // (H // Hkv) (grouped-query attention; Hkv == H is multi-head attention).

    Returns out (B, H, Sq, Dv) float64, plus the (B, H, Sq, Skv) weights when
    ``need_weights``.  ``scale`` defaults to 1/sqrt(Dk).  ``query_padding``
    defaults to True when kv_len is given and Sq == Skv (self-attention
    prefill over a right-padded batch).  ``lib`` selects another build of
    oracle.c (the test suite uses it to run planted mistakes against the pins).

    ``cache_len`` (int32[B]) or ``need_lse`` selects prefill of a chunk against
    a KV cache instead: sequence b has cache_len[b] valid positions (all Skv
    when None), query i sits at position cache_len[b] - Sq + i and sees keys up
    to it (causal, no query padding); with ``need_lse`` the (B, H, Sq)
    log-sum-exp of each row's visible scores is returned too.
    """
    qa, dt = _as_storage(q)
    ka, dt_k = _as_storage(k)
    va, dt_v = _as_storage(v)
    if not (dt == dt_k == dt_v):
        raise TypeError("q, k, v must share one dtype")
    if qa.ndim != 4 or ka.ndim != 4 or va.ndim != 4:
        raise ValueError("q, k, v must be 4-D (B, H, S, D)")
    B, H, Sq, Dk = qa.shape
    Hkv, Skv, Dv = ka.shape[1], ka.shape[2], va.shape[3]
    if ka.shape != (B, Hkv, Skv, Dk) or va.shape[:3] != (B, Hkv, Skv) or Hkv < 1 or H % Hkv:
        raise ValueError("shape mismatch between q, k, v")
    if scale is None:
        scale = 1.0 / np.sqrt(Dk)
    lib = lib or load()
    if cache_len is not None or need_lse:
        if kv_len is not None or need_weights or not causal:
            raise ValueError("the cache form is causal and takes cache_len, not kv_len or weights")
        cl = _kv_len_array(cache_len, B)
        out = np.zeros((B, H, Sq, Dv), dtype=np.float64)
        lse = np.zeros((B, H, Sq), dtype=np.float64)
        rc = lib.oracle_attention_cache(
            qa.ctypes.data, ka.ctypes.data, va.ctypes.data, dt,
            out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            lse.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
            B, H, Hkv, Sq, Skv, Dk, Dv, float(scale), cl.ctypes.data if cl is not None else None,
            _threads(nthreads))
        if rc != 0:
            raise ValueError("oracle_attention_cache rejected its arguments")
        return (out, lse) if need_lse else out
    kl = _kv_len_array(kv_len, B)
    if query_padding is None:
        query_padding = kl is not None and Sq == Skv
    out = np.zeros((B, H, Sq, Dv), dtype=np.float64)
    w = np.zeros((B, H, Sq, Skv), dtype=np.float64) if need_weights else None
    rc = lib.oracle_attention_gqa(
        qa.ctypes.data, ka.ctypes.data, va.ctypes.data, dt,
        out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
        w.ctypes.data_as(ctypes.POINTER(ctypes.c_double)) if w is not None else None,
        B, H, Hkv, Sq, Skv, Dk, Dv, float(scale), int(bool(causal)),
        kl.ctypes.data if kl is not None else None, int(bool(query_padding)),
        _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_attention_gqa rejected its arguments")
    return (out, w) if need_weights else out


def attention_rows(q, k, v, rows, scale=None, causal=False, kv_len=None, query_padding=None,
                   nthreads=None, lib=None):
    """The oracle at selected rows only: ``rows`` is an (n, 3) int array of (b, h, i).

    Returns an (n, Dv) float64 array.
    """
    qa, dt = _as_storage(q)
    ka, _ = _as_storage(k)
    va, _ = _as_storage(v)
    B, H, Sq, Dk = qa.shape
    Hkv, Skv, Dv = ka.shape[1], ka.shape[2], va.shape[3]
    if scale is None:
        scale = 1.0 / np.sqrt(Dk)
    kl = _kv_len_array(kv_len, B)
    if query_padding is None:
        query_padding = kl is not None and Sq == Skv
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 3))
    out = np.zeros((r.shape[0], Dv), dtype=np.float64)
    lib = lib or load()
    rc = lib.oracle_attention_rows_gqa(
        qa.ctypes.data, ka.ctypes.data, va.ctypes.data, dt,
        out.ctypes.data_as(ctypes.POINTER(ctypes.c_double)),
        B, H, Hkv, Sq, Skv, Dk, Dv, float(scale), int(bool(causal)),
        kl.ctypes.data if kl is not None else None, int(bool(query_padding)),
        r.ctypes.data, int(r.shape[0]), _threads(nthreads))
    if rc != 0:
        raise ValueError("oracle_attention_rows_gqa rejected its arguments")
    return out


def decode(q, kcache, vcache, kv_len=None, scale=None, nthreads=None):
    """Single-query decode: q (B, H, D) against a (B, Hkv, Skv, D) cache.

    The query sees every cached key j < L_b ("Scaled dot-product attention with
    masking", "Adding the causal mask": no mask for seq_q = 1).  Returns (B, H, D).
    """
    qa, _ = _as_storage(q)
    B, H, D = qa.shape
    q4 = q.reshape(B, H, 1, D) if hasattr(q, "reshape") else qa.reshape(B, H, 1, D)
    out = attention(q4, kcache, vcache, scale=scale, causal=False, kv_len=kv_len,
                    query_padding=False, nthreads=nthreads)
    return out.reshape(B, H, -1)
