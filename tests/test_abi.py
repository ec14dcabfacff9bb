"""Host-side tests of the C ABI that need no GPU: the library loads, exports
every function include/attn.h declares, and rejects bad arguments before any
CUDA call (so these run on a machine without a GPU)."""
from __future__ import annotations

import ctypes
import os
import re

import pytest

import transformer_scaled_dot_fwd_gb300 as attn

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn.h")


def declared_functions():
    text = open(HEADER).read()
    return re.findall(r"ATTN_API\s+[\w\s\*]+?\b(attn_\w+)\s*\(", text)


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("attn_fwd", "attn_decode", "attn_last_error", "attn_release",
                 "attn_decode_splits", "attn_device_status"):
        assert must in names


def test_library_exports_every_declared_symbol(attn_lib):
    for name in declared_functions():
        assert hasattr(attn_lib, name), f"{name} declared in attn.h but not exported"
    assert set(declared_functions()) == set(attn.SIGNATURES), "binding and header disagree"


def test_status_codes_match_header():
    text = open(HEADER).read()
    for name in ("ATTN_OK", "ATTN_EINVAL", "ATTN_EUNSUPPORTED", "ATTN_ECUDA", "ATTN_ENOMEM",
                 "ATTN_ETIMEOUT", "ATTN_ECONFLICT", "ATTN_F32", "ATTN_BF16"):
        m = re.search(rf"#define\s+{name}\s+\(?(-?\d+)\)?", text)
        assert m, name
        assert int(m.group(1)) == getattr(attn, name)


# Fake, distinct, 16-byte-aligned addresses: validation rejects the call before
# anything is dereferenced or any CUDA call is made.
Q, K, V, O, KL = (ctypes.c_void_p(0x10000000 * (i + 1)) for i in range(5))


def fwd(lib, q=Q, k=K, v=V, o=O, B=2, H=2, Sq=16, Skv=16, D=128, scale=0.125, causal=1, kl=None,
        dtype=attn.ATTN_BF16):
    return lib.attn_fwd(q, k, v, o, B, H, Sq, Skv, D, scale, causal, kl, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), attn.ATTN_EINVAL),
    (dict(o=None), attn.ATTN_EINVAL),
    (dict(B=0), attn.ATTN_EINVAL),
    (dict(H=-1), attn.ATTN_EINVAL),
    (dict(Sq=-3), attn.ATTN_EINVAL),
    (dict(D=0), attn.ATTN_EINVAL),
    (dict(D=96), attn.ATTN_EUNSUPPORTED),
    (dict(D=256), attn.ATTN_EUNSUPPORTED),
    (dict(dtype=7), attn.ATTN_EINVAL),
    (dict(scale=float("nan")), attn.ATTN_EINVAL),
    (dict(scale=float("inf")), attn.ATTN_EINVAL),
    (dict(scale=-1.0), attn.ATTN_EINVAL),
    (dict(causal=2), attn.ATTN_EINVAL),
    (dict(Sq=17, Skv=16), attn.ATTN_EINVAL),                 # causal with Sq > Skv
    (dict(causal=1, Sq=8, kl=KL), attn.ATTN_EINVAL),         # causal kv_len needs Sq == Skv
    (dict(q=ctypes.c_void_p(0x10000008)), attn.ATTN_EINVAL),  # misaligned
    (dict(kl=ctypes.c_void_p(0x50000002)), attn.ATTN_EINVAL),
    (dict(o=ctypes.c_void_p(0x10000000 + 4096)), attn.ATTN_EINVAL),  # out overlaps q
    (dict(B=1 << 16, H=1 << 16), attn.ATTN_EINVAL),          # too many rows
])
def test_fwd_rejects_bad_arguments(attn_lib, kw, code):
    assert fwd(attn_lib, **kw) == code
    assert attn.attn_last_error() != ""


def test_fwd_empty_query_is_a_no_op(attn_lib):
    assert fwd(attn_lib, Sq=0, causal=0) == attn.ATTN_OK
    assert attn.attn_last_error() == ""


def dec(lib, q=Q, k=K, v=V, o=O, B=2, H=2, Skv=64, D=128, kl=None, dtype=attn.ATTN_BF16):
    return lib.attn_decode(q, k, v, o, B, H, Skv, D, kl, dtype, None)


@pytest.mark.parametrize("kw,code", [
    (dict(k=None), attn.ATTN_EINVAL),
    (dict(B=0), attn.ATTN_EINVAL),
    (dict(Skv=-1), attn.ATTN_EINVAL),
    (dict(D=-4), attn.ATTN_EINVAL),
    (dict(D=80), attn.ATTN_EUNSUPPORTED),
    (dict(dtype=attn.ATTN_F32, D=80), attn.ATTN_EUNSUPPORTED),
    (dict(dtype=3), attn.ATTN_EINVAL),
    (dict(v=ctypes.c_void_p(0x30000004)), attn.ATTN_EINVAL),
    (dict(o=ctypes.c_void_p(0x10000000 + 256)), attn.ATTN_EINVAL),
])
def test_decode_rejects_bad_arguments(attn_lib, kw, code):
    assert dec(attn_lib, **kw) == code
    assert attn.attn_last_error() != ""


def test_decode_splits_cover_the_cache(attn_lib):
    for B, H, Skv in ((64, 32, 8192), (1, 1, 100), (2, 4, 0), (1, 32, 65536)):
        n = attn_lib.attn_decode_splits(B, H, Skv, 128)
        assert n >= 1
        if Skv:
            chunk = -(-Skv // n)
            assert chunk <= 1024 and n * 1024 >= Skv
    assert attn_lib.attn_decode_splits(0, 1, 10, 128) == attn.ATTN_EINVAL


def test_binding_refuses_cpu_tensors(attn_lib):
    import torch
    x = torch.zeros(1, 1, 4, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd(x, x, x)
    with pytest.raises(ValueError):
        attn.attn_decode(x[:, :, 0], x, x)


def test_product_path_does_not_import_the_oracle():
    import subprocess
    import sys
    code = ("import sys, transformer_scaled_dot_fwd_gb300, transformer_scaled_dot_fwd_gb300.workloads;"
            "bad=[m for m in sys.modules if m == 'oracle' or m.startswith('oracle.')];"
            "print(bad); sys.exit(1 if bad else 0)")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    src_dir = os.path.join(ROOT, "transformer_scaled_dot_fwd_gb300")
    for dirpath, _, files in os.walk(src_dir):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b|liboracle|oracle\.c", text, re.M), \
                    f"{f} loads the oracle"


def test_new_entry_points_reject_bad_arguments(attn_lib):
    """Grouped-query, chunked and debug entry points validate on the host
    before any CUDA call (fake pointers are never dereferenced)."""
    f, i = ctypes.c_float, attn.ATTN_EINVAL
    # attn_fwd_gqa: H_kv must divide H
    assert attn_lib.attn_fwd_gqa(Q, K, V, O, 2, 6, 4, 16, 16, 128, f(0.1), 1, None, attn.ATTN_BF16, None) == i
    assert attn_lib.attn_fwd_gqa(Q, K, V, O, 2, 6, 0, 16, 16, 128, f(0.1), 1, None, attn.ATTN_BF16, None) == i
    # attn_fwd_chunked: the chunk cannot be longer than the cache
    assert attn_lib.attn_fwd_chunked(Q, K, V, O, None, 2, 4, 2, 17, 16, 128, f(0.1), None,
                                     attn.ATTN_BF16, None) == i
    # attn_fwd_chunked: lse must be 4-byte aligned and must not overlap out
    assert attn_lib.attn_fwd_chunked(Q, K, V, O, ctypes.c_void_p(0x60000002), 2, 4, 2, 8, 16, 128, f(0.1),
                                     None, attn.ATTN_BF16, None) == i
    assert attn_lib.attn_fwd_chunked(Q, K, V, O, O, 2, 4, 2, 8, 16, 128, f(0.1), None,
                                     attn.ATTN_BF16, None) == i
    # attn_fwd_debug: head depths and key count bounds
    assert attn_lib.attn_fwd_debug(Q, K, V, O, None, 1, 2, 2, 4, 7, 257, 2, f(0.5), 0, None,
                                   attn.ATTN_F32, None) == i
    assert attn_lib.attn_fwd_debug(Q, K, V, O, None, 1, 2, 2, 4, 7, 4, 0, f(0.5), 0, None,
                                   attn.ATTN_F32, None) == i
    assert attn_lib.attn_fwd_debug(Q, K, V, O, None, 1, 2, 2, 4, 16385, 4, 2, f(0.5), 0, None,
                                   attn.ATTN_F32, None) == attn.ATTN_EUNSUPPORTED
    assert attn_lib.attn_fwd_debug(Q, K, V, O, None, 1, 2, 2, 8, 4, 4, 2, f(0.5), 1, None,
                                   attn.ATTN_F32, None) == i  # causal with Sq > Skv
    # attn_decode_gqa: H_kv must divide H
    assert attn_lib.attn_decode_gqa(Q, K, V, O, 2, 8, 3, 64, 128, None, attn.ATTN_BF16, None) == i
    assert attn.attn_last_error() != ""
    # attn_fwd_host: the same checks, before any device work
    assert attn_lib.attn_fwd_host(Q, K, V, O, 2, 6, 4, 16, 16, 128, f(0.1), 1, None, attn.ATTN_BF16, None) == i
    assert attn_lib.attn_fwd_host(None, K, V, O, 2, 4, 4, 16, 16, 128, f(0.1), 1, None, attn.ATTN_BF16, None) == i
    assert attn_lib.attn_fwd_host(Q, K, V, O, 2, 4, 4, 17, 16, 128, f(0.1), 1, None, attn.ATTN_BF16, None) == i
    assert attn_lib.attn_fwd_host(Q, K, V, O, 2, 4, 4, 8, 16, 128, f(0.1), 1, Q, attn.ATTN_BF16, None) == i
    assert attn_lib.attn_fwd_host(Q, K, V, Q, 2, 4, 4, 16, 16, 128, f(0.1), 1, None, attn.ATTN_BF16, None) == i
    assert attn_lib.attn_fwd_host(Q, K, V, O, 2, 4, 4, 16, 16, 96, f(0.1), 1, None,
                                  attn.ATTN_BF16, None) == attn.ATTN_EUNSUPPORTED
    assert attn_lib.attn_fwd_host(Q, K, V, O, 2, 4, 4, 0, 16, 128, f(0.1), 0, None, attn.ATTN_BF16, None) == 0
