"""Seeded random configurations of every fast entry point against the oracle.

The parametrised tests elsewhere walk each axis on its own; here each case
draws all of them at once -- batch, heads and key/value grouping, query and key
lengths (tile-aligned, one off, ragged), head size, dtype, causal or not,
per-sequence lengths (including 0 and values outside [0, Skv]), scale -- for
prefill (`attn_fwd`), a chunk against a cache (`attn_fwd_chunked`, with the
row log-sum-exp) and decode (`attn_decode`), and compares with the fp64 oracle
at the standard tolerances (bf16: max 2e-2, mean 2e-3; fp32: max 1e-4).
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_fwd_gb300 as attn
from transformer_scaled_dot_fwd_gb300 import workloads as wl
from helpers import assert_close

pytestmark = pytest.mark.gpu

N_CASES = 48


def _length(rng, lo, hi):
    """A length in [lo, hi], biased towards tile edges (multiples of 128 +- 1)."""
    if rng.random() < 0.4:
        t = int(rng.integers(0, hi // 128 + 1)) * 128 + int(rng.integers(-1, 2))
        return int(min(max(t, lo), hi))
    return int(rng.integers(lo, hi + 1))


def _heads(rng):
    H = int(rng.choice([1, 2, 3, 4, 6, 8]))
    divisors = [d for d in range(1, H + 1) if H % d == 0]
    return H, int(rng.choice(divisors))


def _dtype(rng):
    return torch.float32 if rng.random() < 0.25 else torch.bfloat16


@pytest.mark.parametrize("case", range(N_CASES))
def test_prefill_fuzz(gpu, case):
    rng = np.random.default_rng(1000 + case)
    B = int(rng.integers(1, 4))
    H, H_kv = _heads(rng)
    D = int(rng.choice([64, 128]))
    dtype = _dtype(rng)
    causal = bool(rng.random() < 0.6)
    Skv = _length(rng, 1, 700)
    padded = rng.random() < 0.5
    if causal and padded:
        Sq = Skv  # causal key padding is self-attention over a right-padded batch
    elif causal:
        Sq = _length(rng, 1, Skv)
    else:
        Sq = _length(rng, 1, 700)
    kv = None
    if padded:
        lens = rng.integers(-3, Skv + 4, B)  # values outside [0, Skv] are clamped
        kv = torch.tensor(lens, dtype=torch.int32, device="cuda")
    scale = float(rng.choice([1.0 / math.sqrt(D), 0.05, 0.3]))
    q = wl.random_tensors((B, H, Sq, D), 2000 + case, count=1, dtype=dtype)[0]
    k, v = wl.random_tensors((B, H_kv, Skv, D), 3000 + case, count=2, dtype=dtype)
    out = attn.attn_fwd(q, k, v, scale=scale, causal=causal, kv_len=kv)
    attn.attn_device_status()
    ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale=scale, causal=causal,
                           kv_len=None if kv is None else kv.cpu().numpy())
    assert_close(out, ref, dtype, f"prefill case {case}: B{B} H{H}/{H_kv} Sq{Sq} Skv{Skv} D{D} "
                                  f"{dtype} causal={causal} lens={None if kv is None else kv.tolist()}")


@pytest.mark.parametrize("case", range(N_CASES // 2))
def test_chunked_fuzz(gpu, case):
    rng = np.random.default_rng(5000 + case)
    B = int(rng.integers(1, 4))
    H, H_kv = _heads(rng)
    D = int(rng.choice([64, 128]))
    dtype = _dtype(rng)
    Skv = _length(rng, 1, 700)
    Sq = _length(rng, 1, Skv)
    lens = rng.integers(Sq, Skv + 1, B) if rng.random() < 0.7 else None
    q = wl.random_tensors((B, H, Sq, D), 6000 + case, count=1, dtype=dtype)[0]
    kc, vc = wl.random_tensors((B, H_kv, Skv, D), 7000 + case, count=2, dtype=dtype)
    cl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    out, lse = attn.attn_fwd_chunked(q, kc, vc, cache_len=cl, return_lse=True)
    attn.attn_device_status()
    ref, ref_lse = oracle.attention(q.cpu(), kc.cpu(), vc.cpu(), causal=True, need_lse=True,
                                    cache_len=None if lens is None else np.asarray(lens, np.int32))
    what = f"chunk case {case}: B{B} H{H}/{H_kv} Sq{Sq} Skv{Skv} D{D} {dtype} lens={lens}"
    assert_close(out, ref, dtype, what)
    tol = 1e-4 if dtype == torch.float32 else 2e-3
    assert np.max(np.abs(lse.cpu().double().numpy() - ref_lse)) <= tol, what + " (lse)"


@pytest.mark.parametrize("case", range(N_CASES // 2))
def test_decode_fuzz(gpu, case):
    rng = np.random.default_rng(8000 + case)
    B = int(rng.integers(1, 6))
    H = int(rng.choice([1, 4, 8, 16, 32]))
    H_kv = int(rng.choice([d for d in (1, 2, 4, 8, 16, 32) if d <= H and H % d == 0]))
    D = int(rng.choice([64, 128]))
    dtype = _dtype(rng)
    Skv = _length(rng, 1, 5000)
    lens = rng.integers(-2, Skv + 3, B) if rng.random() < 0.7 else None
    q = wl.random_tensors((B, H, D), 9000 + case, count=1, dtype=dtype)[0]
    kc, vc = wl.random_tensors((B, H_kv, Skv, D), 9500 + case, count=2, dtype=dtype)
    kl = None if lens is None else torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = attn.attn_decode(q, kc, vc, kv_len=kl)
    attn.attn_device_status()
    ref = oracle.decode(q.cpu(), kc.cpu(), vc.cpu(), kv_len=None if lens is None else np.asarray(lens, np.int32))
    assert_close(out, ref, dtype, f"decode case {case}: B{B} H{H}/{H_kv} Skv{Skv} D{D} {dtype} lens={lens}")
