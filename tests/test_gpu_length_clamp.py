"""GPU parity tests of the length contract's edges: kv_len / cache_len values
below 0 and above Skv.

include/attn.h promises that each length is clamped to [0, Skv] inside the
kernels (no host synchronisation), and the oracle clamps the same way (its pin
'lengths outside range are clamped' ties that to PyTorch's float64 SDPA).  The
padding mask itself ("Attention from Scratch" (kube-dojo), Part 3) is defined
only for valid lengths, so this edge is the library's own contract: a length
above Skv means every key is valid, a negative one means none is.  Every
entry point that reads a length array is covered: prefill (tensor cores and
fp32), the chunk against a cache, and decode on each of its kernels (multi-head,
grouped CUDA-core, grouped tensor-core, fp32, and the no-allocation entry).
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_fwd_gb300 as attn
from transformer_scaled_dot_fwd_gb300 import workloads as wl
from helpers import assert_close

pytestmark = pytest.mark.gpu

DTYPES = [torch.bfloat16, torch.float32]


def _lens(Skv):
    # above the capacity (small and large excess), negative, and valid ones around a tile edge
    return [Skv + 1, Skv + 1000, -1, -(1 << 30), 129, Skv, 0, 2 ** 31 - 1]


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("D", [64, 128])
def test_prefill_clamps_lengths(gpu, dtype, causal, D):
    S = 300
    lens = _lens(S)
    B, H = len(lens), 2
    q = wl.random_tensors((B, H, S, D), 700 + D, dtype=dtype, count=1)[0]
    k, v = wl.random_tensors((B, H, S, D), 701 + D, dtype=dtype, count=2)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = attn.attn_fwd(q, k, v, causal=causal, kv_len=kl)
    attn.attn_device_status()
    ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=causal, kv_len=np.array(lens, np.int32))
    assert_close(out, ref, dtype, f"prefill lengths outside [0, Skv], causal={causal} D={D}")
    # the clamped lengths give exactly the in-range calls' results
    clamped = torch.tensor([min(max(L, 0), S) for L in lens], dtype=torch.int32, device="cuda")
    assert torch.equal(out, attn.attn_fwd(q, k, v, causal=causal, kv_len=clamped))
    for b, L in enumerate(lens):
        if L <= 0:
            assert torch.count_nonzero(out[b]) == 0


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("H,H_kv", [(4, 4), (4, 1)])
def test_chunk_clamps_cache_lengths(gpu, dtype, H, H_kv):
    Sq, Skv, D = 130, 600, 128
    lens = _lens(Skv)
    B = len(lens)
    q = wl.random_tensors((B, H, Sq, D), 710, dtype=dtype, count=1)[0]
    kc, vc = wl.random_tensors((B, H_kv, Skv, D), 711, dtype=dtype, count=2)
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out, lse = attn.attn_fwd_chunked(q, kc, vc, cache_len=cl, return_lse=True)
    attn.attn_device_status()
    ref, ref_lse = oracle.attention(q.cpu(), kc.cpu(), vc.cpu(), causal=True,
                                    cache_len=np.array(lens, np.int32), need_lse=True)
    assert_close(out, ref, dtype, f"chunk with cache lengths outside [0, Skv], H={H} H_kv={H_kv}")
    got = lse.double().cpu().numpy()
    assert np.array_equal(np.isinf(got), np.isinf(ref_lse))
    fin = ~np.isinf(ref_lse)
    assert np.abs(got[fin] - ref_lse[fin]).max() <= (2e-4 if dtype == torch.bfloat16 else 2e-5)
    for b, L in enumerate(lens):
        if L <= 0:
            assert torch.count_nonzero(out[b]) == 0


@pytest.mark.parametrize("dtype,H,H_kv", [(torch.bfloat16, 8, 8),   # multi-head split-KV kernel
                                          (torch.bfloat16, 8, 4),   # grouped, CUDA cores (G = 2)
                                          (torch.bfloat16, 8, 1),   # grouped, tensor cores (G = 8)
                                          (torch.float32, 8, 2)])   # fp32 kernel
def test_decode_clamps_lengths(gpu, dtype, H, H_kv):
    Skv, D = 1000, 128
    lens = _lens(Skv)
    B = len(lens)
    q = wl.random_tensors((B, H, D), 720 + H_kv, dtype=dtype, count=1)[0]
    kc, vc = wl.random_tensors((B, H_kv, Skv, D), 721 + H_kv, dtype=dtype, count=2)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = attn.attn_decode(q, kc, vc, kv_len=kl)
    attn.attn_device_status()
    ref = oracle.decode(q.cpu(), kc.cpu(), vc.cpu(), kv_len=np.array(lens, np.int32))
    assert_close(out, ref, dtype, f"decode lengths outside [0, Skv], H={H} H_kv={H_kv}")
    for b, L in enumerate(lens):
        if L <= 0:
            assert torch.count_nonzero(out[b]) == 0
    if H_kv == H:
        got = attn.attn_decode_noalloc(q, kc, vc, torch.empty_like(q), kv_len=kl)
        attn.attn_device_status()
        assert_close(got, ref, dtype, "no-allocation decode, lengths outside [0, Skv]")
