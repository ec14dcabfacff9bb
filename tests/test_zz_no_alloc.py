"""GPU test of attn_decode_noalloc, the decode entry point that never
allocates device memory (for callers that have reserved all device memory up
front, or cannot afford the device synchronisation an allocation may cause).

It is called through the C ABI with raw device pointers and compared with the
regular attn_decode on the same inputs, on two calls in a row with different
sizes (the second call must not be disturbed by what the first left in the
library's fixed scratch), and both are held to the fp64 oracle as well.  This
file is named to be collected last.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_fwd_gb300 as attn
from transformer_scaled_dot_fwd_gb300 import workloads as wl
from helpers import BF16_MAX, BF16_MEAN, assert_close

pytestmark = pytest.mark.gpu

P = ctypes.c_void_p


def _inputs(B, H, Skv, D, lens, seed):
    q = wl.random_tensors((B, H, D), seed, count=1)[0]
    kc, vc = wl.random_tensors((B, H, Skv, D), seed + 1, count=2)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    return q, kc, vc, kl


def _noalloc(lib, q, kc, vc, kl, out):
    B, H, D = q.shape
    Skv = kc.shape[2]
    stream = P(torch.cuda.current_stream().cuda_stream)
    return lib.attn_decode_noalloc(P(q.data_ptr()), P(kc.data_ptr()), P(vc.data_ptr()), P(out.data_ptr()),
                                   B, H, Skv, D, P(kl.data_ptr()), attn.ATTN_BF16, stream)


def test_noalloc_matches_decode_on_two_calls(gpu):
    lib = attn.lib()
    cases = [(4, 8, 3000, 128, [3000, 1, 1500, 2049], 11),   # first call
             (2, 4, 700, 64, [700, 129], 12)]                # second call, other sizes
    for B, H, Skv, D, lens, seed in cases:
        q, kc, vc, kl = _inputs(B, H, Skv, D, lens, seed)
        out = torch.full((B, H, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert _noalloc(lib, q, kc, vc, kl, out) == attn.ATTN_OK, attn.attn_last_error()
        attn.attn_device_status()
        ref = attn.attn_decode(q, kc, vc, kv_len=kl)
        attn.attn_device_status()
        err = (out.float() - ref.float()).abs()
        assert torch.isfinite(out.float()).all()
        assert err.max().item() <= BF16_MAX and err.mean().item() <= BF16_MEAN
        exact = oracle.decode(q.cpu(), kc.cpu(), vc.cpu(), kv_len=np.array(lens, np.int32))
        assert_close(out, exact, torch.bfloat16, f"no-allocation decode B{B} H{H} Skv{Skv} D{D} vs oracle")


def test_noalloc_rejects_sizes_beyond_its_scratch(gpu):
    lib = attn.lib()
    # 4096 heads x 16 splits x 130 floats x 4 bytes = 34 MB > the 32 MiB scratch
    B, H, Skv, D = 128, 32, 8192, 128
    assert attn.attn_decode_splits(B, H, Skv, D) * B * H * (D + 2) * 4 > (32 << 20)
    fake = [P((i + 1) << 36) for i in range(4)]  # 64 GB apart: no overlap with an 8.6 GB cache
    rc = lib.attn_decode_noalloc(fake[0], fake[1], fake[2], fake[3], B, H, Skv, D, None, attn.ATTN_BF16, None)
    assert rc == attn.ATTN_EINVAL
    assert "scratch" in attn.attn_last_error()
