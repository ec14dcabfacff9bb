"""GPU parity tests of fp32 decode (attn_decode / attn_decode_gqa /
attn_decode_noalloc with ATTN_F32): fp32 inputs, accumulation and output on
the CUDA cores, against the fp64 oracle within the fp32 tolerance (max abs
error 1e-4)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_fwd_gb300 as attn
from transformer_scaled_dot_fwd_gb300 import workloads as wl
from helpers import assert_close

pytestmark = pytest.mark.gpu


def _case(B, H, H_kv, Skv, D, lens=None, seed=0, noalloc=False):
    q = wl.random_tensors((B, H, D), seed, dtype=torch.float32, count=1)[0]
    kc, vc = wl.random_tensors((B, H_kv, Skv, D), seed + 1, dtype=torch.float32, count=2)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens is not None else None
    if noalloc:
        out = torch.empty_like(q)
        attn.attn_decode_noalloc(q, kc, vc, out, kv_len=kl)
    else:
        out = attn.attn_decode(q, kc, vc, kv_len=kl)
    attn.attn_device_status()
    assert out.dtype == torch.float32
    ref = oracle.decode(q.cpu(), kc.cpu(), vc.cpu(), kv_len=None if lens is None else np.array(lens, np.int32))
    return out, ref


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(4, 4), (8, 2), (8, 1)])
@pytest.mark.parametrize("Skv", [1, 63, 65, 700, 3000])
def test_f32_decode(gpu, H, H_kv, Skv, D):
    out, ref = _case(2, H, H_kv, Skv, D, seed=Skv + H + D)
    assert_close(out, ref, torch.float32, f"fp32 decode H={H} H_kv={H_kv} Skv={Skv} D={D}")


def test_f32_decode_lengths_and_empty_sequences(gpu):
    lens = [2000, 0, 1, 511, 512, 513, 1999]
    out, ref = _case(len(lens), 4, 2, 2000, 128, lens=lens, seed=9)
    assert_close(out, ref, torch.float32, "fp32 decode, per-sequence lengths")
    assert torch.count_nonzero(out[1]) == 0


def test_f32_decode_noalloc_equals_allocating_path(gpu):
    lens = [900, 5, 0]
    a, ref = _case(3, 8, 8, 900, 64, lens=lens, seed=13)
    b, _ = _case(3, 8, 8, 900, 64, lens=lens, seed=13, noalloc=True)
    assert torch.equal(a, b)
    assert_close(b, ref, torch.float32, "fp32 decode without allocation")


def test_f32_decode_workload_shape_sampled(gpu):
    """The decode workload's shape (B64 H32 D128, cache 8192, lengths
    U{4096..8192}) in fp32; the oracle checks sampled sequences."""
    w = wl.DECODE
    g = torch.Generator(device="cuda").manual_seed(w.seed + 7)
    q = torch.randn(w.B, w.H, w.D, device="cuda", generator=g)
    kc = torch.randn(w.B, w.H, w.Skv, w.D, device="cuda", generator=g)
    vc = torch.randn(w.B, w.H, w.Skv, w.D, device="cuda", generator=g)
    lens = wl.draw_lengths(w.B, w.kv_len_range, w.seed)
    out = attn.attn_decode(q, kc, vc, kv_len=lens.cuda())
    attn.attn_device_status()
    bs = np.array([0, 31, w.B - 1])
    ref = oracle.decode(q[bs].cpu(), kc[bs].cpu(), vc[bs].cpu(), kv_len=lens[bs].numpy())
    assert_close(out[bs], ref, torch.float32, "fp32 decode workload shape, sampled sequences")
