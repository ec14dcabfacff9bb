"""Seeded synthetic inputs shaped like the pages' attention workloads.

This module holds no attention arithmetic: it only draws Q, K, V (i.i.d.
N(0, 1), float32 draws rounded to the target dtype) and per-sequence lengths
from explicit seeds, so that the CUDA library and the CPU oracle see exactly
the same numbers.  Shapes follow the pages: d_model 4096 split into 32 heads
of d_head 128 ("Attention from First Principles", section 5 "Why multiple
heads": d=4096, h=32, d_head=128), prefill at S = 2048 and decode against a
KV cache (section 6 "Under the hood").
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from typing import Optional, Tuple

import torch


@dataclass(frozen=True)
class PrefillWorkload:
    name: str
    B: int
    H: int
    S: int
    D: int
    dtype: str                      # "bf16" or "f32"
    causal: bool
    seed: int
    kv_len_range: Optional[Tuple[int, int]] = None  # inclusive range of valid lengths
    scale: Optional[float] = None   # default 1/sqrt(D)

    @property
    def torch_dtype(self):
        return torch.bfloat16 if self.dtype == "bf16" else torch.float32

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale is not None else 1.0 / math.sqrt(self.D)


@dataclass(frozen=True)
class DecodeWorkload:
    name: str
    B: int
    H: int
    Skv: int
    D: int
    seed: int
    kv_len_range: Optional[Tuple[int, int]] = None


# The five workloads: a small fp32 case the oracle finishes in well under a
# second, causal bf16 prefill at (B4, H32, S2048, D128), causal + key padding
# at (B8, H16, S4096), long-context causal at S16384, and KV-cache decode.
TINY_F32 = PrefillWorkload("causal fp32 prefill B2 H4 S128 D64", 2, 4, 128, 64, "f32", True, 0,
                           scale=1.0 / 8.0)
PREFILL = PrefillWorkload("causal MHA prefill B4 H32 S2048 D128 bf16", 4, 32, 2048, 128, "bf16",
                          True, 1)
PADDED = PrefillWorkload("causal + key-padding prefill B8 H16 S4096 D128 bf16", 8, 16, 4096, 128,
                         "bf16", True, 2, kv_len_range=(1024, 4096))
LONG = PrefillWorkload("long-context causal prefill B1 H32 S16384 D128 bf16", 1, 32, 16384, 128,
                       "bf16", True, 3)
DECODE = DecodeWorkload("KV-cache decode B64 H32 D128 Skv<=8192 bf16", 64, 32, 8192, 128, 4,
                        kv_len_range=(4096, 8192))

PREFILL_WORKLOADS = {"tiny_f32": TINY_F32, "prefill": PREFILL, "padded": PADDED, "long": LONG}

# Sequence-length sweep at fixed batch ('Attention from First Principles',
# Exercises, D: S from 128 to 4096), extended to 65536, where a materialised
# (B, H, S, S) bf16 score tensor of this batch (2.2 TB) no longer fits in HBM.
S_SWEEP_SHAPE = dict(B=4, H=32, D=128, seed=5)
S_SWEEP = (128, 256, 512, 1024, 2048, 4096, 8192, 16384, 32768, 65536)


def _normal(shape, gen, device, dtype):
    x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
    return x.to(dtype)


def _generator(seed, device):
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def draw_lengths(B: int, lo_hi: Optional[Tuple[int, int]], seed: int) -> Optional[torch.Tensor]:
    """Per-sequence valid lengths, uniform on the inclusive range, CPU int32."""
    if lo_hi is None:
        return None
    g = _generator(seed, "cpu")
    return torch.randint(lo_hi[0], lo_hi[1] + 1, (B,), generator=g, dtype=torch.int64).to(torch.int32)


def prefill_inputs(w: PrefillWorkload, device="cuda", seed: Optional[int] = None):
    """(q, k, v, kv_len) for a prefill workload.  kv_len is an int32 tensor on
    ``device`` or None.  Large tensors are drawn directly on the device."""
    seed = w.seed if seed is None else seed
    g = _generator(seed, device if str(device).startswith("cuda") else "cpu")
    shape = (w.B, w.H, w.S, w.D)
    q = _normal(shape, g, device, w.torch_dtype)
    k = _normal(shape, g, device, w.torch_dtype)
    v = _normal(shape, g, device, w.torch_dtype)
    kv_len = draw_lengths(w.B, w.kv_len_range, seed)
    if kv_len is not None:
        kv_len = kv_len.to(device)
    return q, k, v, kv_len


def decode_inputs(w: DecodeWorkload, device="cuda", seed: Optional[int] = None):
    """(q, kcache, vcache, kv_len) for a decode workload; q is (B, H, D)."""
    seed = w.seed if seed is None else seed
    g = _generator(seed, device if str(device).startswith("cuda") else "cpu")
    q = _normal((w.B, w.H, w.D), g, device, torch.bfloat16)
    kc = _normal((w.B, w.H, w.Skv, w.D), g, device, torch.bfloat16)
    vc = _normal((w.B, w.H, w.Skv, w.D), g, device, torch.bfloat16)
    kv_len = draw_lengths(w.B, w.kv_len_range, seed)
    if kv_len is not None:
        kv_len = kv_len.to(device)
    return q, kc, vc, kv_len


def random_tensors(shape, seed, device="cuda", dtype=torch.bfloat16, count=3):
    """``count`` i.i.d. N(0, 1) tensors of one shape from one seed (test helper)."""
    g = _generator(seed, device if str(device).startswith("cuda") else "cpu")
    return [_normal(shape, g, device, dtype) for _ in range(count)]


def s_sweep_inputs(S: int, device="cuda", rank: int = 0):
    """Q, K, V (B, H, S, D) bf16 of the sequence-length sweep at length S."""
    sh = S_SWEEP_SHAPE
    g = _generator(sh["seed"] + S + 1000 * rank, device)
    return [_normal((sh["B"], sh["H"], S, sh["D"]), g, device, torch.bfloat16) for _ in range(3)]
