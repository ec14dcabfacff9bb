"""GPU parity tests of grouped-query and multi-query decode with query
groups of G = H / H_kv >= 4 heads, which runs on the tensor cores: the G queries of
a cached head are the rows of one 128-row tile, keys stream through in 64-key
tiles in chunks merged by the decode combine.  Tolerances are those of
test_gpu_decode.py (bf16 max 2e-2, mean 2e-3 against the fp64 oracle).
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


def _case(B, H, H_kv, Skv, D, lens=None, seed=0, k_scale=None):
    q = wl.random_tensors((B, H, D), seed, count=1)[0]
    kc, vc = wl.random_tensors((B, H_kv, Skv, D), seed + 1, count=2)
    if k_scale is not None:
        kc = (kc.float() * k_scale).to(torch.bfloat16)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens is not None else None
    out = attn.attn_decode(q, kc, vc, kv_len=kl)
    attn.attn_device_status()
    ref = oracle.decode(q.cpu(), kc.cpu(), vc.cpu(), kv_len=None if lens is None else np.array(lens, np.int32))
    return out, ref


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(4, 1), (8, 1), (16, 1), (32, 1), (64, 2), (128, 1), (32, 4), (32, 8)])
@pytest.mark.parametrize("Skv", [1, 64, 65, 1000, 4097])
def test_large_group_decode(gpu, H, H_kv, Skv, D):
    out, ref = _case(2, H, H_kv, Skv, D, seed=Skv + H)
    assert_close(out, ref, torch.bfloat16, f"decode H={H} H_kv={H_kv} Skv={Skv} D={D}")


@pytest.mark.parametrize("H,H_kv", [(32, 1), (16, 2), (16, 4)])
def test_large_group_decode_lengths(gpu, H, H_kv):
    # lengths at and around the 64-key tiles and the chunk boundaries, and empty sequences
    lens = [3000, 0, 1, 63, 64, 65, 1152, 1153, 2999, 2048]
    out, ref = _case(len(lens), H, H_kv, 3000, 128, lens=lens, seed=11)
    assert_close(out, ref, torch.bfloat16, "large-group decode, per-sequence lengths")
    assert torch.count_nonzero(out[1]) == 0  # a sequence with no keys gives zeros


@pytest.mark.parametrize("B,H,H_kv,Skv,kind", [
    (1, 32, 1, 20000, "full"),          # one long sequence: many chunks of one cached head
    (300, 8, 2, 200, "random"),         # many short sequences of random length
    (5, 16, 4, 700, "empty"),           # no keys at all: every output is zero
    (70, 32, 8, 129, "mostly_empty"),   # few keys in the whole batch
    (3, 64, 16, 4096, "ragged"),        # sequences of very different lengths
])
def test_batch_shapes(gpu, B, H, H_kv, Skv, kind):
    rng = np.random.default_rng(B + Skv)
    lens = {"full": [Skv] * B, "random": rng.integers(0, Skv + 1, B).tolist(), "empty": [0] * B,
            "mostly_empty": [0] * (B - 3) + [1, 64, Skv], "ragged": [Skv, 1, 777]}[kind]
    out, ref = _case(B, H, H_kv, Skv, 128, lens=lens, seed=B * 7 + H)
    assert_close(out, ref, torch.bfloat16, f"batch B={B} H={H} H_kv={H_kv} Skv={Skv} {kind}")
    for b, L in enumerate(lens):
        if L == 0:
            assert torch.count_nonzero(out[b]) == 0


def test_growing_scores_rescale_mid_stream(gpu):
    """Keys scaled up along the cache: each later tile's scores exceed the
    running max by more than 2^8, so O is rescaled again and again."""
    Skv = 2048
    ramp = torch.linspace(0.2, 6.0, Skv, device="cuda").view(1, 1, Skv, 1)
    out, ref = _case(3, 32, 1, Skv, 128, seed=21, k_scale=ramp)
    assert_close(out, ref, torch.bfloat16, "rescale mid-stream")


def test_group_above_the_tile_uses_the_other_path(gpu):
    out, ref = _case(2, 256, 1, 500, 64, seed=31)  # G = 256 > 128 rows
    assert_close(out, ref, torch.bfloat16, "G = 256 decode")


def test_mqa_decode_workload_sampled(gpu):
    """The decode workload's shape as multi-query attention (B64 H32 H_kv1,
    cache 8192, lengths U{4096..8192}), in the benchmark's launch
    configuration; the oracle checks sampled sequences."""
    w = wl.DECODE
    g = torch.Generator(device="cuda").manual_seed(w.seed + 1)
    q = torch.randn(w.B, w.H, w.D, device="cuda", generator=g).to(torch.bfloat16)
    kc = torch.randn(w.B, 1, w.Skv, w.D, device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn(w.B, 1, w.Skv, w.D, device="cuda", generator=g).to(torch.bfloat16)
    lens = wl.draw_lengths(w.B, w.kv_len_range, w.seed)
    out = attn.attn_decode(q, kc, vc, kv_len=lens.cuda())
    attn.attn_device_status()
    bs = np.array([0, 1, 17, 40, w.B - 1])
    ref = oracle.decode(q[bs].cpu(), kc[bs].cpu(), vc[bs].cpu(), kv_len=lens[bs].numpy())
    assert_close(out[bs], ref, torch.bfloat16, "B64 H32 H_kv1 decode, sampled sequences")
