"""GPU tests of attn_fwd_host: prefill from host buffers with the copies
pipelined against the computation.

Each chunk of (b, h) slices is computed by the same kernel and arithmetic as
a single attn_fwd call over the whole batch, so the host path must equal the
device path bit for bit; the device path itself is checked against the
oracle in test_gpu_prefill.py.  The shapes below select each way the batch is
cut: one chunk, whole sequences per chunk (kv_len offsets per chunk), and runs
of key/value heads of one sequence (multi-head and grouped-query).
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

CASES = [  # (B, H, H_kv, Sq, Skv, D, causal, lengths, dtype)
    (2, 4, 4, 1000, 1000, 128, True, None, torch.bfloat16),           # one chunk, ragged tiles
    (1, 16, 16, 4096, 4096, 128, True, None, torch.bfloat16),         # key/value heads of one sequence
    (1, 32, 8, 4096, 4096, 128, True, None, torch.bfloat16),          # the same, grouped-query
    (16, 8, 8, 2048, 2048, 64, True, "random", torch.bfloat16),       # whole sequences per chunk
    (1, 16, 16, 2048, 2048, 64, True, None, torch.float32),           # fp32, several chunks
    (4, 4, 2, 100, 700, 128, False, [700, 333, 1, 0], torch.bfloat16),  # cross-attention, padded source
]


def _inputs(case, seed):
    B, H, H_kv, Sq, Skv, D, causal, lengths, dtype = case
    q = wl.random_tensors((B, H, Sq, D), seed, dtype=dtype, count=1)[0]
    k, v = wl.random_tensors((B, H_kv, Skv, D), seed + 1, dtype=dtype, count=2)
    if lengths == "random":
        lengths = wl.draw_lengths(B, (1, Skv), seed).tolist()
    return q, k, v, lengths


@pytest.mark.parametrize("case", CASES)
def test_host_path_equals_device_path(gpu, case):
    B, H, H_kv, Sq, Skv, D, causal, _, dtype = case
    q, k, v, lengths = _inputs(case, 90 + Sq + B)
    kl_dev = torch.tensor(lengths, dtype=torch.int32, device="cuda") if lengths is not None else None
    ref = attn.attn_fwd(q, k, v, causal=causal, kv_len=kl_dev)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    out = attn.attn_fwd_host(hq, hk, hv, causal=causal, kv_len=lengths)
    attn.attn_device_status()
    assert out.device.type == "cpu" and out.is_pinned()
    assert torch.equal(out, ref.cpu())


def test_host_path_against_the_oracle(gpu):
    """Sampled rows of a multi-chunk call against the oracle directly."""
    case = CASES[3]
    q, k, v, lengths = _inputs(case, 7)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    out = attn.attn_fwd_host(hq, hk, hv, causal=True, kv_len=lengths)
    rng = np.random.default_rng(0)
    B, H, S = q.shape[0], q.shape[1], q.shape[2]
    rows = np.stack([rng.integers(0, B, 64), rng.integers(0, H, 64), rng.integers(0, S, 64)], 1).astype(np.int64)
    ref = oracle.attention_rows(hq, hk, hv, rows, causal=True, kv_len=np.array(lengths, np.int32))
    got = out[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, ref, torch.bfloat16, "attn_fwd_host sampled rows")


def test_pageable_memory_and_empty_keys(gpu):
    q, k, v, _ = _inputs(CASES[0], 3)
    hq, hk, hv = q.cpu(), k.cpu(), v.cpu()  # pageable
    out = attn.attn_fwd_host(hq, hk, hv, causal=True)
    assert not out.is_pinned()
    assert torch.equal(out, attn.attn_fwd(q, k, v, causal=True).cpu())
    # no keys: every row is zero
    e = torch.empty(2, 4, 0, 128, dtype=torch.bfloat16)
    z = attn.attn_fwd_host(hq[:, :, :16].contiguous(), e, e.clone(), causal=False)
    assert torch.count_nonzero(z) == 0


def test_stream_argument_and_repeated_calls(gpu):
    q, k, v, _ = _inputs(CASES[2], 5)
    hq, hk, hv = (t.cpu().pin_memory() for t in (q, k, v))
    s = torch.cuda.Stream()
    ref = attn.attn_fwd(q, k, v, causal=True).cpu()
    out = torch.empty_like(hq).pin_memory()
    for _ in range(3):
        out.zero_()
        attn.attn_fwd_host(hq, hk, hv, out=out, causal=True, stream=s)
        assert torch.equal(out, ref)
    attn.attn_release()
    assert torch.equal(attn.attn_fwd_host(hq, hk, hv, causal=True), ref)
