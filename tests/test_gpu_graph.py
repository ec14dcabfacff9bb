"""The library's calls captured in a CUDA graph and replayed.

A decode loop replays the same launches once per token, so launch overhead
matters; a CUDA graph removes it.  After one ordinary call (which sizes the
decode workspace), attn_fwd and attn_decode can be captured: the persistent
prefill kernel's work counter is reset by its last CTA, so every replay
starts from zero, and the decode partials live in the library's workspace.
Replays with new data copied into the captured buffers must equal ordinary
calls bit for bit.
"""
from __future__ import annotations

import torch
import pytest

import transformer_scaled_dot_fwd_gb300 as attn
from transformer_scaled_dot_fwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def test_capture_and_replay_prefill_and_decode(gpu):
    B, H, S, D = 2, 8, 1000, 128
    q, k, v = wl.random_tensors((B, H, S, D), 40)
    kl = torch.tensor([1000, 377], dtype=torch.int32, device="cuda")
    qd = wl.random_tensors((B, H, D), 41, count=1)[0]
    qg = wl.random_tensors((B, 4 * H, D), 42, count=1)[0]  # grouped decode: 4 query heads per cached head
    out, od, og = torch.empty_like(q), torch.empty_like(qd), torch.empty_like(qg)

    def calls():
        attn.attn_fwd(q, k, v, out=out, causal=True, kv_len=kl)
        attn.attn_decode(qd, k, v, out=od, kv_len=kl)
        attn.attn_decode(qg, k, v, out=og, kv_len=kl)

    calls()  # sizes the workspace and caches device attributes
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        calls()
    for seed in (50, 60):
        # new inputs in the captured buffers
        for t, s in ((q, seed), (k, seed + 1), (v, seed + 2), (qd, seed + 3), (qg, seed + 4)):
            t.copy_(wl.random_tensors(tuple(t.shape), s, count=1)[0])
        kl.copy_(torch.tensor([seed * 10, 999], dtype=torch.int32, device="cuda"))
        g.replay()
        torch.cuda.synchronize()
        got = (out.clone(), od.clone(), og.clone())
        calls()
        torch.cuda.synchronize()
        attn.attn_device_status()
        for a, b in zip(got, (out, od, og)):
            assert torch.equal(a, b)
