"""The library's calls captured in a CUDA graph and replayed.

A decode loop replays the same launches once per token, so launch overhead
matters; a CUDA graph removes it.  After one ordinary call (which sizes the
decode workspace), attn_fwd and attn_decode can be captured: the persistent
prefill kernel's work counter is reset by the CTA that draws the launch's
last item number, so every replay starts from zero, and the decode partials live in the library's workspace.
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


def test_replay_beside_many_direct_launches(gpu):
    """A captured prefill keeps its work counter for every replay.  Captured
    launches take counters outside the 64 that direct calls rotate through,
    so a replay running on one stream while 70 direct calls run on another
    never shares a counter with them: both sets of outputs must equal
    ordinary calls bit for bit, and the device status must stay clean."""
    q1, k1, v1 = wl.random_tensors((2, 8, 1536, 128), 70)
    q2, k2, v2 = wl.random_tensors((1, 4, 640, 128), 71)
    ref1 = attn.attn_fwd(q1, k1, v1, causal=True).clone()
    ref2 = attn.attn_fwd(q2, k2, v2, causal=False).clone()
    out1 = torch.empty_like(q1)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        attn.attn_fwd(q1, k1, v1, out=out1, causal=True)
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    replays, directs = [], []
    for r in range(6):
        with torch.cuda.stream(sa):
            g.replay()
            replays.append(out1.clone())
        with torch.cuda.stream(sb):
            for _ in range(12):
                directs.append(attn.attn_fwd(q2, k2, v2, causal=False, stream=sb))
    sa.synchronize()
    sb.synchronize()
    attn.attn_device_status()
    assert len(directs) >= 70
    for o in replays:
        assert torch.equal(o, ref1)
    for o in directs:
        assert torch.equal(o, ref2)


def test_shared_counter_is_reported_or_harmless(gpu):
    """Direct calls rotate through 64 work counters, so a 65th call in flight
    takes the counter of the first.  Here a long launch (B1 H32 S8192) runs on
    one stream while 63 short launches on a second stream move the rotation
    on, and a 65th launch on a third stream lands on the long launch's
    counter while it may still be running.  Either the two launches did not
    overlap and every output equals an ordinary call, or the overlap was
    detected and attn_device_status reports ATTN_ECONFLICT; it must never be
    wrong without a report.  Nothing here waits on another kernel: the
    launches only share a counter."""
    ql, kl_, vl = wl.random_tensors((1, 32, 8192, 128), 72)
    qs, ks, vs = wl.random_tensors((1, 2, 128, 64), 73)
    ref_l = attn.attn_fwd(ql, kl_, vl, causal=True).clone()
    ref_s = attn.attn_fwd(qs, ks, vs, causal=True).clone()
    torch.cuda.synchronize()
    s1, s2, s3 = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    long_out, clash = torch.empty_like(ql), torch.empty_like(ql)
    go = torch.cuda.Event()
    with torch.cuda.stream(s1):
        # hold the long launch (about 5 ms of a one-SM spin) until every call below is enqueued
        torch.cuda._sleep(10_000_000)
        go.record(s1)
        attn.attn_fwd(ql, kl_, vl, out=long_out, causal=True, stream=s1)
    with torch.cuda.stream(s2):
        shorts = [attn.attn_fwd(qs, ks, vs, causal=True, stream=s2) for _ in range(63)]
    s3.wait_event(go)
    with torch.cuda.stream(s3):
        attn.attn_fwd(ql, kl_, vl, out=clash, causal=True, stream=s3)
    torch.cuda.synchronize()
    try:
        attn.attn_device_status()
    except attn.AttnError as e:
        assert e.code == attn.ATTN_ECONFLICT, e
        # the shared counter may be left unbalanced: with nothing in flight,
        # attn_release clears every counter, and later launches are clean again
        attn.attn_release()
        for _ in range(70):
            assert torch.equal(attn.attn_fwd(qs, ks, vs, causal=True), ref_s)
        attn.attn_device_status()
        return
    assert torch.equal(long_out, ref_l)
    assert torch.equal(clash, ref_l)
    for o in shorts:
        assert torch.equal(o, ref_s)


def test_decode_capture_survives_workspace_growth(gpu):
    """Growing the decode workspace keeps the old buffer (until attn_release),
    so a graph captured before a larger call still replays correctly; a call
    that would need a larger workspace during a capture is refused instead of
    allocating."""
    torch.cuda.synchronize()
    attn.attn_release()  # start from an empty workspace
    B, H, S, D = 2, 4, 640, 128
    q = wl.random_tensors((B, H, D), 80, count=1)[0]
    k, v = wl.random_tensors((B, H, S, D), 81, count=2)
    out = torch.empty_like(q)
    ref = attn.attn_decode(q, k, v).clone()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        attn.attn_decode(q, k, v, out=out)
    # a much larger call grows the workspace
    qb = wl.random_tensors((64, 32, D), 82, count=1)[0]
    kb, vb = wl.random_tensors((64, 32, 4096, D), 83, count=2)
    big = attn.attn_decode(qb, kb, vb)
    torch.cuda.synchronize()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    attn.attn_device_status()
    assert torch.equal(out, ref)
    # capturing a call larger than the workspace (65536 heads: 34 MB of partials) is
    # refused on the host, with nothing enqueued, so its inputs are never read
    qh = torch.empty((512, 128, D), dtype=torch.bfloat16, device="cuda")
    kh = torch.empty((512, 128, 64, D), dtype=torch.bfloat16, device="cuda")
    vh = torch.empty_like(kh)
    g2 = torch.cuda.CUDAGraph()
    with pytest.raises(attn.AttnError) as err:
        with torch.cuda.graph(g2):
            attn.attn_decode(qh, kh, vh)
    assert err.value.code == attn.ATTN_EINVAL
    del big, g, g2, qh, kh, vh
    torch.cuda.synchronize()
