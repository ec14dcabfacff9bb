"""GPU tests of calls chained on one stream without synchronisation.

Every kernel of the path is launched with programmatic stream serialisation:
it may be placed while the previous kernel in the stream is still running and
must wait for it before reading its inputs or writing its output.  Here each
call reads the previous call's output (prefill -> prefill, decode -> decode,
prefill -> decode through the cache, and fp32 as well), with no
synchronisation in between, and the chain must equal, bit for bit, the same
chain with a device synchronisation after every call.  A write-after-read
case (a call overwriting the buffer the previous call reads) is included.
"""
from __future__ import annotations

import pytest
import torch

import transformer_scaled_dot_fwd_gb300 as attn
from transformer_scaled_dot_fwd_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


def _chain(step, x0, n, sync):
    xs = [x0]
    for _ in range(n):
        xs.append(step(xs[-1]))
        if sync:
            torch.cuda.synchronize()
    torch.cuda.synchronize()
    attn.attn_device_status()
    return xs


@pytest.mark.parametrize("dtype,D", [(torch.bfloat16, 128), (torch.bfloat16, 64), (torch.float32, 64)])
def test_prefill_chain(gpu, dtype, D):
    q, k, v = wl.random_tensors((2, 8, 700, D), 71, dtype=dtype)
    step = lambda x: attn.attn_fwd(x, k, v, causal=True)  # noqa: E731
    fast = _chain(step, q, 6, sync=False)
    slow = _chain(step, q, 6, sync=True)
    for a, b in zip(fast, slow):
        assert torch.equal(a, b)


@pytest.mark.parametrize("H_kv,dtype", [(32, torch.bfloat16), (8, torch.bfloat16), (1, torch.bfloat16),
                                        (2, torch.bfloat16), (32, torch.float32)])
def test_decode_chain(gpu, H_kv, dtype):
    B, H, Skv, D = 4, 32, 3000, 128
    q = wl.random_tensors((B, H, D), 72, count=1, dtype=dtype)[0]
    kc, vc = wl.random_tensors((B, H_kv, Skv, D), 73, count=2, dtype=dtype)
    lens = torch.tensor([3000, 1, 1500, 2049], dtype=torch.int32, device="cuda")
    step = lambda x: attn.attn_decode(x, kc, vc, kv_len=lens)  # noqa: E731
    fast = _chain(step, q, 8, sync=False)
    slow = _chain(step, q, 8, sync=True)
    for a, b in zip(fast, slow):
        assert torch.equal(a, b)


def test_prefill_output_feeds_decode_cache(gpu):
    """The decode reads a cache that the prefill launched just before it writes."""
    B, H, S, D = 2, 8, 1024, 128
    q, k, v = wl.random_tensors((B, H, S, D), 74)
    qd = wl.random_tensors((B, H, D), 75, count=1)[0]

    def run(sync):
        cache = attn.attn_fwd(q, k, v, causal=True)          # (B, H, S, D), becomes the keys
        if sync:
            torch.cuda.synchronize()
        out = attn.attn_decode(qd, cache, v)
        torch.cuda.synchronize()
        attn.attn_device_status()
        return out

    assert torch.equal(run(False), run(True))


def test_overwrite_after_read(gpu):
    """A call that writes the buffer the previous call reads (as its keys) must
    not start writing before that call has finished reading."""
    B, H, S, D = 2, 8, 2048, 128
    q, k, v = wl.random_tensors((B, H, S, D), 76)
    q2 = wl.random_tensors((B, H, S, D), 77, count=1)[0]
    ref = attn.attn_fwd(q, k, v, causal=True)
    torch.cuda.synchronize()
    for _ in range(3):
        k_work = k.clone()
        torch.cuda.synchronize()
        out = attn.attn_fwd(q, k_work, v, causal=True)     # reads k_work
        attn.attn_fwd(q2, k, v, out=k_work, causal=True)   # then overwrites it
        torch.cuda.synchronize()
        attn.attn_device_status()
        assert torch.equal(out, ref)


def test_captured_chain_replays(gpu):
    """A chain of dependent calls captured in one CUDA graph (the programmatic
    launches become programmatic edges) replays to the eager chain's result."""
    B, H, S, D = 2, 8, 900, 128
    q, k, v = wl.random_tensors((B, H, S, D), 80)
    qd = wl.random_tensors((B, H, D), 81, count=1)[0]
    kl = torch.tensor([900, 333], dtype=torch.int32, device="cuda")
    x1, x2, x3 = (torch.empty_like(q) for _ in range(3))
    d1, d2 = torch.empty_like(qd), torch.empty_like(qd)

    def chain():
        attn.attn_fwd(q, k, v, out=x1, causal=True)
        attn.attn_fwd(x1, k, v, out=x2, causal=True)          # reads x1
        attn.attn_fwd(x2, x1, v, out=x3, causal=True)         # reads x2 and x1
        attn.attn_decode(qd, x3, v, out=d1, kv_len=kl)        # the cache is x3
        attn.attn_decode(d1, x3, x2, out=d2, kv_len=kl)       # reads d1

    chain()  # sizes the decode workspace
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    for seed in (90, 95):
        for t, s in ((q, seed), (k, seed + 1), (v, seed + 2), (qd, seed + 3)):
            t.copy_(wl.random_tensors(tuple(t.shape), s, count=1)[0])
        g.replay()
        torch.cuda.synchronize()
        got = [t.clone() for t in (x1, x2, x3, d1, d2)]
        for t in (x1, x2, x3, d1, d2):
            t.fill_(float("nan"))
        chain()
        torch.cuda.synchronize()
        attn.attn_device_status()
        for a, b in zip(got, (x1, x2, x3, d1, d2)):
            assert torch.equal(a, b)
