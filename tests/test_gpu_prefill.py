"""GPU parity tests of attn_fwd (through the C ABI) against the fp64 oracle.

Tolerances (absolute, vs. the oracle on the same seeded inputs): fp32 max
1e-4; bf16 max 2e-2 and mean 2e-3 (bf16 operands, fp32 accumulation).
Bit-exact checks where the answer is exact: padded query rows and rows that
see no key are exactly zero, causal row 0 equals V[0].
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_fwd_gb300 as attn
from transformer_scaled_dot_fwd_gb300 import workloads as wl
from helpers import assert_close, to_f64

pytestmark = pytest.mark.gpu


def run_case(B, H, Sq, Skv, D, causal, dtype=torch.bfloat16, kv_len=None, seed=0, scale=None):
    q = wl.random_tensors((B, H, Sq, D), seed, dtype=dtype, count=1)[0]
    k, v = wl.random_tensors((B, H, Skv, D), seed + 1000, dtype=dtype, count=2)
    kl = torch.tensor(kv_len, dtype=torch.int32, device="cuda") if kv_len is not None else None
    out = attn.attn_fwd(q, k, v, scale=scale, causal=causal, kv_len=kl)
    attn.attn_device_status()
    ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale=scale, causal=causal,
                           kv_len=None if kv_len is None else np.array(kv_len, np.int32))
    return q, k, v, out, ref


def test_tiny_fp32_workload(gpu):
    w = wl.TINY_F32
    q, k, v, kl = wl.prefill_inputs(w, device="cuda")
    out = attn.attn_fwd(q, k, v, scale=w.softmax_scale, causal=w.causal)
    attn.attn_device_status()
    ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale=w.softmax_scale, causal=True)
    assert_close(out, ref, torch.float32, "fp32 B2 H4 S128 D64")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1, 2, 17, 127, 128, 129, 255, 256, 257, 300, 513])
@pytest.mark.parametrize("causal", [True, False])
def test_fp32_shapes(gpu, S, D, causal):
    _, _, _, out, ref = run_case(2, 3, S, S, D, causal, dtype=torch.float32, seed=S)
    assert_close(out, ref, torch.float32, f"fp32 S={S} D={D} causal={causal}")


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("S", [1, 2, 17, 127, 128, 129, 255, 256, 257, 300, 383, 513, 1000])
@pytest.mark.parametrize("causal", [True, False])
def test_bf16_shapes(gpu, S, D, causal):
    _, _, v, out, ref = run_case(2, 3, S, S, D, causal, seed=S)
    assert_close(out, ref, torch.bfloat16, f"bf16 S={S} D={D} causal={causal}")
    if causal:  # row 0 sees only key 0: exactly V[0]
        assert torch.equal(out[:, :, 0], v[:, :, 0])


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Sq,Skv,causal", [(4, 7, False), (100, 300, False), (300, 100, False),
                                           (1, 513, False), (129, 130, True), (64, 1000, True),
                                           (1, 300, True), (255, 256, True)])
def test_cross_and_chunked(gpu, Sq, Skv, D, causal):
    """T_q != T_k: cross-attention shape test ("Attention from Scratch" (kube-dojo),
    Part 7) and a causal chunk of queries aligned to the end of the keys."""
    _, _, _, out, ref = run_case(1, 2, Sq, Skv, D, causal, seed=Sq * 7 + Skv)
    assert_close(out, ref, torch.bfloat16, f"Sq={Sq} Skv={Skv} causal={causal}")


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [64, 128])
def test_key_padding_edges(gpu, D, dtype):
    S = 300
    lens = [0, 1, 2, 127, 128, 129, 255, 256, 257, 299, 300]
    q, k, v, out, ref = run_case(len(lens), 2, S, S, D, True, dtype=dtype, kv_len=lens, seed=D)
    assert_close(out, ref, dtype, f"key padding D={D}")
    for b, L in enumerate(lens):
        assert torch.count_nonzero(out[b, :, L:]) == 0, f"padded rows of sequence {b} not zero"
        if L > 0:
            assert torch.equal(out[b, :, 0], v[b, :, 0])


def test_key_padding_non_causal(gpu):
    lens = [5, 130, 256, 1]
    _, _, _, out, ref = run_case(4, 2, 256, 256, 128, False, kv_len=lens, seed=11)
    assert_close(out, ref, torch.bfloat16, "non-causal key padding")


def test_scale_zero_gives_visible_mean(gpu):
    """scale = 0: every visible key has the same score, so the output is the
    mean of the visible V rows (oracle pin 'uniform scores')."""
    _, _, _, out, ref = run_case(2, 2, 200, 200, 128, True, kv_len=[150, 200], scale=0.0, seed=5)
    assert_close(out, ref, torch.bfloat16, "scale 0")


def test_large_logits_are_stable(gpu):
    """Scores of magnitude ~100 (large scale) exercise the running max and the
    lazy rescale without overflow."""
    _, _, _, out, ref = run_case(1, 4, 512, 512, 128, True, scale=2.0, seed=6)
    assert_close(out, ref, torch.bfloat16, "scale 2.0")


def test_masked_positions_are_selected_out(gpu):
    """Masking is a select, not an add: keys at padded positions hold inf/NaN
    and values there hold huge finite numbers; the output must not change.
    (Values at masked positions must be finite: a tensor-core product 0 * inf
    is NaN, see include/attn.h.)"""
    B, H, S, D = 2, 2, 384, 128
    lens = [200, 301]
    q = wl.random_tensors((B, H, S, D), 21, count=1)[0]
    k, v = wl.random_tensors((B, H, S, D), 22, count=2)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    clean = attn.attn_fwd(q, k, v, causal=True, kv_len=kl).clone()
    k2, v2 = k.clone(), v.clone()
    for b, L in enumerate(lens):
        k2[b, :, L:] = float("nan")
        k2[b, :, L::3] = float("inf")
        v2[b, :, L:] = 1e30
    poisoned = attn.attn_fwd(q, k2, v2, causal=True, kv_len=kl)
    attn.attn_device_status()
    assert torch.equal(clean, poisoned)
    # and future keys under the causal mask: poison Q's view by making later K huge
    k3 = k.clone()
    k3[:, :, 300:] = 1e4
    full = attn.attn_fwd(q, k3, v, causal=True)
    ref = oracle.attention(q.cpu(), k3.cpu(), v.cpu(), causal=True)
    assert_close(full[:, :, :300], ref[:, :, :300], torch.bfloat16, "rows before huge keys")


@pytest.mark.parametrize("D", [64, 128])
def test_scale_zero_with_poisoned_hidden_keys(gpu, D):
    """scale = 0 and NaN/inf keys past kv_len: -inf * 0 would be NaN, so the
    hidden columns must still come out as exact zero weights; the result is the
    mean of the visible V rows (oracle pin 'uniform scores')."""
    B, H, S = 3, 2, 300
    lens = [77, 200, 300]
    q = wl.random_tensors((B, H, S, D), 23, count=1)[0]
    k, v = wl.random_tensors((B, H, S, D), 24, count=2)
    for b, L in enumerate(lens):
        k[b, :, L:] = float("nan")
        k[b, :, L::5] = float("-inf")
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = attn.attn_fwd(q, k, v, scale=0.0, causal=True, kv_len=kl)
    attn.attn_device_status()
    kc = k.clone()
    for b, L in enumerate(lens):
        kc[b, :, L:] = 0  # the oracle never reads hidden keys; keep its input finite anyway
    ref = oracle.attention(q.cpu(), kc.cpu(), v.cpu(), scale=0.0, causal=True,
                           kv_len=np.array(lens, np.int32))
    assert not torch.isnan(out).any()
    assert_close(out, ref, torch.bfloat16, f"scale 0 poisoned D={D}")


def test_no_write_outside_out(gpu):
    B, H, S, D = 1, 3, 257, 128
    q, k, v = wl.random_tensors((B, H, S, D), 30)
    n = B * H * S * D
    guard = 4096
    buf = torch.full((n + 2 * guard,), 7.0, dtype=torch.bfloat16, device="cuda")
    out = buf[guard:guard + n].view(B, H, S, D)
    attn.attn_fwd(q, k, v, out=out, causal=True)
    attn.attn_device_status()
    assert torch.all(buf[:guard] == 7.0) and torch.all(buf[guard + n:] == 7.0)


def test_empty_keys_give_zeros(gpu):
    q = torch.randn(2, 2, 5, 128, device="cuda").to(torch.bfloat16)
    k = torch.empty(2, 2, 0, 128, device="cuda", dtype=torch.bfloat16)
    out = torch.full_like(q, 3.0)
    attn.attn_fwd(q, k, k, out=out, causal=False)
    attn.attn_device_status()
    assert torch.count_nonzero(out) == 0


def test_stream_argument(gpu):
    s = torch.cuda.Stream()
    q, k, v = wl.random_tensors((2, 2, 256, 128), 40)
    with torch.cuda.stream(s):
        out = attn.attn_fwd(q, k, v, causal=True, stream=s)
    s.synchronize()
    ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=True)
    assert_close(out, ref, torch.bfloat16, "side stream")


def test_concurrent_streams_and_repeated_launches(gpu):
    """The persistent kernel hands out work through a device counter per
    launch: launches running at the same time on two streams must each cover
    their own problem, and back-to-back launches must start from a reset
    counter (every launch here reuses counters that earlier launches drained)."""
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    q1, k1, v1 = wl.random_tensors((4, 8, 1024, 128), 41)
    q2, k2, v2 = wl.random_tensors((3, 8, 768, 64), 42)
    ref1 = attn.attn_fwd(q1, k1, v1, causal=True).clone()
    ref2 = attn.attn_fwd(q2, k2, v2, causal=False).clone()
    torch.cuda.synchronize()
    outs = []
    for _ in range(40):
        with torch.cuda.stream(s1):
            o1 = attn.attn_fwd(q1, k1, v1, causal=True, stream=s1)
        with torch.cuda.stream(s2):
            o2 = attn.attn_fwd(q2, k2, v2, causal=False, stream=s2)
        outs.append((o1, o2))
    s1.synchronize()
    s2.synchronize()
    attn.attn_device_status()
    for o1, o2 in outs:
        assert torch.equal(o1, ref1)
        assert torch.equal(o2, ref2)
    r1 = oracle.attention_rows(q1.cpu(), k1.cpu(), v1.cpu(), np.array([[0, 0, 5], [3, 7, 1023]], np.int64),
                               causal=True)
    got = torch.stack([ref1[0, 0, 5], ref1[3, 7, 1023]]).cpu()
    assert_close(got, r1, torch.bfloat16, "two streams, spot rows")


def _sampled_rows(w, kv_len, per_head=6, seed=0):
    rng = np.random.default_rng(seed)
    rows = []
    for b in range(w.B):
        L = w.S if kv_len is None else int(kv_len[b])
        fixed = {0, 1, 127, 128, 129, w.S - 1}
        if kv_len is not None:
            fixed |= {max(L - 1, 0), min(L, w.S - 1)}
        for h in range(w.H):
            pick = set(fixed) | set(rng.integers(0, w.S, size=per_head).tolist())
            rows += [(b, h, i) for i in sorted(pick)]
    return np.array(rows, dtype=np.int64)


@pytest.mark.parametrize("name", ["prefill", "padded"])
def test_full_size_workloads_every_element(gpu, name):
    """The headline workload (B4 H32 S2048 D128 causal) and the padded one (B8
    H16 S4096 D128, causal + key padding) in the benchmark's launch
    configuration, compared with the oracle on every output element.  The
    max and mean bounds apply to every live row (query rows i < L_b); the
    padded query rows are checked bit-exact zero on their own, so that their
    exact zeros do not dilute the mean."""
    w = wl.PREFILL_WORKLOADS[name]
    q, k, v, kl = wl.prefill_inputs(w, device="cuda")
    out = attn.attn_fwd(q, k, v, scale=w.softmax_scale, causal=w.causal, kv_len=kl)
    attn.attn_device_status()
    kv_host = None if kl is None else kl.cpu().numpy()
    ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), scale=w.softmax_scale, causal=w.causal,
                           kv_len=kv_host)
    got = out.cpu()
    if kv_host is None:
        assert_close(got, ref, torch.bfloat16, w.name + ", every element")
        return
    live_got = torch.cat([got[b, :, :int(L)].reshape(-1, w.D) for b, L in enumerate(kv_host)])
    live_ref = np.concatenate([ref[b, :, :int(L)].reshape(-1, w.D) for b, L in enumerate(kv_host)])
    assert_close(live_got, live_ref, torch.bfloat16, w.name + ", every live row")
    for b, L in enumerate(kv_host):
        assert torch.count_nonzero(got[b, :, int(L):]) == 0, f"padded rows of sequence {b} not zero"
        assert np.all(ref[b, :, int(L):] == 0.0)


@pytest.mark.parametrize("name", ["prefill", "padded", "long"])
def test_full_size_workloads_sampled(gpu, name):
    """Full-size workloads in the benchmark's launch configuration; the oracle
    evaluates sampled rows one by one (every head, tile edges, padding edges).
    The long-context workload (2.2 TFLOP of fp64 work for the whole tensor)
    is checked this way only."""
    w = wl.PREFILL_WORKLOADS[name]
    q, k, v, kl = wl.prefill_inputs(w, device="cuda")
    out = attn.attn_fwd(q, k, v, scale=w.softmax_scale, causal=w.causal, kv_len=kl)
    attn.attn_device_status()
    kv_host = None if kl is None else kl.cpu().numpy()
    rows = _sampled_rows(w, kv_host, per_head=4 if name == "long" else 6, seed=w.seed)
    ref = oracle.attention_rows(q.cpu(), k.cpu(), v.cpu(), rows, scale=w.softmax_scale,
                                causal=w.causal, kv_len=kv_host)
    idx = torch.from_numpy(rows).to("cuda")
    got = out[idx[:, 0], idx[:, 1], idx[:, 2]]
    assert_close(got, ref, torch.bfloat16, w.name)
    if kv_host is not None:
        for b, L in enumerate(kv_host):
            assert torch.count_nonzero(out[b, :, int(L):]) == 0
    assert torch.isfinite(out.float()).all()


def test_decode_equals_last_causal_row(gpu):
    """The cache must not change the result ("Attention from scratch"
    (open-llm-engineering), "Decode"): decode of the newest query equals the
    last row of causal prefill over the same keys."""
    B, H, S, D = 3, 4, 777, 128
    q, k, v = wl.random_tensors((B, H, S, D), 50)
    full = attn.attn_fwd(q, k, v, causal=True)
    dec = attn.attn_decode(q[:, :, S - 1].contiguous(), k, v)
    attn.attn_device_status()
    diff = (full[:, :, S - 1].float() - dec.float()).abs().max().item()
    assert diff <= 2e-2


@pytest.mark.parametrize("S", [128, 65536])
@pytest.mark.parametrize("causal", [True, False])
def test_s_sweep_extremes_sampled(gpu, S, causal):
    """The sequence-length sweep's smallest and largest lengths (B4 H32 D128
    bf16; at S = 65536 a materialised score tensor would not fit in HBM), in
    the launch configuration the sweep times.  The oracle evaluates sampled
    rows of three (b, h) slices, each slice passed alone."""
    q, k, v = wl.s_sweep_inputs(S, "cuda")
    out = attn.attn_fwd(q, k, v, causal=causal)
    attn.attn_device_status()
    rng = np.random.default_rng(S + causal)
    B, H = q.shape[0], q.shape[1]
    for b, h in ((0, 0), (B - 1, H - 1), (1, 17)):
        pick = sorted(i for i in {0, 1, 127, 128, S // 2, S - 2, S - 1} | set(rng.integers(0, S, size=8).tolist())
                      if i < S)
        rows = np.array([(0, 0, i) for i in pick], dtype=np.int64)
        sl = (slice(b, b + 1), slice(h, h + 1))
        ref = oracle.attention_rows(q[sl].cpu(), k[sl].cpu(), v[sl].cpu(), rows, causal=causal)
        got = out[b, h, torch.tensor(pick, device="cuda")]
        assert_close(got, ref, torch.bfloat16, f"S={S} causal={causal} (b, h)=({b}, {h})")
    assert torch.isfinite(out[:, :, ::max(1, S // 1024)].float()).all()
