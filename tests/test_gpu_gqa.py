"""GPU parity tests of grouped-query and multi-query attention (H_kv < H).

Query head h reads key/value head h // (H // H_kv): the pages' repeat_interleave
of K and V along the head axis ("Attention from First Principles", section 5;
"Scaled dot-product attention with masking", "Grouped-query attention (GQA)").
The prefill kernel pairs two heads of one group per work item when the group
size is even (one K/V tile in shared memory serves both), and two query tiles
of one head otherwise; both are checked here.  Tolerances as in
test_gpu_prefill.py.
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


def _gqa_case(B, H, H_kv, Sq, Skv, D, causal, dtype=torch.bfloat16, kv_len=None, seed=0):
    q = wl.random_tensors((B, H, Sq, D), seed, dtype=dtype, count=1)[0]
    k, v = wl.random_tensors((B, H_kv, Skv, D), seed + 1000, dtype=dtype, count=2)
    kl = torch.tensor(kv_len, dtype=torch.int32, device="cuda") if kv_len is not None else None
    out = attn.attn_fwd(q, k, v, causal=causal, kv_len=kl)
    attn.attn_device_status()
    ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=causal,
                           kv_len=None if kv_len is None else np.array(kv_len, np.int32))
    return q, k, v, kl, out, ref


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(8, 2), (6, 2), (8, 1), (4, 4), (6, 3)])
@pytest.mark.parametrize("S", [1, 129, 300, 513])
@pytest.mark.parametrize("causal", [True, False])
def test_gqa_prefill_bf16(gpu, H, H_kv, S, D, causal):
    _, _, _, _, out, ref = _gqa_case(2, H, H_kv, S, S, D, causal, seed=S + H * 10 + H_kv)
    assert_close(out, ref, torch.bfloat16, f"H={H} H_kv={H_kv} S={S} D={D} causal={causal}")


@pytest.mark.parametrize("H,H_kv", [(8, 2), (6, 2), (4, 1)])
def test_gqa_prefill_fp32(gpu, H, H_kv):
    _, _, _, _, out, ref = _gqa_case(2, H, H_kv, 130, 130, 64, True, dtype=torch.float32, seed=7)
    assert_close(out, ref, torch.float32, f"fp32 H={H} H_kv={H_kv}")


@pytest.mark.parametrize("H,H_kv", [(8, 2), (6, 2), (8, 1)])
def test_gqa_equals_mha_on_repeated_kv(gpu, H, H_kv):
    """Bit-exact: every (query tile, head) runs the same tile sequence whichever
    way the work items pair them, so grouped K/V must give exactly the output
    of multi-head attention on K/V repeated along the head axis."""
    q, k, v, _, out, _ = _gqa_case(2, H, H_kv, 384, 384, 128, True, seed=11)
    G = H // H_kv
    out_mha = attn.attn_fwd(q, k.repeat_interleave(G, dim=1).contiguous(),
                            v.repeat_interleave(G, dim=1).contiguous(), causal=True)
    attn.attn_device_status()
    assert torch.equal(out, out_mha)


@pytest.mark.parametrize("H,H_kv", [(8, 2), (6, 3)])
def test_gqa_key_padding_and_cross(gpu, H, H_kv):
    lens = [0, 1, 127, 128, 300]
    _, _, _, _, out, ref = _gqa_case(len(lens), H, H_kv, 300, 300, 128, True, kv_len=lens, seed=13)
    assert_close(out, ref, torch.bfloat16, "grouped, key padding")
    for b, L in enumerate(lens):
        assert torch.count_nonzero(out[b, :, L:]) == 0
    _, _, _, _, out, ref = _gqa_case(1, H, H_kv, 100, 700, 128, True, seed=14)
    assert_close(out, ref, torch.bfloat16, "grouped, chunk against a longer key sequence")


def test_gqa_full_size_sampled(gpu):
    """Llama-like grouping at the prefill benchmark size: B4 H32 H_kv 8 S2048 D128."""
    B, H, H_kv, S, D = 4, 32, 8, 2048, 128
    g = torch.Generator(device="cuda").manual_seed(21)
    q = torch.randn(B, H, S, D, device="cuda", generator=g).to(torch.bfloat16)
    k = torch.randn(B, H_kv, S, D, device="cuda", generator=g).to(torch.bfloat16)
    v = torch.randn(B, H_kv, S, D, device="cuda", generator=g).to(torch.bfloat16)
    out = attn.attn_fwd(q, k, v, causal=True)
    attn.attn_device_status()
    rng = np.random.default_rng(0)
    rows = np.array([(b, h, i) for b in range(B) for h in range(H)
                     for i in sorted({0, 127, 128, S - 1} | set(rng.integers(0, S, 3).tolist()))], np.int64)
    ref = oracle.attention_rows(q.cpu(), k.cpu(), v.cpu(), rows, causal=True)
    got = out[rows[:, 0], rows[:, 1], rows[:, 2]]
    assert_close(got, ref, torch.bfloat16, "B4 H32 H_kv8 S2048 sampled rows")


def test_gqa_rejects_bad_grouping(gpu):
    q = torch.zeros(1, 6, 8, 64, device="cuda", dtype=torch.bfloat16)
    k = torch.zeros(1, 4, 8, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        attn.attn_fwd(q, k, k, causal=True)
    out = torch.empty_like(q)
    P = attn.ctypes.c_void_p
    rc = attn.lib().attn_fwd_gqa(P(q.data_ptr()), P(k.data_ptr()), P(k.data_ptr()), P(out.data_ptr()),
                                 1, 6, 4, 8, 8, 64, attn.ctypes.c_float(0.125), 1, None, 1, None)
    assert rc == attn.ATTN_EINVAL and "H_kv" in attn.attn_last_error()


# ----------------------------------------------------------------- decode

def _decode_case(B, H, H_kv, Skv, D, kv_len=None, seed=0):
    q = wl.random_tensors((B, H, D), seed, count=1)[0]
    kc, vc = wl.random_tensors((B, H_kv, Skv, D), seed + 1000, count=2)
    kl = torch.tensor(kv_len, dtype=torch.int32, device="cuda") if kv_len is not None else None
    out = attn.attn_decode(q, kc, vc, kv_len=kl)
    attn.attn_device_status()
    ref = oracle.decode(q.cpu(), kc.cpu(), vc.cpu(),
                        kv_len=None if kv_len is None else np.array(kv_len, np.int32))
    return q, kc, vc, out, ref


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(8, 2), (8, 4), (6, 2), (12, 1), (32, 1), (32, 8)])
@pytest.mark.parametrize("Skv", [1, 63, 65, 700, 3000])
def test_gqa_decode(gpu, H, H_kv, Skv, D):
    """Group sizes 2, 3, 4, 12 (a subgroup of 8 plus one of 4) and 32 (four
    subgroups of 8), ragged chunk tails."""
    _, _, _, out, ref = _decode_case(2, H, H_kv, Skv, D, seed=Skv + H + H_kv)
    assert_close(out, ref, torch.bfloat16, f"decode H={H} H_kv={H_kv} Skv={Skv} D={D}")


@pytest.mark.parametrize("H,H_kv", [(8, 2), (32, 1)])
def test_gqa_decode_lengths(gpu, H, H_kv):
    lens = [0, 1, 64, 65, 511, 512, 513, 2000]
    _, _, _, out, ref = _decode_case(len(lens), H, H_kv, 2000, 128, kv_len=lens, seed=5)
    assert_close(out, ref, torch.bfloat16, "grouped decode, per-sequence lengths")
    assert torch.count_nonzero(out[0]) == 0


def test_gqa_decode_equals_last_causal_row(gpu):
    B, H, H_kv, S, D = 2, 8, 2, 300, 128
    q = wl.random_tensors((B, H, S, D), 31, count=1)[0]
    k, v = wl.random_tensors((B, H_kv, S, D), 32, count=2)
    full = attn.attn_fwd(q, k, v, causal=True)
    dec = attn.attn_decode(q[:, :, S - 1].contiguous(), k, v)
    attn.attn_device_status()
    assert_close(dec, full[:, :, S - 1].double().cpu().numpy(), torch.bfloat16, "decode vs last prefill row")


def test_gqa_decode_full_size_sampled(gpu):
    """The decode workload's shape with Llama-like grouping: B64 H32 H_kv8, cache
    padded to 8192, lengths U{4096..8192}."""
    w = wl.DECODE
    B, H, H_kv, S, D = w.B, w.H, 8, w.Skv, w.D
    g = torch.Generator(device="cuda").manual_seed(41)
    q = torch.randn(B, H, D, device="cuda", generator=g).to(torch.bfloat16)
    kc = torch.randn(B, H_kv, S, D, device="cuda", generator=g).to(torch.bfloat16)
    vc = torch.randn(B, H_kv, S, D, device="cuda", generator=g).to(torch.bfloat16)
    lens = torch.randint(4096, 8193, (B,), generator=torch.Generator().manual_seed(42), dtype=torch.int32)
    out = attn.attn_decode(q, kc, vc, kv_len=lens.cuda())
    attn.attn_device_status()
    bs = [0, 1, 17, 63]
    ref = oracle.decode(q[bs].cpu(), kc[bs].cpu(), vc[bs].cpu(), kv_len=lens[bs].numpy())
    assert_close(out[bs], ref, torch.bfloat16, "B64 H32 H_kv8 decode, sampled sequences")
