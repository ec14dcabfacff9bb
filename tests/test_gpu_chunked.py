"""GPU parity tests of attn_fwd_chunked: a chunk of new queries against a KV
cache, with the log-sum-exp of every row.

Sequence b holds cache_len[b] valid positions, the last Sq of them the chunk's
own keys; query i sits at position cache_len[b] - Sq + i and sees keys up to it
("Scaled dot-product attention with masking", the cache append before causal
attention; "Attention from scratch" (open-llm-engineering), "KV cache position
drift").  Outputs use the bf16/fp32 tolerances of test_gpu_prefill.py.  The
log-sum-exp is fp32 computed from fp32 scores: |error| <= 2e-4 for bf16
inputs and 2e-5 for fp32 inputs (scores of magnitude ~10 at most here).
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

LSE_TOL = {torch.bfloat16: 2e-4, torch.float32: 2e-5}


def _chunk_case(B, H, H_kv, Sq, Skv, D, lens, dtype=torch.bfloat16, seed=0, scale=None):
    q = wl.random_tensors((B, H, Sq, D), seed, dtype=dtype, count=1)[0]
    kc, vc = wl.random_tensors((B, H_kv, Skv, D), seed + 1000, dtype=dtype, count=2)
    cl = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens is not None else None
    out, lse = attn.attn_fwd_chunked(q, kc, vc, cache_len=cl, scale=scale, return_lse=True)
    attn.attn_device_status()
    ref, ref_lse = oracle.attention(q.cpu(), kc.cpu(), vc.cpu(), scale=scale, causal=True,
                                    cache_len=None if lens is None else np.array(lens, np.int32),
                                    need_lse=True)
    return q, kc, vc, out, lse, ref, ref_lse


def _check_lse(lse, ref_lse, dtype, what):
    got = lse.double().cpu().numpy()
    inf = np.isinf(ref_lse)
    assert np.array_equal(np.isinf(got), inf), f"{what}: -inf rows differ"
    assert np.all(got[inf] < 0)
    err = np.abs(got[~inf] - ref_lse[~inf])
    assert err.size == 0 or err.max() <= LSE_TOL[dtype], f"{what}: lse max err {err.max():.3e}"


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("H,H_kv", [(4, 4), (4, 2), (8, 1)])
@pytest.mark.parametrize("Sq,Skv", [(1, 600), (64, 64), (130, 600), (300, 1024)])
def test_chunk_against_cache(gpu, H, H_kv, Sq, Skv, D):
    lens = [Skv, max(Sq, Skv // 2 + 3), Sq, Sq // 2, 0]
    _, _, _, out, lse, ref, ref_lse = _chunk_case(len(lens), H, H_kv, Sq, Skv, D, lens, seed=Sq + Skv)
    what = f"H={H} H_kv={H_kv} Sq={Sq} Skv={Skv} D={D}"
    assert_close(out, ref, torch.bfloat16, what)
    _check_lse(lse, ref_lse, torch.bfloat16, what)
    # rows whose position precedes the sequence are exact zeros
    for b, L in enumerate(lens):
        if L < Sq:
            assert torch.count_nonzero(out[b, :, :Sq - L]) == 0


@pytest.mark.parametrize("H,H_kv", [(4, 4), (4, 2)])
def test_chunk_against_cache_fp32(gpu, H, H_kv):
    lens = [257, 200, 100, 31]
    _, _, _, out, lse, ref, ref_lse = _chunk_case(4, H, H_kv, 100, 257, 64, lens, dtype=torch.float32, seed=3)
    assert_close(out, ref, torch.float32, "fp32 chunk")
    _check_lse(lse, ref_lse, torch.float32, "fp32 chunk")


def test_chunk_without_lengths_equals_causal_prefill(gpu):
    """cache_len NULL: every sequence uses all Skv positions, which is causal
    attn_fwd_gqa with the last query aligned to the last key -- bit-exact."""
    B, H, H_kv, Sq, Skv, D = 2, 8, 2, 200, 700, 128
    q = wl.random_tensors((B, H, Sq, D), 51, count=1)[0]
    kc, vc = wl.random_tensors((B, H_kv, Skv, D), 52, count=2)
    out = attn.attn_fwd_chunked(q, kc, vc)
    ref = attn.attn_fwd(q, kc, vc, causal=True)
    attn.attn_device_status()
    assert torch.equal(out, ref)


def test_lse_merges_split_attention(gpu):
    """The use the log-sum-exp exists for: attention of the last query over a
    whole cache equals the exp(lse)-weighted merge of attention over the first
    half and over the second half of the cache (computed as two chunks whose
    visible keys are exactly those halves)."""
    B, H, S, D = 2, 4, 512, 128
    q = wl.random_tensors((B, H, 1, D), 61, count=1)[0]
    kc, vc = wl.random_tensors((B, H, S, D), 62, count=2)
    full, lse_full = attn.attn_fwd_chunked(q, kc, vc, return_lse=True)
    half = S // 2
    o1, l1 = attn.attn_fwd_chunked(q, kc[:, :, :half].contiguous(), vc[:, :, :half].contiguous(), return_lse=True)
    o2, l2 = attn.attn_fwd_chunked(q, kc[:, :, half:].contiguous(), vc[:, :, half:].contiguous(), return_lse=True)
    attn.attn_device_status()
    lse = torch.logaddexp(l1, l2)
    merged = (torch.exp(l1 - lse)[..., None] * o1.float() + torch.exp(l2 - lse)[..., None] * o2.float())
    assert torch.allclose(lse, lse_full, atol=2e-4, rtol=0)
    assert_close(merged, full.double().cpu().numpy(), torch.bfloat16, "merged halves")


def test_chunked_rejects_bad_arguments(gpu):
    q = torch.zeros(1, 2, 10, 64, device="cuda", dtype=torch.bfloat16)
    kc = torch.zeros(1, 2, 8, 64, device="cuda", dtype=torch.bfloat16)
    with pytest.raises(attn.AttnError) as e:
        attn.attn_fwd_chunked(q, kc, kc)  # Sq > Skv
    assert e.value.code == attn.ATTN_EINVAL
