"""GPU tests of attn_fwd_debug (general attention with weights) and of
non-causal cross-attention with a padded source on the fast paths.

attn_fwd_debug computes in fp32 (one warp per query row): outputs match the
oracle within the fp32 tolerance (1e-4) for fp32 inputs and the bf16
tolerances for bf16 inputs; weights within 1e-5 (fp32 softmax of fp32 scores,
values in [0, 1]).
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_fwd_gb300 as attn
from transformer_scaled_dot_fwd_gb300 import workloads as wl
from helpers import assert_close
from oracle_pins import load_golden

pytestmark = pytest.mark.gpu

W_TOL = 1e-5


@pytest.mark.parametrize("name", ["tiny_example_causal_t3_d2.txt", "kube_dojo_example_dk4_dv2.txt"])
def test_pages_worked_examples_on_gpu(gpu, name):
    """The printed weights and outputs of the pages' worked examples ('Attention
    from First Principles', section 4; 'Attention from Scratch' (kube-dojo),
    Part 2, d_k = 4, d_v = 2) reproduced by the GPU debug path."""
    meta, m = load_golden(name)
    q = torch.tensor(m["Q"], dtype=torch.float32, device="cuda")[None, None].contiguous()
    k = torch.tensor(m["K"], dtype=torch.float32, device="cuda")[None, None].contiguous()
    v = torch.tensor(m["V"], dtype=torch.float32, device="cuda")[None, None].contiguous()
    dk = q.shape[-1]
    scale = 1.0 / math.sqrt(dk) if meta["scale"] == "inv_sqrt_dk" else float(meta["scale"])
    out, w = attn.attn_fwd_debug(q, k, v, scale=scale, causal=bool(int(meta["causal"])), return_weights=True)
    attn.attn_device_status()
    np.testing.assert_allclose(w[0, 0].cpu().numpy(), m["weights"], rtol=0, atol=float(meta["tol_weights"]))
    np.testing.assert_allclose(out[0, 0].cpu().numpy(), m["out"], rtol=0, atol=float(meta["tol_out"]))


CASES = [  # (B, H, H_kv, Sq, Skv, Dk, Dv, causal, kv_len)
    (2, 3, 3, 4, 7, 16, 8, False, None),           # cross-attention, d_v != d_k
    (2, 2, 2, 4, 7, 32, 32, False, [7, 3]),        # padded source (Part 7 shape test)
    (1, 4, 2, 9, 9, 5, 3, True, None),             # odd depths, grouped heads
    (3, 2, 1, 33, 33, 64, 24, True, [33, 10, 0]),  # self-attention batch with padding
    (1, 2, 2, 5, 300, 128, 64, True, None),        # chunk of queries against a longer key set
]


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("case", CASES)
def test_debug_matches_oracle_with_weights(gpu, case, dtype):
    B, H, H_kv, Sq, Skv, Dk, Dv, causal, kl = case
    q = wl.random_tensors((B, H, Sq, Dk), 70 + Sq, dtype=dtype, count=1)[0]
    k = wl.random_tensors((B, H_kv, Skv, Dk), 71 + Skv, dtype=dtype, count=1)[0]
    v = wl.random_tensors((B, H_kv, Skv, Dv), 72 + Dv, dtype=dtype, count=1)[0]
    kl_t = torch.tensor(kl, dtype=torch.int32, device="cuda") if kl is not None else None
    out, w = attn.attn_fwd_debug(q, k, v, causal=causal, kv_len=kl_t, return_weights=True)
    attn.attn_device_status()
    ref, ref_w = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=causal,
                                  kv_len=None if kl is None else np.array(kl, np.int32), need_weights=True)
    assert_close(out, ref, dtype, f"debug {case}")
    got_w = w.double().cpu().numpy()
    assert np.abs(got_w - ref_w).max() <= W_TOL
    # forbidden weights are exact zeros; each row that sees a key sums to one
    assert np.all(got_w[ref_w == 0.0] == 0.0)
    sums = got_w.sum(-1)
    seen = ref_w.sum(-1) > 0
    assert np.abs(sums[seen] - 1.0).max() <= 1e-5
    assert np.all(sums[~seen] == 0.0)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("D", [64, 128])
def test_cross_attention_with_padded_source(gpu, D, dtype):
    """'Attention from Scratch' (kube-dojo), Part 7: T_target = 4, T_source = 7,
    and a source padding mask whose last dimension is 7 -- on the fast paths
    (tensor-core bf16 and fp32), where kv_len with Sq != Skv masks keys only."""
    B, H, Sq, Skv = 3, 2, 4, 7
    lens = [7, 5, 1]
    q = wl.random_tensors((B, H, Sq, D), 81, dtype=dtype, count=1)[0]
    k, v = wl.random_tensors((B, H, Skv, D), 82, dtype=dtype, count=2)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out = attn.attn_fwd(q, k, v, causal=False, kv_len=kl)
    attn.attn_device_status()
    assert out.shape == (B, H, Sq, D)
    ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=False, kv_len=np.array(lens, np.int32))
    assert_close(out, ref, dtype, f"cross-attention D={D}")
    # longer source, several tiles and a ragged tail
    q = wl.random_tensors((3, 4, 100, D), 83, dtype=dtype, count=1)[0]
    k, v = wl.random_tensors((3, 4, 700, D), 84, dtype=dtype, count=2)
    lens = [700, 333, 0]
    out = attn.attn_fwd(q, k, v, causal=False, kv_len=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    attn.attn_device_status()
    ref = oracle.attention(q.cpu(), k.cpu(), v.cpu(), causal=False, kv_len=np.array(lens, np.int32))
    assert_close(out, ref, dtype, f"cross-attention 100x700 D={D}")
    assert torch.count_nonzero(out[2]) == 0  # an empty source gives zero rows
