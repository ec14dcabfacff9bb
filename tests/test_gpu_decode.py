"""GPU parity tests of attn_decode (through the C ABI) against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import transformer_scaled_dot_fwd_gb300 as attn
from transformer_scaled_dot_fwd_gb300 import workloads as wl
from helpers import assert_close

pytestmark = pytest.mark.gpu


def decode_case(B, H, Skv, D, lens=None, seed=0):
    q = wl.random_tensors((B, H, D), seed, count=1)[0]
    kc, vc = wl.random_tensors((B, H, Skv, D), seed + 1, count=2)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda") if lens is not None else None
    out = attn.attn_decode(q, kc, vc, kv_len=kl)
    attn.attn_device_status()
    ref = oracle.decode(q.cpu(), kc.cpu(), vc.cpu(),
                        kv_len=None if lens is None else np.array(lens, np.int32))
    return q, kc, vc, out, ref


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("Skv", [1, 2, 63, 64, 65, 100, 511, 512, 513, 1024, 1500, 4097])
def test_shapes(gpu, Skv, D):
    _, _, _, out, ref = decode_case(2, 3, Skv, D, seed=Skv)
    assert_close(out, ref, torch.bfloat16, f"decode Skv={Skv} D={D}")


@pytest.mark.parametrize("D", [64, 128])
def test_length_edges(gpu, D):
    Skv = 1100
    lens = [0, 1, 63, 64, 65, 511, 512, 513, 1023, 1024, 1025, 1099, 1100]
    _, _, vc, out, ref = decode_case(len(lens), 2, Skv, D, lens=lens, seed=D)
    assert_close(out, ref, torch.bfloat16, f"decode length edges D={D}")
    assert torch.count_nonzero(out[0]) == 0          # kv_len 0 -> zeros
    assert torch.equal(out[1], vc[1, :, 0])           # one key -> its value


def test_split_counts_agree(gpu):
    """Small batches split the cache into shorter chunks; the merged result must
    not depend on how the keys were split (softmax split identity)."""
    D, Skv = 128, 3000
    q = wl.random_tensors((1, 1, D), 3, count=1)[0]
    kc, vc = wl.random_tensors((1, 1, Skv, D), 4, count=2)
    small = attn.attn_decode(q, kc, vc)
    reps = 64  # the same head repeated: a larger batch, longer chunks
    big = attn.attn_decode(q.expand(reps, 1, D).contiguous(), kc.expand(reps, 1, Skv, D).contiguous(),
                           vc.expand(reps, 1, Skv, D).contiguous())
    attn.attn_device_status()
    assert attn.attn_decode_splits(1, 1, Skv, D) != attn.attn_decode_splits(reps, 1, Skv, D)
    assert (small.float() - big[:1].float()).abs().max().item() <= 4e-3
    ref = oracle.decode(q.cpu(), kc.cpu(), vc.cpu())
    assert_close(small, ref, torch.bfloat16, "few-key chunks")
    assert_close(big[:1], ref, torch.bfloat16, "long chunks")


def test_padding_values_are_never_read(gpu):
    """Cache positions at or past kv_len are never loaded: NaN there changes nothing."""
    B, H, Skv, D = 3, 2, 700, 128
    lens = [100, 513, 700]
    q = wl.random_tensors((B, H, D), 7, count=1)[0]
    kc, vc = wl.random_tensors((B, H, Skv, D), 8, count=2)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    clean = attn.attn_decode(q, kc, vc, kv_len=kl).clone()
    for b, L in enumerate(lens):
        kc[b, :, L:] = float("nan")
        vc[b, :, L:] = float("nan")
    poisoned = attn.attn_decode(q, kc, vc, kv_len=kl)
    attn.attn_device_status()
    assert torch.equal(clean, poisoned)


def test_full_size_decode_workload(gpu):
    """B64 H32 D128, cache padded to 8192, lengths uniform on [4096, 8192]: every
    (b, h) output against the oracle."""
    w = wl.DECODE
    q, kc, vc, kl = wl.decode_inputs(w, device="cuda")
    out = attn.attn_decode(q, kc, vc, kv_len=kl)
    attn.attn_device_status()
    ref = oracle.decode(q.cpu(), kc.cpu(), vc.cpu(), kv_len=kl.cpu().numpy())
    assert_close(out, ref, torch.bfloat16, w.name)


def test_repeat_calls_are_deterministic(gpu):
    _, kc, vc, out, _ = decode_case(4, 4, 2000, 128, lens=[2000, 10, 1500, 999], seed=9)
    q = wl.random_tensors((4, 4, 128), 9, count=1)[0]
    kl = torch.tensor([2000, 10, 1500, 999], dtype=torch.int32, device="cuda")
    again = attn.attn_decode(q, kc, vc, kv_len=kl)
    attn.attn_device_status()
    assert torch.equal(out, again)


def test_device_wait_timeout_is_reported(gpu):
    """A device-side wait that can never complete gives up after its limit and
    surfaces as ATTN_ETIMEOUT on the host; the context stays usable."""
    attn.attn_device_status()  # clean slate
    attn.attn_selftest_wait_timeout(1_000_000)
    with pytest.raises(attn.AttnError) as e:
        attn.attn_device_status()
    assert e.value.code == attn.ATTN_ETIMEOUT
    attn.attn_device_status()  # the word was cleared
    _, _, _, out, ref = decode_case(1, 2, 300, 128, seed=77)  # and the device still works
    assert_close(out, ref, torch.bfloat16, "after timeout self-test")
