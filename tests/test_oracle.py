"""CPU tests of the fp64 oracle: its pins, its row-sampling entry point, and
planted mistakes that the pins must catch."""
from __future__ import annotations

import os
import shutil

import numpy as np
import pytest
import torch

import oracle
from oracle_pins import ALL_PINS


@pytest.mark.parametrize("pin", ALL_PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    pin(oracle.attention)


def test_rows_entry_matches_full():
    g = torch.Generator().manual_seed(3)
    B, H, S, D = 2, 3, 37, 16
    q, k, v = (torch.randn(B, H, S, D, generator=g).to(torch.bfloat16) for _ in range(3))
    kv_len = torch.tensor([37, 20], dtype=torch.int32)
    full = oracle.attention(q, k, v, causal=True, kv_len=kv_len)
    rows = np.array([(b, h, i) for b in range(B) for h in range(H) for i in (0, 1, 19, 20, 36)])
    got = oracle.attention_rows(q, k, v, rows, causal=True, kv_len=kv_len)
    want = np.stack([full[b, h, i] for b, h, i in rows])
    assert np.array_equal(got, want)


def test_rows_entry_matches_full_grouped():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((2, 6, 9, 4)).astype(np.float32)
    k = rng.standard_normal((2, 2, 9, 4)).astype(np.float32)
    v = rng.standard_normal((2, 2, 9, 4)).astype(np.float32)
    kl = np.array([9, 5], np.int32)
    full = oracle.attention(q, k, v, causal=True, kv_len=kl)
    rows = np.array([[0, 0, 0], [0, 5, 8], [1, 3, 4], [1, 4, 7], [1, 1, 2]], np.int64)
    got = oracle.attention_rows(q, k, v, rows, causal=True, kv_len=kl)
    assert np.array_equal(got, full[rows[:, 0], rows[:, 1], rows[:, 2]])


def test_bf16_inputs_are_widened_exactly():
    g = torch.Generator().manual_seed(4)
    q, k, v = (torch.randn(1, 2, 9, 8, generator=g).to(torch.bfloat16) for _ in range(3))
    a = oracle.attention(q, k, v, causal=True)
    b = oracle.attention(q.float(), k.float(), v.float(), causal=True)
    assert np.array_equal(a, b)


def test_decode_helper_shape():
    g = torch.Generator().manual_seed(5)
    q = torch.randn(3, 2, 8, generator=g)
    kc, vc = torch.randn(3, 2, 10, 8, generator=g), torch.randn(3, 2, 10, 8, generator=g)
    kv_len = torch.tensor([10, 1, 0], dtype=torch.int32)
    out = oracle.decode(q, kc, vc, kv_len=kv_len)
    assert out.shape == (3, 2, 8)
    np.testing.assert_array_equal(out[1], vc[1, :, 0].double().numpy())  # one key: its value
    assert np.all(out[2] == 0.0)


def test_rejects_bad_arguments():
    q = np.zeros((1, 1, 2, 4), np.float32)
    with pytest.raises(ValueError):
        oracle.attention(q, np.zeros((1, 1, 3, 5), np.float32), np.zeros((1, 1, 3, 4), np.float32))
    with pytest.raises(ValueError):
        oracle.attention_rows(q, q, q, [(0, 0, 2)])


# Planted mistakes: each replaces one fragment of oracle.c in a private copy.
# Every mutant stays inside its arrays; each must fail at least one pin.
MUTANTS = {
    "mask_polarity_flipped": ("if (causal && j > i + off)", "if (causal && j < i + off)"),
    "causal_diagonal_excluded": ("if (causal && j > i + off)", "if (causal && j >= i + off)"),
    "scale_dropped": ("s_row[j] = scale * dot;", "s_row[j] = dot;"),
    "max_not_subtracted": ("exp(s_row[j] - m)", "exp(s_row[j])"),
    "not_normalised": ("double w = exp(s_row[j] - m) / z;", "double w = exp(s_row[j] - m);"),
    "padding_off_by_one": ("if (j >= Lb)\n        return 0;", "if (j > Lb)\n        return 0;"),
    "value_rows_reversed": ("v_bh + (size_t)j * Dv + d", "v_bh + (size_t)(Skv - 1 - j) * Dv + d"),
    "dot_drops_last_term": ("for (d = 0; d < Dk; d++)\n            dot +=",
                            "for (d = 0; d < Dk - 1; d++)\n            dot +="),
    "padded_queries_kept": ("if (query_padding && i >= Lb)\n        return;",
                            "if (query_padding && i >= Lb && 0)\n        return;"),
    "lse_without_max": ("*lse = m + log(z);", "*lse = log(z);"),
    "cache_offset_from_capacity": ("Lb - Sq, Skv, Dk, Dv, scale, 1, Lb, 0,", "Skv - Sq, Skv, Dk, Dv, scale, 1, Lb, 0,"),
    "kv_head_by_modulo": ("size_t pkv = (size_t)b * Hkv + h / G;", "size_t pkv = (size_t)b * Hkv + h % Hkv;"),
    "length_clamp_dropped": ("    if (L < 0)\n        L = 0;\n    if (L > Skv)\n        L = Skv;\n", ""),
    "keys_from_query_row": ("load_elem(k, dtype, k_bh + (size_t)j * Dk + d)",
                            "load_elem(k, dtype, k_bh + (size_t)j * Dk + d) * 0.0 + "
                            "load_elem(q, dtype, q_bh + (size_t)i * Dk + d)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(os.path.join(os.path.dirname(oracle.__file__), "oracle.c")).read()
    count = src.count(old)
    assert count >= 1, f"mutation anchor for {name} not found in oracle.c"
    mutated = tmp_path / "oracle_mut.c"
    mutated.write_text(src.replace(old, new))
    lib_path = oracle.build(force=True, src=str(mutated), out=str(tmp_path / "liboracle_mut.so"))
    lib = oracle.load(lib_path)

    def att(*a, **kw):
        return oracle.attention(*a, lib=lib, **kw)

    caught = []
    with np.errstate(all="ignore"):
        for pin in ALL_PINS:
            try:
                pin(att)
            except Exception:  # noqa: BLE001 - any failure of a pin counts as a catch
                caught.append(pin.__name__)
    assert caught, f"planted mistake {name} passed every pin"
    shutil.rmtree(tmp_path, ignore_errors=True)
