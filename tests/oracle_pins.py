"""Pins for the fp64 oracle: checks against what the pages and mathematics fix.

Each ``pin_*`` function takes ``att`` (a callable with the signature of
``oracle.attention``) and raises AssertionError when the oracle disagrees with
a printed worked example, a closed form, an invariant or an independent
library routine.  ``test_oracle.py`` runs every pin against the oracle, and
runs them again against copies of ``oracle.c`` with planted mistakes to show
that each mistake is caught by at least one pin.
"""
from __future__ import annotations

import math
import os

import numpy as np
import torch
import torch.nn.functional as F

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    """Parse a worked-example fixture: header keys, then named matrices."""
    meta, mats, cur = {}, {}, None
    with open(os.path.join(GOLDEN, name)) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if len(parts) == 1 and not _is_number(parts[0]):
                cur = parts[0]
                mats[cur] = []
            elif cur is None:
                meta[parts[0]] = parts[1]
            else:
                mats[cur].append([float(x) for x in parts])
    return meta, {k: np.array(v, dtype=np.float64) for k, v in mats.items()}


def _is_number(s):
    try:
        float(s)
        return True
    except ValueError:
        return False


def _golden_case(att, name):
    meta, m = load_golden(name)
    q = m["Q"][None, None].astype(np.float32)
    k = m["K"][None, None].astype(np.float32)
    v = m["V"][None, None].astype(np.float32)
    dk = q.shape[-1]
    scale = 1.0 / math.sqrt(dk) if meta["scale"] == "inv_sqrt_dk" else float(meta["scale"])
    out, w = att(q, k, v, scale=scale, causal=bool(int(meta["causal"])), need_weights=True)
    np.testing.assert_allclose(w[0, 0], m["weights"], rtol=0, atol=float(meta["tol_weights"]))
    np.testing.assert_allclose(out[0, 0], m["out"], rtol=0, atol=float(meta["tol_out"]))


def pin_tiny_example_causal(att):
    """'Attention from First Principles', section 4: printed weights and outputs."""
    _golden_case(att, "tiny_example_causal_t3_d2.txt")


def pin_kube_dojo_example(att):
    """'Attention from Scratch' (kube-dojo), Part 2: d_k = 4, d_v = 2, no mask."""
    _golden_case(att, "kube_dojo_example_dk4_dv2.txt")


def _rand(shape, seed, scale=1.0):
    g = np.random.default_rng(seed)
    return (g.standard_normal(shape) * scale).astype(np.float32)


def pin_rows_are_distributions(att):
    """Each allowed row of weights sums to one; forbidden weights are exactly 0.

    'Attention from scratch' (open-llm-engineering), readable implementation
    asserts; 'Attention from Scratch' (kube-dojo), Part 7 row-sum and
    forbidden-probability checks, for causal + key padding combined.
    """
    B, H, S, D = 3, 2, 9, 5
    q, k, v = _rand((B, H, S, D), 1), _rand((B, H, S, D), 2), _rand((B, H, S, D), 3)
    kv_len = np.array([9, 4, 1], dtype=np.int32)
    _, w = att(q, k, v, causal=True, kv_len=kv_len, need_weights=True)
    for b in range(B):
        L = kv_len[b]
        for i in range(S):
            row = w[b, :, i, :]
            if i >= L:
                assert np.all(row == 0.0)
                continue
            np.testing.assert_allclose(row.sum(-1), 1.0, rtol=0, atol=1e-12)
            forbidden = [j for j in range(S) if j > i or j >= L]
            assert np.all(row[:, forbidden] == 0.0)
            allowed = [j for j in range(S) if j <= i and j < L]
            assert np.all(row[:, allowed] > 0.0)


def pin_causal_first_row_is_v0(att):
    """Causal row 0 can only see key 0, so out[0] = V[0] exactly.

    'Attention from First Principles', section 4 ("Token 0 could only see
    itself, so it got V[0] unchanged").
    """
    q, k, v = _rand((2, 3, 6, 8), 4), _rand((2, 3, 6, 8), 5), _rand((2, 3, 6, 8), 6)
    out = att(q, k, v, causal=True)
    assert np.array_equal(out[:, :, 0, :], v[:, :, 0, :].astype(np.float64))


def pin_zero_qk_prefix_mean(att):
    """Zero queries and keys give uniform causal weights: out[i] = mean(V[0..i]).

    'Attention from scratch' (open-llm-engineering), Exercises, item 1.
    """
    S, D = 7, 4
    q = np.zeros((1, 2, S, D), np.float32)
    k = np.zeros((1, 2, S, D), np.float32)
    v = _rand((1, 2, S, D), 7)
    out, w = att(q, k, v, causal=True, need_weights=True)
    for i in range(S):
        np.testing.assert_allclose(out[:, :, i], v[:, :, : i + 1].astype(np.float64).mean(2),
                                   rtol=0, atol=1e-12)
        np.testing.assert_allclose(w[0, 0, i, : i + 1], 1.0 / (i + 1), rtol=0, atol=1e-15)


def pin_uniform_scores_with_padding(att):
    """scale = 0 makes every visible score equal: out = mean of the visible V rows,
    and padded query rows are zero (causal AND key padding, 'Attention from
    Scratch' (kube-dojo), Part 3)."""
    B, S, D = 2, 6, 3
    q, k, v = _rand((B, 1, S, D), 8), _rand((B, 1, S, D), 9), _rand((B, 1, S, D), 10)
    kv_len = np.array([4, 6], dtype=np.int32)
    out = att(q, k, v, scale=0.0, causal=True, kv_len=kv_len)
    for b in range(B):
        for i in range(S):
            if i >= kv_len[b]:
                assert np.all(out[b, 0, i] == 0.0)
            else:
                vis = min(i, kv_len[b] - 1) + 1
                np.testing.assert_allclose(out[b, 0, i], v[b, 0, :vis].astype(np.float64).mean(0),
                                           rtol=0, atol=1e-12)


def pin_permutation_equivariance(att):
    """Without a mask, permuting K and V rows together leaves the output
    unchanged and permuting Q rows permutes the output rows ('Self-Attention',
    "Related": self-attention is permutation-equivariant)."""
    q, k, v = _rand((1, 2, 5, 6), 11), _rand((1, 2, 7, 6), 12), _rand((1, 2, 7, 3), 13)
    base = att(q, k, v)
    pk = np.random.default_rng(14).permutation(7)
    pq = np.random.default_rng(15).permutation(5)
    np.testing.assert_allclose(att(q, k[:, :, pk], v[:, :, pk]), base, rtol=0, atol=1e-12)
    np.testing.assert_allclose(att(q[:, :, pq], k, v), base[:, :, pq], rtol=0, atol=1e-12)


def pin_shift_invariance_large(att):
    """Adding one vector u to every key shifts row i's scores by scale*q_i.u,
    which the max-subtracted softmax cancels.  With |scale*q_i.u| near 1e3 an
    unsubtracted exp overflows double, so this also pins overflow safety
    ('Attention from Scratch' (kube-dojo), Part 7, stable softmax)."""
    S, D = 6, 4
    q = _rand((1, 1, S, D), 16)
    q[..., 0] = np.abs(q[..., 0]) + 2.0
    # keys on a 2^-8 grid, so that k + 1024 is exact in float32
    k = np.round(_rand((1, 1, S, D), 17) * 256.0).astype(np.float32) / np.float32(256.0)
    v = _rand((1, 1, S, D), 18)
    u = np.zeros(D, np.float32)
    u[0] = 1024.0
    assert np.array_equal((k + u) - u, k)
    base = att(q, k, v)
    shifted = att(q, k + u, v)
    assert np.all(np.isfinite(shifted))
    np.testing.assert_allclose(shifted, base, rtol=0, atol=1e-9)


def pin_large_scale_is_hard_lookup(att):
    """As the scale grows the softmax tends to a one-hot at the best key, so
    attention becomes a hard lookup of that key's value ('Attention from
    Scratch' (kube-dojo), Part 1: soft dictionary lookup)."""
    q, k, v = _rand((1, 1, 4, 8), 19), _rand((1, 1, 9, 8), 20), _rand((1, 1, 9, 3), 21)
    out = att(q, k, v, scale=1e4)
    best = np.argmax(q[0, 0].astype(np.float64) @ k[0, 0].astype(np.float64).T, axis=1)
    np.testing.assert_allclose(out[0, 0], v[0, 0, best].astype(np.float64), rtol=0, atol=1e-9)


def _torch_sdpa_f64(q, k, v, allowed, scale):
    return F.scaled_dot_product_attention(
        torch.from_numpy(q.astype(np.float64)), torch.from_numpy(k.astype(np.float64)),
        torch.from_numpy(v.astype(np.float64)), attn_mask=torch.from_numpy(allowed),
        dropout_p=0.0, scale=scale).numpy()


def pin_matches_library_sdpa(att):
    """Agreement with PyTorch's own scaled_dot_product_attention in float64 on
    CPU, on random tiny shapes with explicit allowed-masks (True = allowed, as
    'Attention from Scratch' (kube-dojo), Part 6 describes).  Rows with no
    allowed key are skipped here; the library gives NaN for them."""
    cases = [  # (B, H, Sq, Skv, Dk, Dv, causal, kv_len)
        (2, 3, 5, 5, 8, 8, True, None),
        (2, 2, 4, 7, 6, 6, False, None),          # cross-attention shape test, Part 7
        (3, 2, 8, 8, 4, 4, True, [8, 3, 5]),      # causal + key padding
        (1, 2, 3, 9, 5, 5, True, None),           # chunk of queries against a longer cache
        (2, 1, 4, 6, 4, 2, False, [6, 2]),        # d_v != d_k, key padding only
    ]
    for n, (B, H, Sq, Skv, Dk, Dv, causal, kl) in enumerate(cases):
        q, k = _rand((B, H, Sq, Dk), 30 + n), _rand((B, H, Skv, Dk), 40 + n)
        v = _rand((B, H, Skv, Dv), 50 + n)
        scale = 1.0 / math.sqrt(Dk) * (1.0 + 0.25 * n)
        allowed = np.ones((B, 1, Sq, Skv), dtype=bool)
        ii = np.arange(Sq)[:, None]
        jj = np.arange(Skv)[None, :]
        if causal:
            allowed &= (jj <= ii + (Skv - Sq))[None, None]
        if kl is not None:
            allowed &= (jj[None] < np.array(kl)[:, None, None])[:, None]
        ref = _torch_sdpa_f64(q, k, v, allowed, scale)
        out = att(q, k, v, scale=scale, causal=causal,
                  kv_len=None if kl is None else np.array(kl, np.int32), query_padding=False)
        ok = allowed.any(-1)  # (B, 1, Sq)
        for b in range(B):
            for i in range(Sq):
                if ok[b, 0, i]:
                    np.testing.assert_allclose(out[b, :, i], ref[b, :, i], rtol=0, atol=1e-12)
                else:
                    assert np.all(out[b, :, i] == 0.0)


def pin_empty_rows_are_zero(att):
    """A row that sees no key, and a padded query row, output exact zeros (the
    library's rule for what the pages treat as an error, 'Attention from
    Scratch' (kube-dojo), Part 2 guard and Part 3 all-masked-row trap)."""
    q, k, v = _rand((2, 2, 5, 4), 60), _rand((2, 2, 5, 4), 61), _rand((2, 2, 5, 4), 62)
    out = att(q, k, v, causal=True, kv_len=np.array([0, 2], np.int32))
    assert np.all(out[0] == 0.0)
    assert np.all(out[1, :, 2:] == 0.0)
    assert np.any(out[1, :, :2] != 0.0)
    # decode-style: no query padding, L_b = 0 still gives zeros
    out = att(q[:, :, :1], k, v, kv_len=np.array([0, 5], np.int32), query_padding=False)
    assert np.all(out[0] == 0.0) and np.any(out[1] != 0.0)


def pin_decode_equals_last_causal_row(att):
    """Decoding the newest token against the cache equals the last row of
    causal attention over the whole prefix ('Attention from scratch'
    (open-llm-engineering), "Decode": the cache must not change the result)."""
    S, D = 11, 8
    q, k, v = _rand((2, 3, S, D), 70), _rand((2, 3, S, D), 71), _rand((2, 3, S, D), 72)
    full = att(q, k, v, causal=True)
    dec = att(q[:, :, S - 1:], k, v, causal=False)
    np.testing.assert_allclose(dec[:, :, 0], full[:, :, S - 1], rtol=0, atol=1e-13)
    # the query sees every cached key: same result with causal alignment on
    dec_c = att(q[:, :, S - 1:], k, v, causal=True)
    np.testing.assert_allclose(dec_c, dec, rtol=0, atol=0)


def pin_chunk_against_cache(att):
    """A chunk of the last T queries against all S keys equals the last T rows
    of full causal attention: positions are absolute ('Attention from scratch'
    (open-llm-engineering), "KV cache position drift")."""
    S, T, D = 10, 4, 6
    q, k, v = _rand((1, 2, S, D), 73), _rand((1, 2, S, D), 74), _rand((1, 2, S, D), 75)
    full = att(q, k, v, causal=True)
    part = att(q[:, :, S - T:], k, v, causal=True)
    np.testing.assert_allclose(part, full[:, :, S - T:], rtol=0, atol=1e-13)


def pin_key_padding_is_truncation(att):
    """Masking keys j >= L equals deleting them ('Attention from Scratch'
    (kube-dojo), Part 3 padding mask over key columns)."""
    S, D, L = 9, 5, 6
    q, k, v = _rand((1, 2, 3, D), 76), _rand((1, 2, S, D), 77), _rand((1, 2, S, D), 78)
    padded = att(q, k, v, kv_len=np.array([L], np.int32), query_padding=False)
    trunc = att(q, k[:, :, :L], v[:, :, :L])
    np.testing.assert_allclose(padded, trunc, rtol=0, atol=1e-13)


def pin_grouped_query_matches_library(att):
    """Grouped-query and multi-query attention: query head h uses key/value head
    h // (H // Hkv), which is what the pages' K.repeat_interleave(H // Hkv,
    dim=1) builds before ordinary attention ('Attention from First
    Principles', section 5 "The full multi-head computation"; 'Scaled
    dot-product attention with masking', "Grouped-query attention (GQA)").
    Checked against PyTorch's scaled_dot_product_attention in float64 on the
    explicitly repeated keys and values."""
    cases = [  # (B, H, Hkv, Sq, Skv, D, causal, kv_len)
        (2, 6, 2, 5, 5, 8, True, None),
        (2, 4, 1, 1, 9, 6, False, [9, 4]),        # multi-query decode with key padding
        (1, 6, 3, 4, 7, 4, True, None),           # chunk of queries, three groups of two
        (2, 8, 4, 6, 6, 5, True, [6, 3]),
    ]
    for n, (B, H, Hkv, Sq, Skv, D, causal, kl) in enumerate(cases):
        q = _rand((B, H, Sq, D), 80 + n)
        k, v = _rand((B, Hkv, Skv, D), 90 + n), _rand((B, Hkv, Skv, D), 100 + n)
        G = H // Hkv
        kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)  # repeat_interleave on dim 1
        allowed = np.ones((B, 1, Sq, Skv), dtype=bool)
        ii, jj = np.arange(Sq)[:, None], np.arange(Skv)[None, :]
        if causal:
            allowed &= (jj <= ii + (Skv - Sq))[None, None]
        if kl is not None:
            allowed &= (jj[None] < np.array(kl)[:, None, None])[:, None]
        scale = 1.0 / math.sqrt(D)
        ref = _torch_sdpa_f64(q, kr, vr, allowed, scale)
        out = att(q, k, v, scale=scale, causal=causal,
                  kv_len=None if kl is None else np.array(kl, np.int32), query_padding=False)
        ok = allowed.any(-1)
        for b in range(B):
            for i in range(Sq):
                if ok[b, 0, i]:
                    np.testing.assert_allclose(out[b, :, i], ref[b, :, i], rtol=0, atol=1e-12)


def pin_cache_chunk_is_tail_of_full_causal(att):
    """A chunk of the last Sq tokens of a sequence, run against its KV cache of
    L_b positions, equals rows L_b - Sq .. L_b - 1 of causal self-attention
    over those L_b tokens ('Scaled dot-product attention with masking', the
    cache append before causal attention; 'Attention from scratch'
    (open-llm-engineering), "KV cache position drift": positions are
    absolute).  Per-sequence lengths shorter than the cache, grouped heads."""
    B, H, Hkv, Skv, Sq, D = 3, 4, 2, 9, 3, 5
    lens = [9, 6, 3]
    qfull = _rand((B, H, Skv, D), 110)
    k, v = _rand((B, Hkv, Skv, D), 111), _rand((B, Hkv, Skv, D), 112)
    q = np.stack([qfull[b, :, L - Sq:L] for b, L in enumerate(lens)])
    out = att(q, k, v, causal=True, cache_len=np.array(lens, np.int32))
    for b, L in enumerate(lens):
        full = att(qfull[b:b + 1, :, :L], k[b:b + 1, :, :L], v[b:b + 1, :, :L], causal=True)
        np.testing.assert_allclose(out[b], full[0, :, L - Sq:L], rtol=0, atol=1e-13)


def pin_lse_is_log_sum_exp(att):
    """The log-sum-exp output is log(sum_j exp(scale * q_i.k_j)) over exactly
    the visible keys, computed here by brute force with numpy's logaddexp;
    -inf for a query whose position precedes the sequence (cache_len < Sq)."""
    B, H, Hkv, Skv, Sq, D = 2, 4, 1, 7, 4, 3
    lens = [7, 2]
    q, k = _rand((B, H, Sq, D), 120), _rand((B, Hkv, Skv, D), 121)
    v = _rand((B, Hkv, Skv, D), 122)
    scale = 0.7
    _, lse = att(q, k, v, scale=scale, causal=True, cache_len=np.array(lens, np.int32), need_lse=True)
    G = H // Hkv
    for b, L in enumerate(lens):
        for h in range(H):
            for i in range(Sq):
                vis = [j for j in range(L) if j <= L - Sq + i]
                s = [scale * float(np.dot(q[b, h, i].astype(np.float64), k[b, h // G, j].astype(np.float64)))
                     for j in vis]
                want = np.logaddexp.reduce(s) if s else -np.inf
                if s:
                    assert abs(lse[b, h, i] - want) <= 1e-12, (b, h, i, lse[b, h, i], want)
                else:
                    assert lse[b, h, i] == -np.inf


def pin_lengths_outside_range_are_clamped(att):
    """Length entries outside [0, Skv] act as the nearest end of the range.  A
    length above the capacity makes every key valid, so prefill equals the
    unpadded call and a chunk against its cache equals the last Sq rows of full
    causal attention over all Skv keys, checked against PyTorch's float64
    scaled_dot_product_attention ('Attention from scratch'
    (open-llm-engineering), "KV cache position drift": positions are absolute).
    A negative length leaves no visible key, so the row is zero (the library's
    rule for a row the pages treat as an error)."""
    B, H, S, D, Sq = 2, 2, 7, 4, 3
    q, k, v = _rand((B, H, S, D), 130), _rand((B, H, S, D), 131), _rand((B, H, S, D), 132)
    scale = 1.0 / math.sqrt(D)
    ii, jj = np.arange(S)[:, None], np.arange(S)[None, :]
    ref = _torch_sdpa_f64(q, k, v, np.broadcast_to((jj <= ii)[None, None], (B, 1, S, S)), scale)
    out = att(q, k, v, scale=scale, causal=True, kv_len=np.array([S + 5, -3], np.int32))
    np.testing.assert_allclose(out[0], ref[0], rtol=0, atol=1e-12)
    assert np.all(out[1] == 0.0)
    qc = np.ascontiguousarray(q[:, :, S - Sq:])
    out_c = att(qc, k, v, scale=scale, causal=True, cache_len=np.array([S + 9, -2], np.int32))
    np.testing.assert_allclose(out_c[0], ref[0, :, S - Sq:], rtol=0, atol=1e-12)
    assert np.all(out_c[1] == 0.0)
    dec = att(q[:, :, S - 1:], k, v, scale=scale, causal=False,
              kv_len=np.array([S + 1, -7], np.int32), query_padding=False)
    np.testing.assert_allclose(dec[0, :, 0], ref[0, :, S - 1], rtol=0, atol=1e-12)
    assert np.all(dec[1] == 0.0)


ALL_PINS = [
    pin_tiny_example_causal,
    pin_kube_dojo_example,
    pin_rows_are_distributions,
    pin_causal_first_row_is_v0,
    pin_zero_qk_prefix_mean,
    pin_uniform_scores_with_padding,
    pin_permutation_equivariance,
    pin_shift_invariance_large,
    pin_large_scale_is_hard_lookup,
    pin_matches_library_sdpa,
    pin_empty_rows_are_zero,
    pin_decode_equals_last_causal_row,
    pin_chunk_against_cache,
    pin_key_padding_is_truncation,
    pin_grouped_query_matches_library,
    pin_cache_chunk_is_tail_of_full_causal,
    pin_lse_is_log_sum_exp,
    pin_lengths_outside_range_are_clamped,
]
