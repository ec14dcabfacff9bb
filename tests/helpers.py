"""Comparison helpers for GPU-vs-oracle parity tests."""
import numpy as np
import torch

# Tolerances (absolute, against the fp64 oracle on the same inputs):
BF16_MAX, BF16_MEAN = 2e-2, 2e-3   # bf16 inputs, fp32 accumulation, N(0, 1) data
F32_MAX = 1e-4                     # fp32 inputs


def to_f64(t):
    return t.detach().float().cpu().double().numpy()


def assert_close(got, ref, dtype, what=""):
    got = to_f64(got) if isinstance(got, torch.Tensor) else np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - ref)
    mx = float(err.max()) if err.size else 0.0
    mean = float(err.mean()) if err.size else 0.0
    if dtype == torch.float32:
        assert mx <= F32_MAX, f"{what}: max abs err {mx:.3e} > {F32_MAX}"
    else:
        assert mx <= BF16_MAX, f"{what}: max abs err {mx:.3e} > {BF16_MAX}"
        assert mean <= BF16_MEAN, f"{what}: mean abs err {mean:.3e} > {BF16_MEAN}"
    return mx, mean
