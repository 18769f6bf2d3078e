"""Shared helpers of the GPU parity tests: tolerances and comparisons against the oracle."""
import numpy as np
import torch

# bf16 inputs (evaluated on the same bf16-rounded values): max-abs and mean-abs bounds.
BF16_MAX_ABS = 1e-2
BF16_MEAN_ABS = 1e-3
# fp32 path: max-abs bound.
FP32_MAX_ABS = 2e-5


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close_bf16(got, want, what, max_abs=BF16_MAX_ABS, mean_abs=BF16_MEAN_ABS):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    err = np.abs(got - want)
    mx, mean = float(err.max()) if err.size else 0.0, float(err.mean()) if err.size else 0.0
    assert mx <= max_abs and mean <= mean_abs, f"{what}: max-abs {mx:.3e} (<= {max_abs}), mean-abs {mean:.3e} (<= {mean_abs})"
    return mx, mean


def assert_close_fp32(got, want, what, max_abs=FP32_MAX_ABS):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite values"
    mx = float(np.abs(got - want).max()) if got.size else 0.0
    assert mx <= max_abs, f"{what}: max-abs {mx:.3e} (<= {max_abs})"
    return mx
