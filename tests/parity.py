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


# ---------------------------------------------------------------------------------------
# Argmax agreement.  The reading for ties (the pages are silent) is the lowest key index
# among exact maxima, in the oracle and the kernels alike.  The kernels' scores are fp32,
# the oracle's float64, so two keys whose float64 scores differ by less than the fp32
# score error may legitimately swap.  That error is bounded per row: each score is a sum
# of D products (exact in fp32 for bf16 operands, one rounding each for fp32 operands)
# accumulated with at most D + 2 roundings of relative size 2^-23 (truncation allowed),
# times the scale, so |s_fp32 - s_64| <= scale (D + 2) 2^-23 sum_d |q_d k_d|.  A row may
# differ from the oracle's argmax only where the float64 gap between the two keys is at
# most twice that bound.  Every check records how many rows it compared, how many were
# near ties by that bound, and how many actually differed; the counts are printed at the
# end of the run (tests/conftest.py).
# ---------------------------------------------------------------------------------------
ARGMAX_LOG = []


def score_error_bound(q, k, scale):
    """Per query row: the largest fp32 score error over the row's keys (float64 q [N_Q, D], k [N_K, D])."""
    D = q.shape[-1]
    return abs(scale) * (D + 2) * 2.0 ** -23 * (np.abs(q) @ np.abs(k).T).max(axis=1)


def check_argmax(S, a_gpu, err, what, m_gpu=None):
    """S: float64 scaled scores [rows, N_K] with -inf at excluded entries; a_gpu: the GPU's
    argmax per row (-1 for a row with no allowed key); err: score_error_bound per row;
    m_gpu: optionally the GPU's row maximum (scaled), which must lie within err of the
    float64 maximum.  Rows whose GPU argmax is not the lowest float64 maximum must be near
    ties: the chosen key's float64 score at most 2 err below the maximum.  Returns the
    number of rows that differed."""
    S = np.asarray(S, dtype=np.float64)
    a_gpu = np.asarray(a_gpu, dtype=np.int64)
    has = np.isfinite(S).any(axis=1)
    m = np.where(has, S.max(axis=1), -np.inf)
    a64 = np.where(has, np.argmax(S == m[:, None], axis=1), -1)
    assert np.array_equal(a_gpu[~has], a64[~has]), f"{what}: rows with no allowed key must give argmax -1"
    if m_gpu is not None:
        mg = np.asarray(m_gpu, dtype=np.float64)[has]
        assert np.all(np.abs(mg - m[has]) <= err[has] + 1e-30), \
            f"{what}: row max beyond the fp32 score-error bound by {np.max(np.abs(mg - m[has]) - err[has]):.3e}"
    srt = np.sort(S, axis=1)
    with np.errstate(invalid="ignore"):
        gap = srt[:, -1] - srt[:, -2] if S.shape[1] > 1 else np.full(S.shape[0], np.inf)
    near = int(np.count_nonzero(has & (gap <= 2 * err)))
    diff = np.nonzero(a_gpu != a64)[0]
    for i in diff:
        assert has[i] and 0 <= a_gpu[i] < S.shape[1], f"{what}: row {i}: argmax {a_gpu[i]} vs {a64[i]}"
        assert S[i, a_gpu[i]] >= m[i] - 2 * err[i], \
            f"{what}: row {i}: argmax {a_gpu[i]} is {m[i] - S[i, a_gpu[i]]:.3e} below the max, beyond 2 x {err[i]:.3e}"
    ARGMAX_LOG.append((what, int(S.shape[0]), near, int(len(diff))))
    return int(len(diff))
