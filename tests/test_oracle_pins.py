"""Pins of the float64 oracle's forward against what the pages and the mathematics fix.

Each test pins the oracle to something other than itself: hand-derived exact
rationals for the page's worked input, a different closed form of phi, the
limit in which ra_softmax must agree with the standard softmax (a library
routine), special cases with an exact answer, invariants the page states, and
a separately written tiled implementation.  No GPU needed.
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

import oracle


def _read_golden(golden_dir):
    rows = {}
    attn = None
    with open(os.path.join(golden_dir, "ra_softmax_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0] == "row":
                rows[(int(parts[1]), parts[2])] = [Fraction(t) for t in parts[3:]]
            elif parts[0] == "attn":
                attn = [Fraction(t) for t in parts[2:]]
    return rows, attn


LOGITS = np.array([[2.0, 1.0, 0.0], [5.0, 1.0, -10.0]])  # the page's worked input


def test_worked_example_probabilities(golden_dir):
    rows, _ = _read_golden(golden_dir)
    p, m, s, a = oracle.ra_softmax(LOGITS)
    for r in range(2):
        exact_p = np.array([float(t) for t in rows[(r, "p")]])
        np.testing.assert_allclose(p[r], exact_p, rtol=2e-15, atol=0)
        assert s[r] == pytest.approx(float(rows[(r, "sum")][0]), rel=2e-15)
    assert list(a) == [0, 0]
    assert list(m) == [2.0, 5.0]


def test_worked_example_phi(golden_dir):
    rows, _ = _read_golden(golden_dir)
    for r in range(2):
        delta = LOGITS[r].max() - LOGITS[r]
        np.testing.assert_allclose(oracle.ra_phi(delta), [float(t) for t in rows[(r, "phi")]],
                                   rtol=2e-15, atol=0)


def test_hand_derived_attention_case(golden_dir):
    _, attn = _read_golden(golden_dir)
    q = np.array([[2.0, 0.0]])
    k = np.array([[1.0, 0.0], [0.0, 0.0], [-7.0, 0.0]])
    v = np.array([[1.0, 0.0], [0.0, 1.0], [5.0, 5.0]])
    O, m, s, a = oracle.ra_attention_head_fwd(q, k, v, 1.0, False)
    np.testing.assert_allclose(O[0], [float(t) for t in attn], rtol=2e-15, atol=0)
    assert a[0] == 0 and m[0] == 2.0


def test_compact_support_is_exactly_zero():
    # the page: phi is set exactly to 0.0 for Delta >= 16
    big = np.array([16.0, np.nextafter(16.0, 17.0), 17.0, 100.0, 1e30])
    assert np.all(oracle.ra_phi(big) == 0.0)
    inside = np.array([np.nextafter(16.0, 0.0), 15.999, 15.0])
    assert np.all(oracle.ra_phi(inside) > 0.0)
    x = np.array([[20.0, 4.0, 4.0001, 0.0, -50.0]])
    p, *_ = oracle.ra_softmax(x)
    assert p[0, 1] == 0.0 and p[0, 3] == 0.0 and p[0, 4] == 0.0 and p[0, 2] > 0.0


def test_phi_equals_exp_of_minus_16_artanh():
    # (1-u)/(1+u) = exp(-2 artanh u), so phi = exp(-16 artanh(Delta/16)): a different
    # closed form that fixes the support width (16) and the power (8) at once.
    delta = np.linspace(0.0, 15.9, 2001)
    want = np.exp(-16.0 * np.arctanh(delta / 16.0))
    np.testing.assert_allclose(oracle.ra_phi(delta), want, rtol=1e-12, atol=0)


def test_cayley_pade_small_shift_series():
    # ln phi = -16 artanh(u) = -Delta - Delta^3/768 - Delta^5/327680 - ...: phi is the
    # Cayley/Pade form of exp(-Delta) with a cubic leading error.
    delta = np.linspace(1e-2, 2.0, 200)
    resid = np.log(oracle.ra_phi(delta)) + delta + delta ** 3 / 768.0
    np.testing.assert_allclose(resid, -delta ** 5 / 327680.0, rtol=0.02, atol=1e-15)


@pytest.mark.parametrize("shape", [(1, 1), (3, 7), (5, 64), (2, 1000)])
def test_softmax_invariants(shape):
    rng = np.random.default_rng(7)
    x = rng.normal(0.0, 6.0, size=shape)
    p, m, s, a = oracle.ra_softmax(x)
    np.testing.assert_allclose(p.sum(-1), 1.0, rtol=0, atol=1e-14 * shape[-1])
    assert np.all(p >= 0) and np.all(p <= 1)
    assert np.all(s >= 1.0)                                      # sum(phi) >= 1
    np.testing.assert_array_equal(a, np.argmax(x, -1))
    np.testing.assert_allclose(p[np.arange(shape[0]), a] * s, 1.0, rtol=1e-15)  # phi_max = 1
    dead = (m[:, None] - x) >= 16.0
    assert np.all(p[dead] == 0.0)
    assert np.all(p[~dead] > 0.0)


def test_shift_invariance_exact():
    rng = np.random.default_rng(3)
    x = rng.integers(-200, 200, size=(4, 33)) / 8.0   # dyadic, so x + c is exact
    p1, *_ = oracle.ra_softmax(x)
    p2, *_ = oracle.ra_softmax(x + 3.25)
    np.testing.assert_array_equal(p1, p2)


def test_not_scale_invariant():
    x = np.array([[1.0, 0.5, -0.25, 3.0]])
    p1, *_ = oracle.ra_softmax(x)
    p2, *_ = oracle.ra_softmax(2.0 * x)
    assert np.max(np.abs(p1 - p2)) > 1e-2


def test_small_spread_agrees_with_standard_softmax():
    # For a row spread of at most Delta_max, phi_j = exp(-Delta_j) exp(-eps_j) with
    # 0 <= eps_j <= eps = -ln phi(Delta_max) - Delta_max, so |p_ra - p_std| <= (e^eps - 1) p_std.
    rng = np.random.default_rng(11)
    x = rng.uniform(-0.25, 0.25, size=(16, 40))
    p, *_ = oracle.ra_softmax(x)
    ref = scipy.special.softmax(x, axis=-1)
    dmax = (x.max(-1, keepdims=True) - x).max()
    eps = -np.log(oracle.ra_phi(dmax)) - dmax
    assert np.all(np.abs(p - ref) <= math.expm1(eps) * ref + 1e-16)
    assert np.max(np.abs(p - ref)) > 0  # and it is not the standard softmax


def test_attention_matches_sdpa_for_small_scores():
    # Same bound at the attention level: with every score spread below Delta_max the
    # rational weights are within a factor exp(+-eps) of softmax weights, so
    # |O_ra - O_sdpa| <= 2 (e^eps - 1) max|V| per row.  A transposed or mis-scaled
    # operand moves O far beyond that bound.
    rng = np.random.default_rng(5)
    B, H, N, D = 1, 2, 24, 8
    q = rng.normal(size=(B, H, N, D))
    k = rng.normal(size=(B, H, N, D))
    v = rng.normal(size=(B, H, N, D))
    scale = 0.05
    for causal in (False, True):
        O, *_ = oracle.ra_attention_fwd(q, k, v, scale=scale, causal=causal)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v),
            is_causal=causal, scale=scale).numpy()
        S = scale * np.einsum("bhid,bhjd->bhij", q, k)
        dmax = S.max() - S.min()
        eps = -np.log(oracle.ra_phi(dmax)) - dmax
        bound = 2 * math.expm1(eps) * np.abs(v).max()
        assert np.max(np.abs(O - ref)) <= bound
        # the effect of the scores themselves is far larger than the bound
        uniform = v.mean(axis=2, keepdims=True) if not causal else \
            np.cumsum(v, axis=2) / np.arange(1, N + 1)[None, None, :, None]
        assert np.max(np.abs(ref - uniform)) > 5 * bound


def test_single_key_gives_O_equal_V():
    rng = np.random.default_rng(0)
    q = rng.normal(size=(2, 3, 9, 16))
    k = rng.normal(size=(2, 3, 1, 16))
    v = rng.normal(size=(2, 3, 1, 16))
    O, m, s, a = oracle.ra_attention_fwd(q, k, v, scale=0.3, causal=False)
    np.testing.assert_array_equal(O, np.broadcast_to(v, O.shape))
    assert np.all(s == 1.0) and np.all(a == 0)


def test_causal_first_row_is_V0_and_equal_scores_average():
    rng = np.random.default_rng(1)
    q = rng.normal(size=(1, 2, 10, 8))
    k = rng.normal(size=(1, 2, 10, 8))
    v = rng.normal(size=(1, 2, 10, 8))
    O, *_ = oracle.ra_attention_fwd(q, k, v, scale=0.7, causal=True)
    np.testing.assert_array_equal(O[:, :, 0], v[:, :, 0])
    # all scores equal (q = 0): uniform weights over the allowed keys
    O0, *_ = oracle.ra_attention_fwd(np.zeros_like(q), k, v, scale=0.7, causal=True)
    want = np.cumsum(v, axis=2) / np.arange(1, 11)[None, None, :, None]
    np.testing.assert_allclose(O0, want, rtol=1e-14, atol=1e-15)


def test_scores_beyond_support_give_one_hot():
    # every non-maximal score at least 16 below the max: weights are exactly one-hot
    D = 4
    k = np.zeros((6, D))
    k[:, 0] = np.array([0.0, 1.0, 2.0, 3.0, 4.0, 5.0]) * 20.0
    q = np.zeros((3, D))
    q[:, 0] = [1.0, -1.0, 2.0]
    v = np.arange(6 * D, dtype=float).reshape(6, D)
    O, m, s, a = oracle.ra_attention_head_fwd(q, k, v, 1.0, False)
    assert list(a) == [5, 0, 5]
    np.testing.assert_array_equal(O, v[a])
    assert np.all(s == 1.0)


def test_causality_probe():
    # position t must not see t+1: changing keys/values after t leaves O[:t+1] bit-identical
    rng = np.random.default_rng(2)
    q = rng.normal(size=(1, 1, 12, 8))
    k = rng.normal(size=(1, 1, 12, 8))
    v = rng.normal(size=(1, 1, 12, 8))
    O1, *_ = oracle.ra_attention_fwd(q, k, v, scale=0.5, causal=True)
    t = 6
    k2, v2 = k.copy(), v.copy()
    k2[:, :, t + 1:] += 5.0
    v2[:, :, t + 1:] -= 3.0
    O2, *_ = oracle.ra_attention_fwd(q, k2, v2, scale=0.5, causal=True)
    np.testing.assert_array_equal(O1[:, :, :t + 1], O2[:, :, :t + 1])
    assert np.max(np.abs(O1[:, :, t + 1:] - O2[:, :, t + 1:])) > 0.1


@pytest.mark.parametrize("n_q,n_k", [(1, 1), (2, 5), (5, 5), (7, 9), (17, 17), (9, 4)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("tiles", [(4, 4), (3, 5)])
def test_tiled_equals_materialised(n_q, n_k, causal, tiles):
    rng = np.random.default_rng(n_q * 100 + n_k)
    D = 6
    q = rng.normal(0, 2.5, size=(n_q, D))
    k = rng.normal(0, 2.5, size=(n_k, D))
    v = rng.normal(size=(n_k, D))
    scale = 0.6
    O, m, s, a = oracle.ra_attention_head_fwd(q, k, v, scale, causal)
    Ot, mt, st, at = oracle.ra_attention_tiled_head(q, k, v, scale, causal, *tiles)
    np.testing.assert_allclose(Ot, O, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(mt, m, rtol=1e-15, atol=0)
    np.testing.assert_allclose(st, s, rtol=1e-13, atol=0)
    np.testing.assert_array_equal(at, a)


def test_sampled_rows_equal_full_head():
    rng = np.random.default_rng(9)
    q = rng.normal(size=(40, 8))
    k = rng.normal(size=(40, 8))
    v = rng.normal(size=(40, 8))
    rows = np.array([0, 3, 17, 39])
    for causal in (False, True):
        O, m, s, a = oracle.ra_attention_head_fwd(q, k, v, 0.8, causal)
        Or, mr, sr, ar = oracle.ra_attention_rows_fwd(q, k, v, rows, 0.8, causal)
        np.testing.assert_allclose(Or, O[rows], rtol=1e-13, atol=1e-14)
        np.testing.assert_array_equal(ar, a[rows])


def test_default_scale_is_inverse_sqrt_d():
    assert oracle.default_scale(64, None) == 0.125
    assert oracle.default_scale(64, 0.0) == 0.125
    assert oracle.default_scale(64, 0.5) == 0.5
