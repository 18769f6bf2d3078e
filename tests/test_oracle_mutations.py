"""The oracle's pins catch plausible mistakes: plant one in the oracle (on the CPU) and
check that a pin fails.  Mutations: wrong power, wrong support width, a dropped
argmax correction in the backward, swapped query/key operands, and in the attn_mask
handling an ignored, a transposed, or an OR-ed (instead of AND-ed) mask."""
import numpy as np
import pytest

import oracle
from oracle import ra_oracle

LOGITS = np.array([[2.0, 1.0, 0.0], [5.0, 1.0, -10.0]])
EXACT_P_ROW0 = [300283484326400961 / 450821375485925827, 110324037687890625 / 450821375485925827,
                40213853471634241 / 450821375485925827]


def _worked_example_holds():
    p, *_ = ra_oracle.ra_softmax(LOGITS)
    return np.allclose(p[0], EXACT_P_ROW0, rtol=2e-15, atol=0)


def _artanh_identity_holds():
    delta = np.linspace(0.0, 15.9, 101)
    return np.allclose(ra_oracle.ra_phi(delta), np.exp(-16.0 * np.arctanh(delta / 16.0)), rtol=1e-12, atol=0)


def test_pins_hold_on_the_unmutated_oracle():
    assert _worked_example_holds() and _artanh_identity_holds()


@pytest.mark.parametrize("attr,value", [("POWER", 7), ("POWER", 9), ("SUPPORT", 8.0), ("SUPPORT", 17.0)])
def test_constant_mutations_are_caught(monkeypatch, attr, value):
    monkeypatch.setattr(ra_oracle, attr, value)
    assert not (_worked_example_holds() and _artanh_identity_holds())


def test_dropped_argmax_correction_is_caught():
    rng = np.random.default_rng(0)
    x = rng.normal(0, 4.0, size=(1, 5))
    dy = rng.normal(size=x.shape)
    good = ra_oracle.ra_softmax_bwd(x, dy)
    bad = good.copy()
    bad[0, np.argmax(x)] = 0.0          # the mistake: x_max treated as a constant
    h = 1e-6
    fd = np.zeros_like(x)
    for j in range(x.shape[1]):
        xp, xm = x.copy(), x.copy()
        xp[0, j] += h
        xm[0, j] -= h
        fd[0, j] = ((ra_oracle.ra_softmax(xp)[0] - ra_oracle.ra_softmax(xm)[0]) * dy).sum() / (2 * h)
    assert np.allclose(good, fd, rtol=1e-6, atol=1e-8)
    assert not np.allclose(bad, fd, rtol=1e-6, atol=1e-8)
    assert abs(bad.sum()) > 1e-6        # and the row-sum pin fails too


def test_swapped_operands_are_caught():
    # with query and key roles swapped the causal-row-0 pin (O_0 = V_0) breaks
    rng = np.random.default_rng(1)
    q = rng.normal(size=(8, 4))
    k = rng.normal(size=(8, 4))
    v = rng.normal(size=(8, 4))
    O, *_ = oracle.ra_attention_head_fwd(q, k, v, 0.7, True)
    Ob, *_ = oracle.ra_attention_head_fwd(k, q, v, 0.7, True)
    assert np.array_equal(O[0], v[0])
    # swapped: row 0 still sees only key 0, but the later rows change
    assert not np.allclose(O[1:], Ob[1:])


def _mask_pins_hold():
    """The attn_mask pins of tests/test_oracle_mask.py in compact form: a key-padding mask
    equals deleting the keys, a row with no allowed key gives zeros, a lower-triangular mask
    equals causal, and an all-True mask leaves causal unchanged."""
    rng = np.random.default_rng(6)
    q, k, v = (rng.normal(size=(1, 1, 6, 4)) for _ in range(3))
    keep = np.array([0, 2, 3, 5])
    mask = np.zeros((6, 6), dtype=bool)
    mask[:, keep] = True
    O, *_ = oracle.ra_attention_fwd(q, k, v, mask=mask)
    O2, *_ = oracle.ra_attention_fwd(q, k[:, :, keep], v[:, :, keep])
    pad_ok = O.shape == O2.shape and np.allclose(O, O2, rtol=0, atol=1e-14)
    empty = mask.copy()
    empty[2] = False
    Oe, _, se, ae = oracle.ra_attention_fwd(q, k, v, mask=empty)
    empty_ok = bool(np.all(Oe[0, 0, 2] == 0) and se[0, 0, 2] == 0 and ae[0, 0, 2] == -1)
    tri = np.tril(np.ones((6, 6), dtype=bool))
    causal = oracle.ra_attention_fwd(q, k, v, causal=True)
    tri_ok = all(np.array_equal(a, b) for a, b in zip(oracle.ra_attention_fwd(q, k, v, mask=tri), causal))
    ones_ok = all(np.array_equal(a, b) for a, b in
                  zip(oracle.ra_attention_fwd(q, k, v, causal=True, mask=np.ones((6, 6), dtype=bool)), causal))
    return pad_ok and empty_ok and tri_ok and ones_ok


def test_mask_pins_hold_on_the_unmutated_oracle():
    assert _mask_pins_hold()


_REAL_ALLOWED = ra_oracle._allowed


def _ignore_mask(n_q, n_k, causal, mask):
    return _REAL_ALLOWED(n_q, n_k, causal, None)


def _transposed_mask(n_q, n_k, causal, mask):
    return _REAL_ALLOWED(n_q, n_k, causal, None if mask is None else np.asarray(mask).T)


def _mask_or_causal(n_q, n_k, causal, mask):
    if mask is None or not causal:
        return _REAL_ALLOWED(n_q, n_k, causal, mask)
    return _REAL_ALLOWED(n_q, n_k, True, None) | np.asarray(mask, dtype=bool)


@pytest.mark.parametrize("mutant", [_ignore_mask, _transposed_mask, _mask_or_causal])
def test_mask_mutations_are_caught(monkeypatch, mutant):
    monkeypatch.setattr(ra_oracle, "_allowed", mutant)
    assert not _mask_pins_hold()
