"""Pins for the attention oracle's boolean attn_mask (True = the query may attend to the key)."""
import numpy as np
import pytest

import oracle


def _qkv(rng, B, H, nq, nk, D):
    return rng.normal(size=(B, H, nq, D)), rng.normal(size=(B, H, nk, D)), rng.normal(size=(B, H, nk, D))


def test_all_true_mask_is_no_mask():
    rng = np.random.default_rng(0)
    q, k, v = _qkv(rng, 1, 2, 7, 9, 8)
    want = oracle.ra_attention_fwd(q, k, v)
    got = oracle.ra_attention_fwd(q, k, v, mask=np.ones((7, 9), dtype=bool))
    for g, w in zip(got, want):
        np.testing.assert_array_equal(g, w)


def test_lower_triangular_mask_is_causal():
    rng = np.random.default_rng(1)
    q, k, v = _qkv(rng, 2, 1, 6, 6, 4)
    tri = np.tril(np.ones((6, 6), dtype=bool))
    for g, w in zip(oracle.ra_attention_fwd(q, k, v, mask=tri), oracle.ra_attention_fwd(q, k, v, causal=True)):
        np.testing.assert_array_equal(g, w)
    do = rng.normal(size=q.shape)
    for g, w in zip(oracle.ra_attention_bwd(q, k, v, do, mask=tri), oracle.ra_attention_bwd(q, k, v, do, causal=True)):
        np.testing.assert_array_equal(g, w)


def test_fully_masked_row_gives_zero_output_and_gradients():
    rng = np.random.default_rng(2)
    q, k, v = _qkv(rng, 1, 1, 5, 6, 4)
    mask = rng.random((5, 6)) < 0.6
    mask[2] = False
    mask[:, 0] |= np.arange(5) != 2   # every other row keeps at least one key
    O, m, s, a = oracle.ra_attention_fwd(q, k, v, mask=mask)
    assert np.all(O[0, 0, 2] == 0) and s[0, 0, 2] == 0 and a[0, 0, 2] == -1
    # the other rows are unaffected by row 2 (rows are independent)
    keep = [0, 1, 3, 4]
    O2, *_ = oracle.ra_attention_fwd(q[:, :, keep], k, v, mask=mask[keep])
    np.testing.assert_array_equal(O[:, :, keep], O2)
    do = rng.normal(size=q.shape)
    dq, dk, dv = oracle.ra_attention_bwd(q, k, v, do, mask=mask)
    assert np.all(dq[0, 0, 2] == 0)
    # row 2 contributes nothing to dk, dv: same gradients with its upstream gradient zeroed
    do0 = do.copy()
    do0[0, 0, 2] = 0
    for g, w in zip((dk, dv), oracle.ra_attention_bwd(q, k, v, do0, mask=mask)[1:]):
        np.testing.assert_allclose(g, w, rtol=0, atol=1e-14)


def test_mask_broadcasts_over_batch_and_heads():
    rng = np.random.default_rng(3)
    q, k, v = _qkv(rng, 2, 3, 4, 5, 4)
    mask_h = rng.random((3, 4, 5)) < 0.7
    mask_h[..., 0] = True
    O, *_ = oracle.ra_attention_fwd(q, k, v, mask=mask_h[None])
    for b in range(2):
        for h in range(3):
            Oh, *_ = oracle.ra_attention_head_fwd(q[b, h], k[b, h], v[b, h], 0.5, False, mask=mask_h[h])
            np.testing.assert_array_equal(O[b, h], Oh)


@pytest.mark.parametrize("causal", [False, True])
def test_masked_backward_matches_finite_differences(causal):
    rng = np.random.default_rng(4 + int(causal))
    q, k, v = _qkv(rng, 1, 1, 5, 7, 3)
    q, k = q * 2.0, k * 2.0
    mask = rng.random((5, 7)) < 0.6
    mask[:, 0] = True
    do = rng.normal(size=q.shape)
    grads = oracle.ra_attention_bwd(q, k, v, do, causal=causal, mask=mask)

    def f(a, b, c):
        return float((oracle.ra_attention_fwd(a, b, c, causal=causal, mask=mask)[0] * do).sum())

    eps = 1e-6
    args = [q, k, v]
    for i, g in enumerate(grads):
        num = np.zeros_like(args[i])
        it = np.nditer(args[i], flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            p, mnus = [x.copy() for x in args], [x.copy() for x in args]
            p[i][idx] += eps
            mnus[i][idx] -= eps
            num[idx] = (f(*p) - f(*mnus)) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=1e-5, atol=1e-7, err_msg=f"argument {i}")


def test_key_padding_mask_equals_deleting_the_keys():
    """A mask that removes the same keys from every row is the unmasked attention over the
    remaining keys: same output; zero dk, dv for the removed keys and the unmasked
    gradients for the others."""
    rng = np.random.default_rng(6)
    q, k, v = _qkv(rng, 1, 2, 6, 9, 4)
    keep = np.array([0, 2, 3, 5, 8])
    mask = np.zeros((6, 9), dtype=bool)
    mask[:, keep] = True
    O, m, s, _ = oracle.ra_attention_fwd(q, k, v, mask=mask)
    O2, m2, s2, _ = oracle.ra_attention_fwd(q, k[:, :, keep], v[:, :, keep])
    np.testing.assert_allclose(O, O2, rtol=0, atol=1e-14)
    np.testing.assert_array_equal(m, m2)
    do = rng.normal(size=q.shape)
    dq, dk, dv = oracle.ra_attention_bwd(q, k, v, do, mask=mask)
    dq2, dk2, dv2 = oracle.ra_attention_bwd(q, k[:, :, keep], v[:, :, keep], do)
    np.testing.assert_allclose(dq, dq2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dk[:, :, keep], dk2, rtol=0, atol=1e-13)
    np.testing.assert_allclose(dv[:, :, keep], dv2, rtol=0, atol=1e-13)
    gone = np.setdiff1d(np.arange(9), keep)
    assert np.all(dk[:, :, gone] == 0) and np.all(dv[:, :, gone] == 0)
