"""Pins of the float64 oracle's backward.

The page gives only the closed form d phi/du = -16 phi/(1-u^2) (section 3,
ra_softmax, "Closed-Form Backward Pass"); the rest of the backward is the
chain rule, including the path through x_max.  It is pinned by
  * central finite differences of the oracle's own FORWARD (a different
    computation from the closed-form backward), on tiny inputs whose top-2
    score gap is wide enough that the argmax does not move under the probe;
  * torch float64 autograd of an independently written forward (a library
    routine differentiating a separate formula);
  * row sums of the score gradient being zero (shift invariance of ra_softmax).
"""
import numpy as np
import pytest
import torch

import oracle


def _fd_grad(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        idx = it.multi_index
        xp = x.copy()
        xm = x.copy()
        xp[idx] += h
        xm[idx] -= h
        g[idx] = (f(xp) - f(xm)) / (2 * h)
    return g


def _wide_gap_rows(rng, shape, sigma):
    # rejection-sample rows whose top-2 gap exceeds 1e-2 (so FD never crosses an argmax switch)
    while True:
        x = rng.normal(0.0, sigma, size=shape)
        srt = np.sort(x, axis=-1)
        if shape[-1] == 1 or np.all(srt[..., -1] - srt[..., -2] > 1e-2):
            return x


@pytest.mark.parametrize("cols", [1, 2, 3, 5, 9])
def test_softmax_bwd_matches_finite_differences(cols):
    rng = np.random.default_rng(cols)
    x = _wide_gap_rows(rng, (3, cols), 5.0)
    dy = rng.normal(size=x.shape)
    dx = oracle.ra_softmax_bwd(x, dy)
    fd = _fd_grad(lambda z: float((oracle.ra_softmax(z)[0] * dy).sum()), x)
    np.testing.assert_allclose(dx, fd, rtol=1e-6, atol=1e-8)


def test_softmax_bwd_row_sums_vanish_and_support_is_respected():
    rng = np.random.default_rng(4)
    x = rng.normal(0.0, 8.0, size=(6, 50))
    dy = rng.normal(size=x.shape)
    dx = oracle.ra_softmax_bwd(x, dy)
    np.testing.assert_allclose(dx.sum(-1), 0.0, atol=1e-12)
    dead = (x.max(-1, keepdims=True) - x) >= 16.0
    assert np.all(dx[dead] == 0.0)


@pytest.mark.parametrize("n,d", [(2, 2), (3, 4), (5, 2), (8, 4)])
@pytest.mark.parametrize("causal", [False, True])
def test_attention_bwd_matches_finite_differences(n, d, causal):
    rng = np.random.default_rng(10 * n + d + causal)
    scale = 0.9
    while True:
        q = rng.normal(0, 1.5, size=(n, d))
        k = rng.normal(0, 1.5, size=(n, d))
        S = scale * q @ k.T
        if causal:
            S = np.where(np.arange(n)[None, :] <= np.arange(n)[:, None], S, -np.inf)
        srt = np.sort(S, axis=-1)
        gaps = srt[:, -1] - srt[:, -2]
        ok = np.where(np.isfinite(gaps), gaps, 1.0)
        if np.all(ok > 2e-2):
            break
    v = rng.normal(size=(n, d))
    do = rng.normal(size=(n, d))
    dq, dk, dv = oracle.ra_attention_head_bwd(q, k, v, do, scale, causal)

    def loss(qq, kk, vv):
        O, *_ = oracle.ra_attention_head_fwd(qq, kk, vv, scale, causal)
        return float((O * do).sum())

    np.testing.assert_allclose(dq, _fd_grad(lambda z: loss(z, k, v), q), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dk, _fd_grad(lambda z: loss(q, z, v), k), rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(dv, _fd_grad(lambda z: loss(q, k, z), v), rtol=1e-6, atol=1e-8)


def _torch_reference(q, k, v, do, scale, causal):
    """Independent torch float64 formulation, differentiated by autograd.

    Masking by boolean selection (no -inf arithmetic), the max via torch.max
    (whose gradient is routed to the returned index), phi built from a clamped
    u so that no NaN gradient leaks out of the dead branch.
    """
    q = torch.tensor(q, requires_grad=True)
    k = torch.tensor(k, requires_grad=True)
    v = torch.tensor(v, requires_grad=True)
    s = scale * torch.einsum("bhid,bhjd->bhij", q, k)
    n_q, n_k = s.shape[-2:]
    keep = torch.ones(n_q, n_k, dtype=torch.bool)
    if causal:
        keep = torch.tril(keep)
    low = s.detach().min() - 100.0
    s_for_max = torch.where(keep, s, low)
    smax = torch.max(s_for_max, dim=-1, keepdim=True).values
    u = (smax - s) / 16.0
    live = keep & (u < 1.0)
    uc = torch.clamp(u, max=1.0)
    w = torch.where(live, ((1.0 - uc) / (1.0 + uc)) ** 8, torch.zeros_like(u))
    p = w / w.sum(-1, keepdim=True)
    o = torch.einsum("bhij,bhjd->bhid", p, v)
    (o * torch.tensor(do)).sum().backward()
    return o.detach().numpy(), q.grad.numpy(), k.grad.numpy(), v.grad.numpy()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("n,d,sigma", [(16, 8, 1.0), (33, 16, 2.5), (24, 4, 6.0)])
def test_attention_bwd_matches_torch_autograd(causal, n, d, sigma):
    rng = np.random.default_rng(n + d)
    q = rng.normal(0, sigma, size=(1, 2, n, d))
    k = rng.normal(0, sigma, size=(1, 2, n, d))
    v = rng.normal(size=(1, 2, n, d))
    do = rng.normal(size=(1, 2, n, d))
    scale = d ** -0.5
    o_ref, dq_ref, dk_ref, dv_ref = _torch_reference(q, k, v, do, scale, causal)
    O, *_ = oracle.ra_attention_fwd(q, k, v, scale=scale, causal=causal)
    dq, dk, dv = oracle.ra_attention_bwd(q, k, v, do, scale=scale, causal=causal)
    np.testing.assert_allclose(O, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq, dq_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, dk_ref, rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, dv_ref, rtol=1e-10, atol=1e-12)


def test_attention_score_gradient_rows_sum_to_zero():
    # dq = scale dS k with sum_j dS_ij = 0, so adding a constant vector c to every key
    # leaves dq unchanged only through ... ; test directly on dS via ra_softmax_bwd
    rng = np.random.default_rng(12)
    q = rng.normal(size=(20, 8))
    k = rng.normal(size=(20, 8))
    v = rng.normal(size=(20, 8))
    do = rng.normal(size=(20, 8))
    S = 0.7 * q @ k.T
    dS = oracle.ra_softmax_bwd(S, do @ v.T)
    np.testing.assert_allclose(dS.sum(-1), 0.0, atol=1e-12)
    # consequence: shifting every key by the same vector does not change dq
    dq1, _, _ = oracle.ra_attention_head_bwd(q, k, v, do, 0.7, False)
    dq2, _, _ = oracle.ra_attention_head_bwd(q, k + 0.5, v, do, 0.7, False)
    np.testing.assert_allclose(dq1, dq2, rtol=1e-9, atol=1e-11)


def test_argmax_override_is_the_branch_of_the_tied_entry():
    # At an exact tie the max is not differentiable; routing the gradient to the second tied
    # entry must give the gradient of the function in which that entry is (just) the maximum.
    rng = np.random.default_rng(21)
    x = rng.normal(0, 3.0, size=(1, 7))
    x[0, 5] = x[0, 2] = x.max() + 0.5          # tie between columns 2 and 5
    dy = rng.normal(size=x.shape)
    default = oracle.ra_softmax_bwd(x, dy)                       # lowest index: column 2
    routed = oracle.ra_softmax_bwd(x, dy, argmax=np.array([5]))
    xp = x.copy()
    xp[0, 5] += 1e-9                                              # column 5 strictly largest
    np.testing.assert_allclose(routed, oracle.ra_softmax_bwd(xp, dy), rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(default, oracle.ra_softmax_bwd(x, dy, argmax=np.array([2])), rtol=0, atol=0)
    assert not np.allclose(default, routed)


def test_argmax_override_with_the_true_argmax_changes_nothing():
    rng = np.random.default_rng(22)
    q, k, v, do = (rng.normal(size=(12, 4)) for _ in range(4))
    S = 0.8 * q @ k.T
    a = np.argmax(np.where(np.tril(np.ones((12, 12), bool)), S, -np.inf), axis=-1)
    base = oracle.ra_attention_head_bwd(q, k, v, do, 0.8, True)
    routed = oracle.ra_attention_head_bwd(q, k, v, do, 0.8, True, argmax=a)
    for g0, g1 in zip(base, routed):
        np.testing.assert_allclose(g1, g0, rtol=1e-13, atol=1e-14)
