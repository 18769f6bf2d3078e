"""Pins for the RaAttention module oracle (oracle/ra_module.py), CPU only."""
import numpy as np
import pytest
import torch

import oracle


def test_layer_norm_is_the_textbook_definition():
    """Against torch.nn.functional.layer_norm in float64 on the CPU (a library routine)."""
    rng = np.random.default_rng(0)
    x = rng.normal(size=(3, 5, 64)) * 3.0 + 1.5
    w, b = rng.normal(size=64), rng.normal(size=64)
    want = torch.nn.functional.layer_norm(torch.from_numpy(x), (64,), torch.from_numpy(w), torch.from_numpy(b),
                                          eps=oracle.ra_module.LN_EPS).numpy()
    np.testing.assert_allclose(oracle.layer_norm(x, w, b), want, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_identity_projections_reduce_to_ra_attention(causal):
    """One head, W_qkv = [I; I; I] and W_proj = I: the module is ra_attention(x, x, x)."""
    rng = np.random.default_rng(1)
    B, N, C = 2, 9, 16
    x = rng.normal(size=(B, N, C))
    eye = np.eye(C)
    y = oracle.ra_attention_module_fwd(x, np.concatenate([eye, eye, eye]), None, eye, None, 1, causal=causal)
    o, *_ = oracle.ra_attention_fwd(x[:, None], x[:, None], x[:, None], causal=causal)
    np.testing.assert_allclose(y, o[:, 0], rtol=0, atol=1e-13)


def test_head_split_matches_explicit_slicing():
    """Head h uses rows [h*hd, (h+1)*hd) of each of the q, k, v blocks of W_qkv and
    columns [h*hd, (h+1)*hd) of W_proj (bias included)."""
    rng = np.random.default_rng(2)
    B, N, C, H = 2, 7, 24, 3
    hd = C // H
    x = rng.normal(size=(B, N, C))
    w_qkv, b_qkv = rng.normal(size=(3 * C, C)) / 5, rng.normal(size=3 * C) / 5
    w_proj, b_proj = rng.normal(size=(C, C)) / 5, rng.normal(size=C) / 5
    y = oracle.ra_attention_module_fwd(x, w_qkv, b_qkv, w_proj, b_proj, H, causal=True)
    want = np.tile(b_proj, (B, N, 1)).astype(np.float64)
    for h in range(H):
        rows = slice(h * hd, (h + 1) * hd)
        q = x @ w_qkv[0 * C:1 * C][rows].T + b_qkv[0 * C:1 * C][rows]
        k = x @ w_qkv[1 * C:2 * C][rows].T + b_qkv[1 * C:2 * C][rows]
        v = x @ w_qkv[2 * C:3 * C][rows].T + b_qkv[2 * C:3 * C][rows]
        o, *_ = oracle.ra_attention_fwd(q[:, None], k[:, None], v[:, None], causal=True)
        want = want + o[:, 0] @ w_proj[:, rows].T
    np.testing.assert_allclose(y, want, rtol=0, atol=1e-12)


def test_qk_norm_applies_per_head_layer_norm():
    rng = np.random.default_rng(3)
    B, N, C, H = 1, 6, 12, 2
    x = rng.normal(size=(B, N, C))
    w_qkv, w_proj = rng.normal(size=(3 * C, C)), rng.normal(size=(C, C))
    qn = (rng.normal(size=C // H), rng.normal(size=C // H))
    kn = (rng.normal(size=C // H), rng.normal(size=C // H))
    y = oracle.ra_attention_module_fwd(x, w_qkv, None, w_proj, None, H, q_norm=qn, k_norm=kn)
    qkv = (x @ w_qkv.T).reshape(B, N, 3, H, C // H).transpose(2, 0, 3, 1, 4)
    q = oracle.layer_norm(qkv[0], *qn)
    k = oracle.layer_norm(qkv[1], *kn)
    o, *_ = oracle.ra_attention_fwd(q, k, qkv[2])
    np.testing.assert_allclose(y, o.transpose(0, 2, 1, 3).reshape(B, N, C) @ w_proj.T, rtol=0, atol=1e-12)


@pytest.mark.parametrize("causal", [False, True])
def test_module_backward_matches_finite_differences(causal):
    """Central differences of sum(dy * y) in x, W_qkv, b_qkv, W_proj, b_proj (float64)."""
    rng = np.random.default_rng(4 + int(causal))
    B, N, C, H = 1, 5, 8, 2
    x = rng.normal(size=(B, N, C))
    w_qkv, b_qkv = rng.normal(size=(3 * C, C)) / 3, rng.normal(size=3 * C) / 3
    w_proj, b_proj = rng.normal(size=(C, C)) / 3, rng.normal(size=C) / 3
    dy = rng.normal(size=(B, N, C))
    args = [x, w_qkv, b_qkv, w_proj, b_proj]
    grads = oracle.ra_attention_module_bwd(x, w_qkv, b_qkv, w_proj, b_proj, H, dy, causal=causal)

    def f(vals):
        return float((oracle.ra_attention_module_fwd(*vals, H, causal=causal) * dy).sum())

    eps = 1e-6
    for i, (arg, g) in enumerate(zip(args, grads)):
        num = np.zeros_like(arg)
        it = np.nditer(arg, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            plus = [a.copy() for a in args]
            minus = [a.copy() for a in args]
            plus[i][idx] += eps
            minus[i][idx] -= eps
            num[idx] = (f(plus) - f(minus)) / (2 * eps)
        np.testing.assert_allclose(g, num, rtol=1e-5, atol=1e-7, err_msg=f"argument {i}")
