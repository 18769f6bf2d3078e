"""Float64 CPU oracle of the RaAttention module.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check and the
benchmark's CPU-baseline leg may import this module; the product path never does, and
this module imports nothing from the product package.

Source page: "Ra-Family: Rational Neural Architecture", section 3, "ra_attention &
RaAttention": a multi-head attention module built on ra_attention.  The page gives the
module's constructor (dim, num_heads, qk_norm, attn_drop, proj_drop, causal) and a call
on x of shape [B, N, dim], not its body.  Readings taken (listed in the design notes):
  * one projection x W_qkv^T (+ b_qkv) to 3*dim values per token, read as (3, heads,
    dim / heads): q, k, v of every head;
  * qk_norm: layer normalisation of q and of k over the head dimension (its own weight
    and bias each, eps 1e-5);
  * ra_attention per head with the default scale 1/sqrt(dim / heads), causal as given;
  * heads concatenated back to dim values per token, then x W_proj^T (+ b_proj);
  * no dropout (the probabilities are 0; stochastic dropout is not part of this path).

Pins: tests/test_oracle_module.py (layer normalisation against its textbook definition
as computed by a library routine; identity projections reduce the module to
ra_attention; the head split against an explicit per-head slicing; the backward against
finite differences of the forward).
"""
from __future__ import annotations

import numpy as np

from .ra_oracle import ra_attention_bwd, ra_attention_fwd

LN_EPS = 1e-5


def layer_norm(x, weight, bias, eps=LN_EPS):
    """(x - mean) / sqrt(var + eps) * weight + bias over the last axis (biased variance)."""
    x = np.asarray(x, dtype=np.float64)
    mean = x.mean(axis=-1, keepdims=True)
    var = ((x - mean) ** 2).mean(axis=-1, keepdims=True)
    return (x - mean) / np.sqrt(var + eps) * weight + bias


def _split_heads(qkv, num_heads):
    """[B, N, 3*dim] -> q, k, v each [B, H, N, dim/H]."""
    B, N, three_dim = qkv.shape
    dim = three_dim // 3
    hd = dim // num_heads
    t = qkv.reshape(B, N, 3, num_heads, hd).transpose(2, 0, 3, 1, 4)
    return t[0], t[1], t[2]


def _merge_heads(o):
    """[B, H, N, hd] -> [B, N, H*hd]."""
    B, H, N, hd = o.shape
    return o.transpose(0, 2, 1, 3).reshape(B, N, H * hd)


def ra_attention_module_fwd(x, w_qkv, b_qkv, w_proj, b_proj, num_heads, causal=False, q_norm=None,
                            k_norm=None, eps=LN_EPS):
    """y [B, N, dim] for x [B, N, dim].  w_qkv [3 dim, dim], w_proj [dim, dim]; biases may be
    None; q_norm / k_norm: (weight, bias) of the per-head layer normalisation, or None."""
    x = np.asarray(x, dtype=np.float64)
    qkv = x @ np.asarray(w_qkv, dtype=np.float64).T
    if b_qkv is not None:
        qkv = qkv + np.asarray(b_qkv, dtype=np.float64)
    q, k, v = _split_heads(qkv, num_heads)
    if q_norm is not None:
        q = layer_norm(q, *q_norm, eps=eps)
    if k_norm is not None:
        k = layer_norm(k, *k_norm, eps=eps)
    o, _, _, _ = ra_attention_fwd(q, k, v, causal=causal)
    y = _merge_heads(o) @ np.asarray(w_proj, dtype=np.float64).T
    if b_proj is not None:
        y = y + np.asarray(b_proj, dtype=np.float64)
    return y


def ra_attention_module_bwd(x, w_qkv, b_qkv, w_proj, b_proj, num_heads, dy, causal=False):
    """Gradients of sum(dy * y) without qk_norm: returns (dx, dw_qkv, db_qkv, dw_proj, db_proj)
    (bias gradients None where the bias is None).  Linear maps by their transposes, the
    attention by the closed-form backward of the attention oracle."""
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    w_qkv = np.asarray(w_qkv, dtype=np.float64)
    w_proj = np.asarray(w_proj, dtype=np.float64)
    qkv = x @ w_qkv.T
    if b_qkv is not None:
        qkv = qkv + np.asarray(b_qkv, dtype=np.float64)
    q, k, v = _split_heads(qkv, num_heads)
    o, _, _, _ = ra_attention_fwd(q, k, v, causal=causal)
    om = _merge_heads(o)
    B, N, dim = x.shape
    dw_proj = dy.reshape(-1, dim).T @ om.reshape(-1, dim)
    db_proj = dy.reshape(-1, dim).sum(axis=0) if b_proj is not None else None
    dom = dy @ w_proj
    hd = dim // num_heads
    do = dom.reshape(B, N, num_heads, hd).transpose(0, 2, 1, 3)
    dq, dk, dv = ra_attention_bwd(q, k, v, do, causal=causal)
    dqkv = np.stack([dq, dk, dv]).transpose(1, 3, 0, 2, 4).reshape(B, N, 3 * dim)
    dx = dqkv @ w_qkv
    dw_qkv = dqkv.reshape(-1, 3 * dim).T @ x.reshape(-1, dim)
    db_qkv = dqkv.reshape(-1, 3 * dim).sum(axis=0) if b_qkv is not None else None
    return dx, dw_qkv, db_qkv, dw_proj, db_proj
