"""Float64 CPU oracle for rational-softmax (Ra-family) attention.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the test suite, the smoke check
and the benchmark's CPU-baseline leg may import this module; the product path
(the CUDA library and its Python binding) never does, and this module imports
nothing from the product package.

Everything here is deliberately plain: the full score matrix is materialised
per (batch, head), every step is a NumPy float64 array expression that can be
checked against the page by eye, and no step is blocked, fused or reordered.

Source page: "Ra-Family: Rational Neural Architecture" (LuminaV-Optimizer
docs/nn/README.md), section 3 "Rational Attention & Softmax".

  * ra_softmax bullets: shift Delta_i = x_max - x_i; for Delta_i < 16 the
    rational numerator u_i = Delta_i/16, q_i = (1-u_i)/(1+u_i), phi_i = q_i^8;
    phi_i is exactly 0 for Delta_i >= 16; the normaliser sum(phi) is >= 1
    because the maximum has phi = 1; backward from the closed form
    d phi/du = -16 phi / (1-u^2) on u < 1.
  * ra_attention bullets: (Q, K, V) -> O with the ra_softmax of the scores
    in place of the standard softmax, a drop-in for scaled_dot_product_attention
    (so scores = scale * Q K^T, default scale 1/sqrt(D), is_causal = top-left
    mask j <= i), tiled so that [B, H, N_Q, N_K] is never stored.

Readings taken where the page is silent (each is listed with its reason in the
design notes of the repository):
  * the gradient goes through x_max as well (the true derivative of the
    composite function): the argmax entry of each row receives minus the sum
    of the other entries' gradients;
  * the argmax is the lowest index among exact maxima;
  * masked entries are excluded from the max and get phi = 0; a row with no
    allowed entry gives p = 0, O = 0, sum = 0, argmax = -1;
  * scale <= 0 means 1/sqrt(D).

Parity pins for every function here live in tests/test_oracle_*.py; none of
this module is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

# Width of the compact support: phi is exactly zero once Delta >= SUPPORT.
SUPPORT = 16.0
# Power applied to the Cayley ratio q = (1-u)/(1+u).
POWER = 8


def ra_phi(delta):
    """phi(Delta): the unnormalised ra_softmax weight of an entry at shift Delta.

    Page "Ra-Family: Rational Neural Architecture", section 3, ra_softmax:
    u = Delta/16, q = (1-u)/(1+u), phi = q^8 for Delta < 16 and exactly 0
    for Delta >= 16.
    """
    delta = np.asarray(delta, dtype=np.float64)
    u = delta / SUPPORT
    live = u < 1.0
    q = np.where(live, (1.0 - u) / (1.0 + u), 0.0)
    return np.where(live, q ** POWER, 0.0)


def _row_max_and_argmax(x, allowed):
    """Row maximum over the allowed entries and the lowest index attaining it."""
    xm = np.where(allowed, x, -np.inf)
    m = xm.max(axis=-1)
    has_any = allowed.any(axis=-1)
    # argmax of a boolean array returns the first True, i.e. the lowest index.
    a = np.argmax(allowed & (xm == m[..., None]), axis=-1).astype(np.int64)
    a = np.where(has_any, a, -1)
    m = np.where(has_any, m, 0.0)
    return m, a, has_any


def ra_softmax(x, allowed=None):
    """ra_softmax along the last axis of a float64 array.

    Page "Ra-Family: Rational Neural Architecture", section 3, ra_softmax:
    Delta_i = x_max - x_i, phi_i from ra_phi, p_i = phi_i / sum_j phi_j.
    `allowed` (bool, same shape) excludes entries from the max and the sum.
    Returns (p, m, s, a): probabilities, row max, row sum of phi, argmax.
    """
    x = np.asarray(x, dtype=np.float64)
    if allowed is None:
        allowed = np.ones(x.shape, dtype=bool)
    m, a, has_any = _row_max_and_argmax(x, allowed)
    delta = m[..., None] - x
    phi = np.where(allowed, ra_phi(np.where(allowed, delta, SUPPORT)), 0.0)
    s = phi.sum(axis=-1)
    p = np.where(has_any[..., None], phi / np.where(s > 0, s, 1.0)[..., None], 0.0)
    return p, m, s, a


def ra_softmax_bwd(x, dy, allowed=None, argmax=None):
    """Gradient of sum(dy * ra_softmax(x)) with respect to x, last axis.

    Built from the page's closed form d phi/du = -16 phi/(1-u^2) on u < 1
    (section 3, ra_softmax, "Closed-Form Backward Pass") and the chain rule:
      dL/dphi_j = (dy_j - D)/sum(phi),   D = sum_k p_k dy_k
      u_j = (x_max - x_j)/16  ->  du_j/dx_j = -1/16 (j != argmax), du_j/dx_max = 1/16
    so for j != a (a = argmax): dx_j = p_j (dy_j - D) / (1 - u_j^2), zero if
    u_j >= 1 or j is masked, and dx_a = -sum_{j != a} dx_j.

    `argmax` (optional, int array of the row shape) names the entry treated as
    x_max.  The max is not differentiable at a tie, and two entries whose values
    differ by less than rounding are both valid choices; passing the index a
    fixed-precision implementation chose reproduces its branch of the gradient
    (x_max is then x[argmax], the value that implementation's weights used).
    """
    x = np.asarray(x, dtype=np.float64)
    dy = np.asarray(dy, dtype=np.float64)
    if allowed is None:
        allowed = np.ones(x.shape, dtype=bool)
    if argmax is None:
        p, m, s, a = ra_softmax(x, allowed)
    else:
        a = np.asarray(argmax, dtype=np.int64)
        # a row with no allowed entry carries argmax -1: its phi, p and gradient are 0
        m = np.take_along_axis(x, np.maximum(a, 0)[..., None], axis=-1)[..., 0]
        phi = np.where(allowed, ra_phi(np.where(allowed, m[..., None] - x, SUPPORT)), 0.0)
        tot = phi.sum(axis=-1, keepdims=True)
        p = phi / np.where(tot > 0, tot, 1.0)
    D = (p * dy).sum(axis=-1, keepdims=True)
    u = (m[..., None] - x) / SUPPORT
    live = allowed & (u < 1.0)
    idx = np.arange(x.shape[-1])
    not_arg = idx != a[..., None]
    denom = np.where(live, 1.0 - u * u, 1.0)
    e = np.where(live & not_arg, p * (dy - D) / denom, 0.0)
    r = e.sum(axis=-1)
    dx = e.copy()
    rows = np.nonzero(a >= 0)
    dx[rows + (a[rows],)] = -r[rows]
    return dx


def _causal_allowed(n_q, n_k):
    """Top-left causal mask of scaled_dot_product_attention: key j visible to query i iff j <= i."""
    return np.arange(n_k)[None, :] <= np.arange(n_q)[:, None]


def default_scale(D, scale):
    return 1.0 / np.sqrt(D) if (scale is None or scale <= 0) else float(scale)


def _allowed(n_q, n_k, causal, mask):
    """Entries that take part: the causal mask (if any) and a boolean attn_mask [N_Q, N_K]
    (True = the query may attend to the key), as scaled_dot_product_attention reads them."""
    allowed = _causal_allowed(n_q, n_k) if causal else np.ones((n_q, n_k), dtype=bool)
    if mask is not None:
        allowed = allowed & np.asarray(mask, dtype=bool)
    return allowed


def ra_attention_head_fwd(q, k, v, scale, causal, mask=None):
    """One (batch, head): O = ra_softmax(scale * q k^T [+ causal mask] [+ attn_mask]) v.

    Page "Ra-Family: Rational Neural Architecture", section 3, ra_attention
    bullets (functional form, drop-in for scaled_dot_product_attention).
    q: [N_Q, D], k, v: [N_K, D] float64; mask: optional boolean [N_Q, N_K].
    Returns O [N_Q, D] and the per-row statistics (m = max scaled score,
    s = sum phi, a = argmax key index); a row with no allowed key gives O = 0.
    """
    S = scale * (q @ k.T)
    allowed = _allowed(q.shape[0], k.shape[0], causal, mask)
    P, m, s, a = ra_softmax(S, allowed)
    O = P @ v
    return O, m, s, a


def ra_attention_head_bwd(q, k, v, do, scale, causal, argmax=None, mask=None):
    """One (batch, head): gradients of sum(do * O) with respect to q, k, v.

    The score gradient dS is ra_softmax_bwd applied to the materialised scores
    with upstream gradient dP = do v^T; then dq = scale dS k, dk = scale dS^T q,
    dv = P^T do (the plain chain rule through S = scale q k^T and O = P v).
    `argmax` (optional, per query row) is passed on to ra_softmax_bwd, and P is
    then formed with x_max = S[i, argmax_i] as well.
    """
    S = scale * (q @ k.T)
    allowed = _allowed(q.shape[0], k.shape[0], causal, mask)
    if argmax is None:
        P, _, _, _ = ra_softmax(S, allowed)
    else:
        am = np.asarray(argmax, dtype=np.int64)
        m = np.take_along_axis(S, np.maximum(am, 0)[:, None], axis=-1)   # rows with argmax -1 have no allowed key
        phi = np.where(allowed, ra_phi(np.where(allowed, m - S, SUPPORT)), 0.0)
        tot = phi.sum(axis=-1, keepdims=True)
        P = phi / np.where(tot > 0, tot, 1.0)
    dP = do @ v.T
    dS = ra_softmax_bwd(S, dP, allowed, argmax=argmax)
    dq = scale * (dS @ k)
    dk = scale * (dS.T @ q)
    dv = P.T @ do
    return dq, dk, dv


def _head_mask(mask, b, h):
    """The [N_Q, N_K] slice of a mask broadcastable to [B, H, N_Q, N_K] (or None)."""
    if mask is None:
        return None
    m = np.asarray(mask, dtype=bool)
    while m.ndim < 4:
        m = m[None]
    return m[b if m.shape[0] > 1 else 0, h if m.shape[1] > 1 else 0]


def ra_attention_fwd(q, k, v, scale=None, causal=False, mask=None):
    """Batched [B, H, N, D] forward, one head at a time (float64).

    mask: optional boolean attn_mask broadcastable to [B, H, N_Q, N_K].
    Returns O [B,H,N_Q,D], m [B,H,N_Q], s [B,H,N_Q], a [B,H,N_Q].
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, n_q, D = q.shape
    scale = default_scale(D, scale)
    O = np.zeros((B, H, n_q, v.shape[-1]))
    m = np.zeros((B, H, n_q))
    s = np.zeros((B, H, n_q))
    a = np.zeros((B, H, n_q), dtype=np.int64)
    for b in range(B):
        for h in range(H):
            O[b, h], m[b, h], s[b, h], a[b, h] = ra_attention_head_fwd(q[b, h], k[b, h], v[b, h], scale, causal,
                                                                       _head_mask(mask, b, h))
    return O, m, s, a


def ra_attention_bwd(q, k, v, do, scale=None, causal=False, mask=None):
    """Batched [B, H, N, D] backward, one head at a time (float64); mask as in ra_attention_fwd."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, H, _, D = q.shape
    scale = default_scale(D, scale)
    dq = np.zeros(q.shape)
    dk = np.zeros(k.shape)
    dv = np.zeros(v.shape)
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = ra_attention_head_bwd(q[b, h], k[b, h], v[b, h], do[b, h], scale, causal,
                                                                 mask=_head_mask(mask, b, h))
    return dq, dk, dv


def ra_attention_rows_fwd(q, k, v, rows, scale, causal):
    """Forward for a chosen subset of query rows of one head (for sampled checks at full size).

    q: [N_Q, D], k, v: [N_K, D]; rows: 1-D int array of query indices.
    Each row is independent of the others, so this is the same arithmetic as
    ra_attention_head_fwd restricted to those rows.
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    rows = np.asarray(rows)
    S = scale * (q[rows] @ k.T)
    if causal:
        allowed = np.arange(k.shape[0])[None, :] <= rows[:, None]
    else:
        allowed = np.ones(S.shape, dtype=bool)
    P, m, s, a = ra_softmax(S, allowed)
    return P @ v, m, s, a
