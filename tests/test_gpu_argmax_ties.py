"""Exact argmax ties on the GPU: the lowest key index among exact maxima, with no exemption.

The pages are silent on ties; the reading taken is that the row maximum's index is the
lowest key index among exact maxima, in the oracle and in every kernel.  Random inputs
can only test that up to near ties (parity.check_argmax).  Here the inputs are built so
that the tensor cores' fp32 scores equal the oracle's float64 scores exactly:
  * Q and K hold multiples of 1/4 in [-3/4, 3/4] (exact in bf16 and in fp16, the
    backward's operand format); every product is a multiple of 1/16 and every partial
    sum of a 64- or 128-term dot product stays below 2^7 in magnitude, so each score is
    exact whatever the order and width of the accumulation;
  * the scale is a power of two.
Scores that tie, tie exactly in both precisions, and scores that differ, differ by at
least scale / 16.  So every row's argmax must equal the oracle's default (lowest-index)
choice bit for bit, and so must row_m; the backward is compared with the oracle's
default branch, with no argmax passed in.

Ties are planted where the kernels split a row: key rows duplicated across 32-column
chunk boundaries (the forward's argmax search unit), across the two 64-key halves that a
CTA pair splits each key tile into, across 128-key tile boundaries, within a chunk, far
apart, and three times.  A query row aligned with one duplicated key vector has exactly
those duplicates as its maxima (any other key scores strictly less), so the lowest
visible duplicate must win; causal rows that see only part of a group, rows of q = 0
(every visible score equal: the lowest visible key wins) and rows of random multiples
(chance ties among random keys) complete the set.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import rational_softmax_attention_gb300 as ra

pytestmark = pytest.mark.gpu

# groups of key positions that carry one identical key vector (positions >= N_K dropped)
TIE_GROUPS = [(31, 32), (63, 64), (95, 96), (127, 128), (40, 41), (5, 300), (255, 256), (10, 138, 266),
              (383, 384, 511), (200, 520), (639, 640)]


def tie_inputs(B, H, nq, nk, D, seed):
    """Q, K on the grid {-3/4, ..., 3/4} with planted duplicate keys; V, dO ~ N(0, 1); bf16."""
    g = torch.Generator("cpu").manual_seed(seed)

    def grid(shape):
        return torch.randint(-3, 4, shape, generator=g).to(torch.float32) / 4

    q, k = grid((B, H, nq, D)), grid((B, H, nk, D))
    v = torch.randn((B, H, nk, D), generator=g)
    do = torch.randn((B, H, nq, D), generator=g)
    groups = [tuple(p for p in grp if p < nk) for grp in TIE_GROUPS]
    groups = [grp for grp in groups if len(grp) >= 2]
    for b in range(B):
        for h in range(H):
            hot = []
            for grp in groups:
                vec = torch.where(torch.rand(D, generator=g) < 0.5, -0.75, 0.75)
                k[b, h, list(grp)] = vec
                hot.append(vec)
            for r in range(nq):
                kind = r % 4
                if kind in (0, 2) and hot:      # aligned: that group's duplicates are the exact maxima
                    q[b, h, r] = hot[(r // 4 + b + h) % len(hot)]
                elif kind == 1:                 # every visible score 0
                    q[b, h, r] = 0.0
    return tuple(t.to(torch.bfloat16) for t in (q, k, v, do))


def run_and_check(q, k, v, do, scale, causal, mask_np=None, pair_mode=0):
    B, H, nq, D = q.shape
    nk = k.shape[2]
    qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    pm = None
    if mask_np is not None:
        pm = ra.pack_attn_mask(torch.from_numpy(np.ascontiguousarray(mask_np)).cuda(), B, H, nq, nk)
    ra.debug_fwd_pair(pair_mode)
    try:
        o, rm, rs, ra_, _ = ra.ra_attention_forward(qg, kg, vg, scale=scale, causal=causal, out_dtype=torch.float32,
                                                    mask=pm)
        dq, dk, dv = ra.ra_attention_backward(qg, kg, vg, o, dog, rm, rs, ra_, scale=scale, causal=causal,
                                              grad_dtype=torch.float32, mask=pm)
        torch.cuda.synchronize()
    finally:
        ra.debug_fwd_pair(0)
    assert ra.device_status() == "RA_OK"
    tied_rows = 0
    for b in range(B):
        for h in range(H):
            qd, kd, vd, dod = (t[b, h].double().numpy() for t in (q, k, v, do))
            hm = None if mask_np is None else parity_head_mask(mask_np, b, h)
            O, m, s, a = oracle.ra_attention_head_fwd(qd, kd, vd, scale, causal, mask=hm)
            allowed = np.ones((nq, nk), dtype=bool) if hm is None else hm.copy()
            if causal:
                allowed &= np.tril(np.ones((nq, nk), dtype=bool))
            S = np.where(allowed, scale * (qd @ kd.T), -np.inf)
            has = allowed.any(axis=1)
            tied_rows += int(np.count_nonzero((S == S.max(axis=1, keepdims=True)).sum(axis=1)[has] > 1))
            np.testing.assert_array_equal(ra_[b, h].cpu().numpy(), a, err_msg=f"row_arg [{b},{h}]")
            np.testing.assert_array_equal(parity.f64(rm[b, h])[has], m[has], err_msg=f"row_m [{b},{h}]")
            np.testing.assert_allclose(parity.f64(rs[b, h]), s, rtol=1e-4, err_msg=f"row_s [{b},{h}]")
            parity.assert_close_bf16(parity.f64(o[b, h]), O, f"O[{b},{h}]")
            gq, gk, gv = oracle.ra_attention_head_bwd(qd, kd, vd, dod, scale, causal, mask=hm)
            parity.assert_close_bf16(parity.f64(dq[b, h]), gq, f"dq[{b},{h}]")
            parity.assert_close_bf16(parity.f64(dk[b, h]), gk, f"dk[{b},{h}]")
            parity.assert_close_bf16(parity.f64(dv[b, h]), gv, f"dv[{b},{h}]")
            parity.ARGMAX_LOG.append((f"exact ties [{b},{h}] {nq}x{nk} D{D}", nq, 0, 0))
    # the planted and chance ties must actually be there: at least a third of the rows
    assert tied_rows >= B * H * nq // 3, f"only {tied_rows} rows with tied maxima"
    return ra_


def parity_head_mask(mask_np, b, h):
    m = np.asarray(mask_np, dtype=bool)
    while m.ndim < 4:
        m = m[None]
    return m[b if m.shape[0] > 1 else 0, h if m.shape[1] > 1 else 0]


# (D, forward layout): D = 64 single CTAs; D = 128 as single CTAs (mode 1) and CTA pairs (mode 2)
LAYOUTS = [(64, 0), (128, 1), (128, 2)]


@pytest.mark.parametrize("D,pair_mode", LAYOUTS)
@pytest.mark.parametrize("nq,nk", [(300, 300), (513, 641), (641, 513)])
@pytest.mark.parametrize("causal", [False, True])
def test_exact_ties_take_the_lowest_index(D, pair_mode, nq, nk, causal):
    q, k, v, do = tie_inputs(1, 2, nq, nk, D, seed=nq + nk + D + pair_mode)
    scale = 1.0 / 8.0 if D == 64 else 1.0 / 16.0
    run_and_check(q, k, v, do, scale, causal, pair_mode=pair_mode)


@pytest.mark.parametrize("D,pair_mode", LAYOUTS)
@pytest.mark.parametrize("causal", [False, True])
def test_exact_ties_under_an_attention_mask(D, pair_mode, causal):
    """A mask removes some duplicates of a group: the lowest allowed one must win."""
    nq, nk = 520, 641
    q, k, v, do = tie_inputs(2, 1, nq, nk, D, seed=7 + D + pair_mode + int(causal))
    rng = np.random.default_rng(D + int(causal))
    mask = rng.random((2, 1, nq, nk)) < 0.6
    mask[..., 0] = True
    scale = 1.0 / 8.0 if D == 64 else 1.0 / 16.0
    run_and_check(q, k, v, do, scale, causal, mask_np=mask, pair_mode=pair_mode)


def test_all_scores_equal_gives_the_first_visible_key():
    """q = 0 everywhere: every visible score is 0, so row_arg is 0 (the first key), row_m is
    0, every phi is 1 and O is the running (causal) or full mean of V."""
    B, H, n, D = 1, 2, 700, 128
    _, k, v, do = tie_inputs(B, H, n, n, D, seed=3)
    q = torch.zeros((B, H, n, D), dtype=torch.bfloat16)
    for mode in (1, 2):
        for causal in (False, True):
            a = run_and_check(q, k, v, do, 1.0 / 16.0, causal, pair_mode=mode)
            assert torch.all(a == 0)
