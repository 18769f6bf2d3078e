"""GPU parity of ra_attention_bwd against the float64 oracle.

fp32 inputs (CUDA-core path): max-abs 2e-5 on dq, dk, dv.
bf16 inputs (tensor-core path): max-abs 1e-2 and mean-abs 1e-3 on dq, dk, dv
(fp32 gradients), on the same bf16-rounded inputs.  Where the GPU's argmax
differs from the oracle's lowest-index one, the two keys' float64 scores must
lie within twice the fp32 score-error bound (parity.check_argmax); the oracle
then follows the GPU's branch of the (non-differentiable at a tie) max.
Exact ties, with no exemption at all, are tested in test_gpu_argmax_ties.py.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import rational_softmax_attention_gb300 as ra
from rational_softmax_attention_gb300.inputs import ATTN_LONG_WIDE, ATTN_MODULE_SHAPE, attention_inputs, workload_inputs

pytestmark = pytest.mark.gpu


def gpu_fwd_bwd(q, k, v, do, scale, causal, grad_dtype=torch.float32):
    qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, rm, rs, ra_, _ = ra.ra_attention_forward(qg, kg, vg, scale=scale, causal=causal, out_dtype=torch.float32)
    dq, dk, dv = ra.ra_attention_backward(qg, kg, vg, o, dog, rm, rs, ra_, scale=scale, causal=causal,
                                          grad_dtype=grad_dtype)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    return dq, dk, dv


def wide_gap_inputs(B, H, nq, nk, D, seed, sigma, dtype, scale, causal):
    """Draw until every row's top-2 scaled-score gap exceeds 1e-3 (the backward jumps at argmax ties)."""
    for s in range(seed, seed + 50):
        q, k, v, do = attention_inputs(B, H, nq, nk, D, seed=s, sigma_qk=sigma, dtype=dtype)
        S = scale * torch.einsum("bhid,bhjd->bhij", q.double(), k.double())
        if causal:
            S = S.masked_fill(~torch.ones(nq, nk, dtype=torch.bool).tril(), -np.inf)
        top = S.topk(min(2, nk), dim=-1).values
        if nk == 1 or (top[..., 0] - top[..., 1]).min() > 1e-3:
            return q, k, v, do
    raise RuntimeError("no draw without near-ties")


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("nq,nk", [(1, 1), (5, 5), (17, 40), (40, 17), (100, 100)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp32_backward_matches_oracle(D, nq, nk, causal):
    scale = D ** -0.5
    q, k, v, do = wide_gap_inputs(1, 2, nq, nk, D, nq * nk + D, 1.5, torch.float32, scale, causal)
    dq, dk, dv = gpu_fwd_bwd(q, k, v, do, scale, causal)
    rq, rk, rv = oracle.ra_attention_bwd(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                         do.double().numpy(), scale=scale, causal=causal)
    parity.assert_close_fp32(parity.f64(dq), rq, "dq")
    parity.assert_close_fp32(parity.f64(dk), rk, "dk")
    parity.assert_close_fp32(parity.f64(dv), rv, "dv")


def test_fp32_backward_autograd_function():
    q, k, v, do = wide_gap_inputs(1, 2, 33, 33, 64, 1, 1.0, torch.float32, 0.125, True)
    qg, kg, vg = (t.cuda().requires_grad_(True) for t in (q, k, v))
    out = ra.ra_attention(qg, kg, vg, is_causal=True, scale=0.125)
    out.backward(do.cuda())
    rq, rk, rv = oracle.ra_attention_bwd(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                                         do.double().numpy(), scale=0.125, causal=True)
    parity.assert_close_fp32(parity.f64(qg.grad), rq, "dq")
    parity.assert_close_fp32(parity.f64(kg.grad), rk, "dk")
    parity.assert_close_fp32(parity.f64(vg.grad), rv, "dv")


def check_bf16_heads(q, k, v, do, scale, causal, heads=None):
    """Tensor-core backward against the oracle's full-head backward on the given heads."""
    qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, rm, rs, ra_, _ = ra.ra_attention_forward(qg, kg, vg, scale=scale, causal=causal, out_dtype=torch.float32)
    dq, dk, dv = ra.ra_attention_backward(qg, kg, vg, o, dog, rm, rs, ra_, scale=scale, causal=causal,
                                          grad_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    assert torch.isfinite(dq).all() and torch.isfinite(dk).all() and torch.isfinite(dv).all()
    B, H, nq, _ = q.shape
    nk = k.shape[2]
    heads = heads or [(b, h) for b in range(B) for h in range(H)]
    ties = 0
    for b, h in heads:
        qd, kd, vd, dod = (t[b, h].double().numpy() for t in (q, k, v, do))
        S = scale * (qd @ kd.T)
        if causal:
            S = np.where(np.arange(nk)[None, :] <= np.arange(nq)[:, None], S, -np.inf)
        a_gpu = ra_[b, h].cpu().numpy().astype(np.int64)
        nd = parity.check_argmax(S, a_gpu, parity.score_error_bound(qd, kd, scale),
                                 f"backward [{b},{h}] {tuple(q.shape)} x {nk}")
        ties += nd
        # the oracle's own (lowest-index) branch, unless a near tie made the GPU take the other
        # key: then the oracle follows the GPU's branch of the max (either is a valid gradient)
        gq, gk, gv = oracle.ra_attention_head_bwd(qd, kd, vd, dod, scale, causal, argmax=a_gpu if nd else None)
        parity.assert_close_bf16(parity.f64(dq[b, h]), gq, f"dq[{b},{h}]")
        parity.assert_close_bf16(parity.f64(dk[b, h]), gk, f"dk[{b},{h}]")
        parity.assert_close_bf16(parity.f64(dv[b, h]), gv, f"dv[{b},{h}]")
    return ties


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("nq,nk", [(1, 1), (17, 17), (128, 128), (200, 200), (129, 300), (300, 129), (513, 513)])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_backward_matches_oracle(D, nq, nk, causal):
    q, k, v, do = attention_inputs(1, 2, nq, nk, D, seed=nq * 7 + nk + D, sigma_qk=1.0, dtype=torch.bfloat16)
    check_bf16_heads(q, k, v, do, D ** -0.5, causal)


@pytest.mark.parametrize("sigma", [0.3, 3.0])
def test_bf16_backward_score_spreads(sigma):
    q, k, v, do = attention_inputs(1, 2, 384, 384, 128, seed=int(10 * sigma) + 1, sigma_qk=sigma,
                                   dtype=torch.bfloat16)
    check_bf16_heads(q, k, v, do, 128 ** -0.5, False)


def test_module_shape_workload_backward():
    w = ATTN_MODULE_SHAPE
    q, k, v, do = workload_inputs(w)
    check_bf16_heads(q, k, v, do, w.scale, w.causal)


def test_long_wide_workload_backward_sampled_heads():
    w = ATTN_LONG_WIDE
    q, k, v, do = workload_inputs(w)
    check_bf16_heads(q, k, v, do, w.scale, w.causal, heads=[(0, 0), (w.B - 1, w.H - 1)])


def test_bf16_autograd_function_bf16_gradients():
    q, k, v, do = attention_inputs(2, 3, 160, 160, 64, seed=4, dtype=torch.bfloat16)
    qg, kg, vg = (t.cuda().requires_grad_(True) for t in (q, k, v))
    out = ra.ra_attention(qg, kg, vg, is_causal=True, scale=0.125)
    out.backward(do.cuda())
    assert qg.grad.dtype == torch.bfloat16
    for b in range(2):
        for h in range(3):
            qd, kd, vd, dod = (t[b, h].double().numpy() for t in (q, k, v, do))
            gq, gk, gv = oracle.ra_attention_head_bwd(qd, kd, vd, dod, 0.125, True)
            # bf16 gradients: the fp32 bound plus half a bf16 ulp of each value
            for got, ref in ((qg.grad, gq), (kg.grad, gk), (vg.grad, gv)):
                g = parity.f64(got[b, h])
                assert np.all(np.abs(g - ref) <= 1e-2 + np.abs(ref) * 2.0 ** -8)


@pytest.mark.parametrize("causal", [False, True])
def test_fp32_backward_at_scale(causal):
    """fp32 inputs at N = 2048, D = 128: dq, dk, dv of a whole head against the oracle within
    2e-5.  Where the GPU's argmax differs from the oracle's, it must be a near tie within the
    fp32 score-error bound, and the oracle follows it."""
    scale = 128 ** -0.5
    q, k, v, do = attention_inputs(1, 1, 2048, 2048, 128, seed=31 + int(causal), dtype=torch.float32)
    qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, rm, rs, ra_, _ = ra.ra_attention_forward(qg, kg, vg, scale=scale, causal=causal, out_dtype=torch.float32)
    dq, dk, dv = ra.ra_attention_backward(qg, kg, vg, o, dog, rm, rs, ra_, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    qd, kd, vd, dod = (t[0, 0].double().numpy() for t in (q, k, v, do))
    a_gpu = ra_[0, 0].cpu().numpy().astype(np.int64)
    S = scale * (qd @ kd.T)
    if causal:
        S = np.where(np.tril(np.ones_like(S, dtype=bool)), S, -np.inf)
    nd = parity.check_argmax(S, a_gpu, parity.score_error_bound(qd, kd, scale), f"fp32 backward N2048 causal={causal}")
    rq, rk, rv = oracle.ra_attention_head_bwd(qd, kd, vd, dod, scale, causal, argmax=a_gpu if nd else None)
    parity.assert_close_fp32(parity.f64(dq[0, 0]), rq, "dq")
    parity.assert_close_fp32(parity.f64(dk[0, 0]), rk, "dk")
    parity.assert_close_fp32(parity.f64(dv[0, 0]), rv, "dv")
