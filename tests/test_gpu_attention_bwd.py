"""GPU parity of ra_attention_bwd against the float64 oracle.

fp32 inputs (CUDA-core path): max-abs 2e-5 on dq, dk, dv.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import rational_softmax_attention_gb300 as ra
from rational_softmax_attention_gb300.inputs import attention_inputs

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
