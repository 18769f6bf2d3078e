"""The fp16 operand format of the bf16 tensor-core path, at the edges of its range.

The forward forms P V, and the backward every product, with fp16 copies of its bf16
operands (V in the forward; Q, K, V and dO in the backward).  bf16 carries 8 significant
bits and fp16 11, so the copy is exact for normal fp16 values, 2^-14 <= |x| <= 65504.
Below 2^-14 fp16 is subnormal (spacing 2^-24): a value keeps its bits above 2^-24 and is
rounded to that spacing, and below 2^-25 it becomes 0.  Above 65504 (and for NaN) the copy
saturates and the call reports RA_ERR_UNSUPPORTED through ra_device_status().

Checked here: a large |v| (forward) or |q| or non-finite dO (backward) is reported, and the
next call is clean; tiny operands give the oracle's results within the parity bounds, and
scaled back up they equal the oracle evaluated on the operand rounded to fp16, which shows
that rounding is the only loss.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import rational_softmax_attention_gb300 as ra
from rational_softmax_attention_gb300.inputs import attention_inputs

pytestmark = pytest.mark.gpu


def _fwd_bwd(q, k, v, do, scale, causal, backward=True):
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    o, rm, rs, ra_, _ = ra.ra_attention_forward(qg, kg, vg, scale=scale, causal=causal, out_dtype=torch.float32)
    torch.cuda.synchronize()
    st_fwd = ra.device_status()
    grads, st_bwd = None, None
    if backward:
        grads = ra.ra_attention_backward(qg, kg, vg, o, do.cuda(), rm, rs, ra_, scale=scale, causal=causal)
        torch.cuda.synchronize()
        st_bwd = ra.device_status()
    return o, grads, st_fwd, st_bwd


@pytest.mark.parametrize("D", [64, 128])
def test_v_beyond_the_fp16_range_is_reported_by_the_forward(D):
    q, k, v, do = attention_inputs(1, 2, 200, 300, D, seed=40 + D)
    v[0, 1, 17, 3] = 70000.0          # bf16 keeps it (70144); fp16 cannot
    assert ra.device_status() == "RA_OK"
    _, _, st_fwd, _ = _fwd_bwd(q, k, v, do, D ** -0.5, False, backward=False)
    assert st_fwd == "RA_ERR_UNSUPPORTED"
    v[0, 1, 17, 3] = 1.0
    o, _, st_fwd, _ = _fwd_bwd(q, k, v, do, D ** -0.5, False, backward=False)
    assert st_fwd == "RA_OK"
    O, *_ = oracle.ra_attention_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale=D ** -0.5)
    parity.assert_close_bf16(parity.f64(o), O, "O after a reported call")


@pytest.mark.parametrize("what", ["q", "dout_nan"])
def test_operands_beyond_the_fp16_range_are_reported_by_the_backward(what):
    q, k, v, do = attention_inputs(1, 1, 160, 160, 64, seed=44)
    if what == "q":
        q[0, 0, 5, 7] = -1.0e5        # fine for Q K^T in bf16; the backward's fp16 copy saturates
    else:
        do[0, 0, 9, 1] = float("nan")
    _, _, st_fwd, st_bwd = _fwd_bwd(q, k, v, do, 0.125, True)
    assert st_fwd == "RA_OK"
    assert st_bwd == "RA_ERR_UNSUPPORTED"
    q2, k2, v2, do2 = attention_inputs(1, 1, 160, 160, 64, seed=44)
    _, grads, st_fwd, st_bwd = _fwd_bwd(q2, k2, v2, do2, 0.125, True)
    assert (st_fwd, st_bwd) == ("RA_OK", "RA_OK")
    gq, gk, gv = oracle.ra_attention_head_bwd(*(t[0, 0].double().numpy() for t in (q2, k2, v2, do2)), 0.125, True)
    for name, got, want in zip(("dq", "dk", "dv"), grads, (gq, gk, gv)):
        parity.assert_close_bf16(parity.f64(got[0, 0]), want, f"{name} after a reported call")


def _as_fp16(t):
    return t.to(torch.float16).double().numpy()


@pytest.mark.parametrize("exp", [-18, -23])
def test_subnormal_range_operands(exp):
    """V and dO at 2^exp (fp16 subnormals, part of them flushed to 0 at exp = -23): the
    outputs meet the parity bounds, and O / 2^exp, dv / 2^exp equal the oracle on the
    fp16-rounded operands within the bf16 bounds."""
    B, H, n, D = 1, 2, 300, 128
    q, k, v, do = attention_inputs(B, H, n, n, D, seed=50 - exp)
    v = (v.float() * 2.0 ** exp).to(torch.bfloat16)
    do = (do.float() * 2.0 ** exp).to(torch.bfloat16)
    scale = D ** -0.5
    o, (dq, dk, dv), st_fwd, st_bwd = _fwd_bwd(q, k, v, do, scale, True)
    assert (st_fwd, st_bwd) == ("RA_OK", "RA_OK")   # subnormals are not a range error
    for b in range(B):
        for h in range(H):
            qd, kd, vd, dod = (t[b, h].double().numpy() for t in (q, k, v, do))
            O, *_ = oracle.ra_attention_head_fwd(qd, kd, vd, scale, True)
            gq, gk, gv = oracle.ra_attention_head_bwd(qd, kd, vd, dod, scale, True)
            for name, got, want in (("O", o, O), ("dq", dq, gq), ("dk", dk, gk), ("dv", dv, gv)):
                parity.assert_close_bf16(parity.f64(got[b, h]), want, f"{name}[{b},{h}] at 2^{exp}")
            v16, do16 = _as_fp16(v[b, h]), _as_fp16(do[b, h])
            O16, *_ = oracle.ra_attention_head_fwd(qd, kd, v16, scale, True)
            _, _, gv16 = oracle.ra_attention_head_bwd(qd, kd, v16, do16, scale, True)
            s = 2.0 ** -exp
            parity.assert_close_bf16(parity.f64(o[b, h]) * s, O16 * s, f"O / 2^{exp} [{b},{h}] vs fp16-rounded V")
            parity.assert_close_bf16(parity.f64(dv[b, h]) * s, gv16 * s, f"dv / 2^{exp} [{b},{h}] vs fp16-rounded dO")
