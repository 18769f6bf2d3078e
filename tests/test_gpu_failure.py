"""Device-side failure handling without a GPU fault.

With ra_debug_force_timeout on, the MMA thread of each tensor-core kernel first waits on
a barrier that nothing arrives on ("a flag that nothing sets"); with the wait limit set
to 2 ms that wait gives up, the kernel raises its abort flag, every role winds down
(in-flight copies and tensor-core work drained, tensor memory freed) and the kernel
returns.  The status word must read RA_ERR_TIMEOUT, and the context must stay usable:
the next normal call is checked against the oracle.  Small problems keep it short.
"""
import pytest
import torch

import oracle
import parity
import rational_softmax_attention_gb300 as ra
from rational_softmax_attention_gb300.inputs import attention_inputs

pytestmark = pytest.mark.gpu


class forced_timeout:
    def __enter__(self):
        ra.set_wait_limit_ns(2_000_000)
        ra.debug_force_timeout(True)

    def __exit__(self, *exc):
        ra.debug_force_timeout(False)
        ra.set_wait_limit_ns(0)


def test_forward_wait_timeout_is_reported_and_the_context_survives():
    q, k, v = attention_inputs(1, 2, 256, 384, 64, seed=11, dtype=torch.bfloat16, with_dout=False)
    assert ra.device_status() == "RA_OK"
    with forced_timeout():
        ra.ra_attention_forward(q.cuda(), k.cuda(), v.cuda(), scale=0.125, out_dtype=torch.float32)
        torch.cuda.synchronize()
        status = ra.device_status()
    assert status == "RA_ERR_TIMEOUT"
    o, *_ = ra.ra_attention_forward(q.cuda(), k.cuda(), v.cuda(), scale=0.125, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    O, *_ = oracle.ra_attention_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), scale=0.125)
    parity.assert_close_bf16(parity.f64(o), O, "O after a timed-out call")


def test_backward_wait_timeout_is_reported_and_the_context_survives():
    q, k, v, do = attention_inputs(1, 1, 128, 256, 64, seed=12, dtype=torch.bfloat16)
    qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, rm, rs, ra_, _ = ra.ra_attention_forward(qg, kg, vg, scale=0.125, out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    with forced_timeout():
        ra.ra_attention_backward(qg, kg, vg, o, dog, rm, rs, ra_, scale=0.125)
        torch.cuda.synchronize()
        status = ra.device_status()
    assert status == "RA_ERR_TIMEOUT"
    dq, dk, dv = ra.ra_attention_backward(qg, kg, vg, o, dog, rm, rs, ra_, scale=0.125)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    gq, gk, gv = oracle.ra_attention_head_bwd(q[0, 0].double().numpy(), k[0, 0].double().numpy(),
                                              v[0, 0].double().numpy(), do[0, 0].double().numpy(), 0.125, False)
    parity.assert_close_bf16(parity.f64(dq[0, 0]), gq, "dq after a timed-out call")
    parity.assert_close_bf16(parity.f64(dk[0, 0]), gk, "dk after a timed-out call")
    parity.assert_close_bf16(parity.f64(dv[0, 0]), gv, "dv after a timed-out call")


@pytest.mark.parametrize("causal", [False, True])
def test_cta_pair_forward_timeout_is_reported_and_the_context_survives(causal):
    """The D = 128 forward as CTA pairs (the layout of every long D = 128 call): the even
    CTA's issuers give up at the forced wait, each CTA's other roles give up on their own
    CTA's abort flag or wait limit, the even producer settles and drains both CTAs' copies,
    and both CTAs pass the two closing cluster barriers.  The CPU model of this wind-down is
    tests/test_protocol_abort.py."""
    q, k, v = attention_inputs(1, 2, 512, 640, 128, seed=13 + int(causal), dtype=torch.bfloat16, with_dout=False)
    qg, kg, vg = q.cuda(), k.cuda(), v.cuda()
    assert ra.device_status() == "RA_OK"
    ra.debug_fwd_pair(2)
    try:
        with forced_timeout():
            ra.ra_attention_forward(qg, kg, vg, causal=causal, out_dtype=torch.float32)
            torch.cuda.synchronize()
            status = ra.device_status()
        assert status == "RA_ERR_TIMEOUT"
        o, *_ = ra.ra_attention_forward(qg, kg, vg, causal=causal, out_dtype=torch.float32)
        torch.cuda.synchronize()
        assert ra.device_status() == "RA_OK"
    finally:
        ra.debug_fwd_pair(0)
    O, *_ = oracle.ra_attention_fwd(q.double().numpy(), k.double().numpy(), v.double().numpy(), causal=causal)
    parity.assert_close_bf16(parity.f64(o), O, "O after a timed-out CTA-pair call")
