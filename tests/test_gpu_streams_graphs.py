"""The attention calls on a stream other than the default one, and captured in a CUDA graph.

Every entry point enqueues its work on the stream it is given and returns; the binding passes
torch's current stream.  Run on a side stream, and replayed from a captured CUDA graph, the
forward and backward must give exactly the results of the same calls run eagerly on the
default stream: every kernel here is deterministic (fixed reduction orders, no atomics in the
data path), so the comparison is bit for bit.  A first (eager) call precedes any capture, as
the library looks up its device status word on a device's first call.
"""
import pytest
import torch

import rational_softmax_attention_gb300 as ra
from rational_softmax_attention_gb300.inputs import attention_inputs

pytestmark = pytest.mark.gpu


def _fwd_bwd(q, k, v, do, causal, mask=None):
    o, rm, rs, ra_, _ = ra.ra_attention_forward(q, k, v, causal=causal, out_dtype=torch.float32, mask=mask)
    dq, dk, dv = ra.ra_attention_backward(q, k, v, o, do, rm, rs, ra_, causal=causal, mask=mask)
    return o, rm, rs, ra_, dq, dk, dv


@pytest.mark.parametrize("D,n,causal", [(64, 300, True), (128, 640, False), (128, 520, True)])
def test_side_stream_gives_the_default_stream_results(D, n, causal):
    q, k, v, do = (t.cuda() for t in attention_inputs(2, 2, n, n, D, seed=D + n))
    ref = _fwd_bwd(q, k, v, do, causal)
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        got = _fwd_bwd(q, k, v, do, causal)
        assert ra.device_status(side) == "RA_OK"
    torch.cuda.synchronize()
    for a, b in zip(ref, got):
        assert torch.equal(a, b)


@pytest.mark.parametrize("D,n,causal,masked", [(64, 300, True, False), (128, 640, False, False),
                                               (128, 520, True, True)])
def test_graph_replay_gives_the_eager_results(D, n, causal, masked):
    q, k, v, do = (t.cuda() for t in attention_inputs(1, 2, n, n, D, seed=3 * D + n))
    mask = None
    if masked:
        m = torch.rand(n, n, generator=torch.Generator().manual_seed(n)) < 0.7
        m[:, 0] = True
        mask = ra.pack_attn_mask(m.cuda(), 1, 2, n, n)
    ref = _fwd_bwd(q, k, v, do, causal, mask)   # eager, and the first call on this device
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    # static inputs: the graph reads these buffers, refilled between replays (filled before the
    # warm-up too: stale memory could trip the fp16-range flag, which stays set until read)
    sq, sk, sv, sdo = (t.clone() for t in (q, k, v, do))
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        _fwd_bwd(sq, sk, sv, sdo, causal, mask)   # warm-up on the capture stream
    side.synchronize()
    assert ra.device_status(side) == "RA_OK"
    with torch.cuda.graph(g, stream=side):
        outs = _fwd_bwd(sq, sk, sv, sdo, causal, mask)
    for _ in range(2):
        for dst, src in ((sq, q), (sk, k), (sv, v), (sdo, do)):
            dst.copy_(src)
        g.replay()
        torch.cuda.synchronize()
        assert ra.device_status() == "RA_OK"
        for a, b in zip(ref, outs):
            assert torch.equal(a, b)
    # a replay on other inputs gives their own results
    q2 = (q.float() * 0.5).to(q.dtype)
    ref2 = _fwd_bwd(q2, k, v, do, causal, mask)
    sq.copy_(q2)
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(ref2, outs):
        assert torch.equal(a, b)


def test_full_size_results_are_bit_identical_across_calls():
    """The B4 H16 N8192 D128 workload (non-causal, sigma 3) run twice: forward and backward
    outputs equal bit for bit (fixed reduction orders, no atomics in the data path), and the
    status word stays clear."""
    from rational_softmax_attention_gb300.inputs import ATTN_LONG_WIDE, workload_inputs
    w = ATTN_LONG_WIDE
    q, k, v, do = (t.cuda() for t in workload_inputs(w)[:4])

    def run():
        o, rm, rs, ra_, _ = ra.ra_attention_forward(q, k, v, scale=w.scale, causal=w.causal, out_dtype=torch.float32)
        dq, dk, dv = ra.ra_attention_backward(q, k, v, o, do, rm, rs, ra_, scale=w.scale, causal=w.causal)
        return o, rm, rs, ra_, dq, dk, dv
    first = run()
    second = run()
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    for a, b in zip(first, second):
        assert torch.equal(a, b)
