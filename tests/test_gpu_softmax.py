"""GPU parity of the ra_softmax row kernels against the float64 oracle (fp32: max-abs 2e-5)."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import parity
import rational_softmax_attention_gb300 as ra
from rational_softmax_attention_gb300.inputs import RA_SOFTMAX_LONG_ROWS, softmax_inputs

pytestmark = pytest.mark.gpu


def _run(x_cpu):
    y = ra.ra_softmax(x_cpu.cuda())
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    return parity.f64(y)


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 3), (5, 4), (7, 100), (9, 256), (4, 257), (2, 1000),
                                       (3, 1024), (2, 2048), (2, 4096), (3, 8192), (2, 8191), (2, 12288),
                                       (2, 16384), (2, 16388), (1, 40000)])
def test_ra_softmax_matches_oracle(rows, cols):
    x = softmax_inputs(rows, cols, seed=rows * 7 + cols, sigma=4.0)
    got = _run(x)
    want, *_ = oracle.ra_softmax(x.double().numpy())
    parity.assert_close_fp32(got, want, f"ra_softmax[{rows}x{cols}]")
    xd = x.double().numpy()
    dead = (xd.max(-1, keepdims=True) - xd) >= 16.0
    assert np.all(got[dead] == 0.0), "entries at Delta >= 16 must be exactly 0"
    np.testing.assert_allclose(got.sum(-1), 1.0, atol=1e-5)


def test_ra_softmax_worked_example():
    # the page's worked logits; exact rationals are pinned on the oracle side
    x = torch.tensor([[2.0, 1.0, 0.0], [5.0, 1.0, -10.0]])
    got = _run(x)
    want, *_ = oracle.ra_softmax(x.double().numpy())
    parity.assert_close_fp32(got, want, "worked example")


def test_ra_softmax_full_workload():
    w = RA_SOFTMAX_LONG_ROWS
    x = softmax_inputs(w.rows, w.cols, seed=w.seed, sigma=w.sigma)
    got = _run(x)
    want, *_ = oracle.ra_softmax(x.double().numpy())
    parity.assert_close_fp32(got, want, w.name)
    xd = x.double().numpy()
    dead = (xd.max(-1, keepdims=True) - xd) >= 16.0
    assert dead.mean() > 0.3          # the workload really exercises the compact support
    assert np.all(got[dead] == 0.0)


def test_ra_softmax_in_place_and_misaligned_rows():
    x = softmax_inputs(6, 130, seed=3, sigma=3.0)
    want, *_ = oracle.ra_softmax(x.double().numpy())
    xg = x.cuda()
    L = ra.lib()
    st = torch.cuda.current_stream().cuda_stream
    import ctypes
    assert L.ra_softmax_fwd(ctypes.c_void_p(xg.data_ptr()), ctypes.c_void_p(xg.data_ptr()), 6, 130, 0,
                            ctypes.c_void_p(st)) == 0
    torch.cuda.synchronize()
    parity.assert_close_fp32(parity.f64(xg), want, "in place, cols % 4 != 0")
    # a row view starting 4 bytes off a 16-byte boundary takes the generic kernel
    buf = softmax_inputs(1, 4 * 64 + 1, seed=4, sigma=3.0).cuda()
    view = buf[0, 1:].reshape(4, 64)
    got = parity.f64(ra.ra_softmax(view.contiguous()))
    want2, *_ = oracle.ra_softmax(view.double().cpu().numpy())
    parity.assert_close_fp32(got, want2, "offset rows")


@pytest.mark.parametrize("rows,cols", [(1, 1), (3, 5), (4, 64), (2, 1000), (5, 2052), (3, 4096), (2, 8192),
                                       (2, 8196)])
def test_ra_softmax_backward_matches_oracle(rows, cols):
    g = torch.Generator().manual_seed(cols)
    x = torch.randn(rows, cols, generator=g) * 4.0
    dy = torch.randn(rows, cols, generator=g)
    xg = x.cuda()
    p = ra.ra_softmax(xg)
    dx = ra.ra_softmax_backward(xg, p, dy.cuda())
    torch.cuda.synchronize()
    want = oracle.ra_softmax_bwd(x.double().numpy(), dy.double().numpy())
    parity.assert_close_fp32(parity.f64(dx), want, f"ra_softmax_bwd[{rows}x{cols}]")


def test_ra_softmax_backward_ties_and_in_place():
    """Rows whose maximum occurs twice, in columns held by different threads: the gradient of
    the maximum goes to the lowest of them (as in the oracle).  dx written over dy."""
    g = torch.Generator().manual_seed(11)
    rows, cols = 6, 8192
    x = torch.randn(rows, cols, generator=g) * 4.0
    for r, (c1, c2) in enumerate([(5, 4000), (4000, 5), (1023, 1024), (0, 8191), (8190, 8191), (17, 17 + 4 * 256)]):
        top = float(x[r].max()) + 1.0
        x[r, c1] = top
        x[r, c2] = top
    dy = torch.randn(rows, cols, generator=g)
    xg = x.cuda()
    p = ra.ra_softmax(xg)
    dyg = dy.cuda()
    dx = ra.ra_softmax_backward(xg, p, dyg, out=dyg)
    torch.cuda.synchronize()
    assert dx.data_ptr() == dyg.data_ptr()
    want = oracle.ra_softmax_bwd(x.double().numpy(), dy.double().numpy())
    parity.assert_close_fp32(parity.f64(dx), want, "ra_softmax_bwd ties, in place")


def _assert_bf16_rounding_of(got, want, what):
    """got is want (float64) computed in fp32 and rounded once to bf16: within half a bf16 ulp
    of want (2^(floor(log2 |want|) - 8), bf16 keeping 8 significant bits) plus the fp32
    arithmetic (1e-6 absolute) of every element."""
    got = np.asarray(got, dtype=np.float64)
    aw = np.abs(want)
    half_ulp = np.where(aw > 0, 2.0 ** (np.floor(np.log2(np.where(aw > 0, aw, 1.0))) - 8), 0.0)
    bound = half_ulp + 1e-6
    bad = np.abs(got - want) > bound
    assert not bad.any(), f"{what}: {int(bad.sum())} elements beyond half a bf16 ulp, worst {np.abs(got - want).max():.3e}"


@pytest.mark.parametrize("rows,cols", [(1, 8), (4, 512), (5, 1000), (3, 4096), (3, 8192), (2, 8200), (3, 7)])
def test_ra_softmax_bf16_matches_oracle(rows, cols):
    x = softmax_inputs(rows, cols, seed=rows * 11 + cols, sigma=4.0).to(torch.bfloat16)
    got = ra.ra_softmax(x.cuda())
    torch.cuda.synchronize()
    assert got.dtype == torch.bfloat16
    want, *_ = oracle.ra_softmax(x.double().numpy())
    _assert_bf16_rounding_of(parity.f64(got), want, f"ra_softmax bf16 [{rows}x{cols}]")


def test_ra_softmax_bf16_in_place_and_misaligned():
    x = softmax_inputs(3, 4096, seed=21, sigma=4.0).to(torch.bfloat16)
    want, *_ = oracle.ra_softmax(x.double().numpy())
    xg = x.cuda()
    lib = ra.lib()
    code = lib.ra_softmax_fwd(ctypes.c_void_p(xg.data_ptr()), ctypes.c_void_p(xg.data_ptr()), 3, 4096, 1,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    torch.cuda.synchronize()
    _assert_bf16_rounding_of(parity.f64(xg), want, "ra_softmax bf16 in place")
    # rows 2 bytes off a 16-byte boundary take the generic kernel
    buf = softmax_inputs(1, 4 * 64 + 1, seed=22, sigma=3.0).to(torch.bfloat16).cuda()
    view = buf[0, 1:].reshape(4, 64)
    out = torch.empty((4, 64), dtype=torch.bfloat16, device="cuda")
    code = lib.ra_softmax_fwd(ctypes.c_void_p(view.data_ptr()), ctypes.c_void_p(out.data_ptr()), 4, 64, 1,
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 0
    torch.cuda.synchronize()
    want2, *_ = oracle.ra_softmax(view.double().cpu().numpy())
    _assert_bf16_rounding_of(parity.f64(out), want2, "ra_softmax bf16 offset rows")


def test_ra_softmax_bf16_full_workload_sampled_rows():
    """The bench's [16384, 8192] workload in bf16: every row through the kernel, 64 sampled
    rows against the oracle."""
    w = RA_SOFTMAX_LONG_ROWS
    x = softmax_inputs(w.rows, w.cols, seed=w.seed, sigma=w.sigma).to(torch.bfloat16)
    got = ra.ra_softmax(x.cuda())
    torch.cuda.synchronize()
    rows = np.random.default_rng(0).choice(w.rows, size=64, replace=False)
    want, *_ = oracle.ra_softmax(x[rows].double().numpy())
    _assert_bf16_rounding_of(parity.f64(got[rows]), want, "ra_softmax bf16 full workload")


def _bwd_bf16_bound(x, p, dy, want):
    """Error bound for the bf16 backward fed p_hat = bf16(p), p the float64 probabilities.

    With |p_hat - p| <= 2^-9 p (round to nearest, 8 significant bits), D_hat = sum p_hat dy
    is within eD = 2^-9 sum_k p_k |dy_k| of D, and an entry e_j = r_j (dy_j - D) with
    r_j = p_j / (1 - u_j^2) (live entries, u_j < 1) moves by at most
      b_j = 2^-9 r_j |dy_j - D| + (1 + 2^-9) r_j eD;
    the argmax entry (minus the sum of the others) by the sum of the others' b_j.  On top: the
    fp32 arithmetic (2e-5, the fp32 backward's bound) and half a bf16 ulp of the result."""
    m = x.max(axis=-1, keepdims=True)
    u = (m - x) / 16.0
    live = u < 1.0
    r = np.where(live, p / np.where(live, 1.0 - u * u, 1.0), 0.0)
    D = (p * dy).sum(axis=-1, keepdims=True)
    eD = 2.0 ** -9 * (p * np.abs(dy)).sum(axis=-1, keepdims=True)
    b = 2.0 ** -9 * r * np.abs(dy - D) + (1 + 2.0 ** -9) * r * eD
    a = x.argmax(axis=-1)   # lowest index of the maximum
    rows = np.arange(x.shape[0])
    b[rows, a] = b.sum(axis=-1) - b[rows, a]
    mag = np.abs(want) + b
    half_ulp = np.where(mag > 0, 2.0 ** (np.floor(np.log2(np.where(mag > 0, mag, 1.0))) - 8), 0.0)
    return b + half_ulp + 2e-5


@pytest.mark.parametrize("rows,cols", [(1, 8), (3, 5), (4, 512), (5, 1000), (3, 2048), (2, 4096), (3, 8192),
                                       (2, 16384), (2, 8200)])
def test_ra_softmax_backward_bf16_matches_oracle(rows, cols):
    """bf16 x, p and dy (p the float64 probabilities rounded once to bf16, as a bf16 forward
    would save them), fp32 arithmetic, dx rounded once: within the propagated bound of the
    float64 gradient.  Rows of up to 16384 columns in multiples of 8 take the register-held
    kernel; 5 columns (and the misaligned rows of the next test) the generic one."""
    g = torch.Generator().manual_seed(cols + 7)
    x = (torch.randn(rows, cols, generator=g) * 4.0).to(torch.bfloat16)
    dy = torch.randn(rows, cols, generator=g).to(torch.bfloat16)
    xd, dyd = x.double().numpy(), dy.double().numpy()
    p64, *_ = oracle.ra_softmax(xd)
    p = torch.from_numpy(p64).to(torch.bfloat16)
    dx = ra.ra_softmax_backward(x.cuda(), p.cuda(), dy.cuda())
    torch.cuda.synchronize()
    assert dx.dtype == torch.bfloat16 and ra.device_status() == "RA_OK"
    want = oracle.ra_softmax_bwd(xd, dyd)
    bound = _bwd_bf16_bound(xd, p64, dyd, want)
    err = np.abs(parity.f64(dx) - want)
    assert np.all(err <= bound), f"bf16 ra_softmax_bwd [{rows}x{cols}]: {int((err > bound).sum())} beyond the bound"


def test_ra_softmax_backward_bf16_ties_in_place_and_misaligned():
    """Exact maxima twice in a row (the gradient of the maximum goes to the lowest column),
    dx written over dy, and rows 2 bytes off a 16-byte boundary (the generic kernel)."""
    g = torch.Generator().manual_seed(12)
    rows, cols = 4, 8192
    x = (torch.randn(rows, cols, generator=g) * 4.0).to(torch.bfloat16)
    for r, (c1, c2) in enumerate([(5, 4000), (4000, 5), (1023, 1024), (8190, 8191)]):
        top = float(x[r].float().max()) + 1.0
        x[r, c1] = top
        x[r, c2] = top
    dy = torch.randn(rows, cols, generator=g).to(torch.bfloat16)
    xd, dyd = x.double().numpy(), dy.double().numpy()
    p64, *_ = oracle.ra_softmax(xd)
    dyg = dy.cuda()
    dx = ra.ra_softmax_backward(x.cuda(), torch.from_numpy(p64).to(torch.bfloat16).cuda(), dyg, out=dyg)
    torch.cuda.synchronize()
    assert dx.data_ptr() == dyg.data_ptr()
    want = oracle.ra_softmax_bwd(xd, dyd)
    assert np.all(np.abs(parity.f64(dx) - want) <= _bwd_bf16_bound(xd, p64, dyd, want))
    # misaligned rows: a view one element into a flat buffer
    n = 3 * 64
    buf = [(torch.randn(n + 1, generator=g) * s).to(torch.bfloat16) for s in (4.0, 1.0)]
    xv, dyv = (b[1:].reshape(3, 64) for b in buf)
    xd, dyd = xv.double().numpy(), dyv.double().numpy()
    p64, *_ = oracle.ra_softmax(xd)
    pbuf = torch.zeros(n + 1, dtype=torch.bfloat16)
    pbuf[1:] = torch.from_numpy(p64.reshape(-1)).to(torch.bfloat16)
    xg, dyg, pg = (b.cuda()[1:].reshape(3, 64) for b in (buf[0], buf[1], pbuf))
    dx = ra.ra_softmax_backward(xg, pg, dyg)
    torch.cuda.synchronize()
    want = oracle.ra_softmax_bwd(xd, dyd)
    assert np.all(np.abs(parity.f64(dx) - want) <= _bwd_bf16_bound(xd, p64, dyd, want))
