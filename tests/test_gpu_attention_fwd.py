"""GPU parity of ra_attention_fwd against the float64 oracle.

bf16 inputs run on the tensor-core path (D in {64, 128}) and must match the oracle,
evaluated on the same bf16-rounded inputs, within max-abs 1e-2 and mean-abs 1e-3;
fp32 inputs run on the CUDA-core path and must match within max-abs 2e-5.
Sizes span several 128 x 128 tiles with ragged tails; the full-size workloads are
checked on sampled heads and rows that the oracle computes one by one, plus
properties that hold everywhere.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import rational_softmax_attention_gb300 as ra
from rational_softmax_attention_gb300.inputs import (ATTN_LONG_CAUSAL, ATTN_LONG_WIDE, ATTN_MODULE_SHAPE,
                                                     ATTN_TINY_FP32, attention_inputs, workload_inputs)

pytestmark = pytest.mark.gpu


def gpu_fwd(q, k, v, scale, causal, out_dtype=torch.float32):
    o, rm, rs, ra_, counts = ra.ra_attention_forward(q.cuda(), k.cuda(), v.cuda(), scale=scale, causal=causal,
                                                     out_dtype=out_dtype, tile_counts=True)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    return o, rm, rs, ra_, counts


def check_head(o, rm, rs, ra_, q, k, v, scale, causal, rows, bf16, b, h):
    """Compare one head's outputs at the given rows with the oracle's row-by-row forward."""
    qh, kh, vh = (t[b, h].double().numpy() for t in (q, k, v))
    O, _, s, _ = oracle.ra_attention_rows_fwd(qh, kh, vh, rows, scale, causal)
    got = parity.f64(o[b, h])[rows]
    if bf16:
        parity.assert_close_bf16(got, O, f"O[{b},{h}]")
    else:
        parity.assert_close_fp32(got, O, f"O[{b},{h}]")
    np.testing.assert_allclose(parity.f64(rs[b, h])[rows], s, rtol=2e-3 if bf16 else 1e-5)
    S = scale * (qh[rows] @ kh.T)
    if causal:
        S = np.where(np.arange(kh.shape[0])[None, :] <= rows[:, None], S, -np.inf)
    # the row max within the fp32 score-error bound; the argmax equal to the oracle's except
    # at near ties within twice that bound
    err = parity.score_error_bound(qh[rows], kh, scale)
    parity.check_argmax(S, ra_[b, h].cpu().numpy()[rows], err, f"forward O[{b},{h}] {tuple(q.shape)}",
                        m_gpu=parity.f64(rm[b, h])[rows])


def check_all(q, k, v, scale, causal, out_dtype=torch.float32):
    o, rm, rs, ra_, counts = gpu_fwd(q, k, v, scale, causal, out_dtype)
    bf16 = q.dtype == torch.bfloat16
    B, H, NQ, _ = q.shape
    rows = np.arange(NQ)
    for b in range(B):
        for h in range(H):
            check_head(o, rm, rs, ra_, q, k, v, scale, causal, rows, bf16, b, h)
    return o, rm, rs, ra_, counts


def test_tiny_fp32_workload():
    w = ATTN_TINY_FP32
    q, k, v = workload_inputs(w)
    check_all(q, k, v, w.scale, w.causal)


@pytest.mark.parametrize("D", [16, 32, 64, 128])
@pytest.mark.parametrize("nq,nk", [(1, 1), (17, 17), (33, 100), (100, 33), (130, 130)])
@pytest.mark.parametrize("causal", [False, True])
def test_fp32_path_ragged(D, nq, nk, causal):
    q, k, v = attention_inputs(1, 2, nq, nk, D, seed=nq + nk + D, sigma_qk=1.5, dtype=torch.float32,
                               with_dout=False)
    check_all(q, k, v, D ** -0.5, causal)


@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("nq,nk", [(1, 1), (17, 17), (128, 128), (129, 129), (300, 300), (513, 513),
                                   (64, 200), (200, 64), (256, 1)])
@pytest.mark.parametrize("causal", [False, True])
def test_bf16_tensor_core_path_ragged(D, nq, nk, causal):
    q, k, v = attention_inputs(1, 2, nq, nk, D, seed=3 * nq + nk + D, sigma_qk=1.0, dtype=torch.bfloat16,
                               with_dout=False)
    check_all(q, k, v, D ** -0.5, causal)


@pytest.mark.parametrize("sigma", [0.3, 3.0, 6.0])
def test_bf16_score_spreads(sigma):
    # from nearly uniform weights to almost one-hot rows (most entries past the support)
    q, k, v = attention_inputs(1, 2, 384, 384, 128, seed=int(10 * sigma), sigma_qk=sigma, dtype=torch.bfloat16,
                               with_dout=False)
    check_all(q, k, v, 128 ** -0.5, False)


def test_module_shape_workload_forward():
    w = ATTN_MODULE_SHAPE
    q, k, v, _ = workload_inputs(w)
    check_all(q, k, v, w.scale, w.causal, out_dtype=torch.float32)
    o16, *_ = gpu_fwd(q, k, v, w.scale, w.causal, out_dtype=torch.bfloat16)
    o32, *_ = gpu_fwd(q, k, v, w.scale, w.causal, out_dtype=torch.float32)
    # bf16 output is the fp32 output rounded once
    assert torch.equal(o16, o32.to(torch.bfloat16))


def _sampled_full_size(w, out_dtype):
    q, k, v = workload_inputs(w)[:3]
    o, rm, rs, ra_, counts = gpu_fwd(q, k, v, w.scale, w.causal, out_dtype)
    assert torch.isfinite(o).all()
    assert (rs >= 1.0 - 1e-5).all()                       # sum(phi) >= 1
    if w.causal:
        assert (ra_ <= torch.arange(w.N, device=ra_.device, dtype=torch.int32)).all()
    rng = np.random.default_rng(0)
    rows = np.unique(np.concatenate([[0, 1, 127, 128, w.N - 1], rng.choice(w.N, 96, replace=False)]))
    for b, h in ((0, 0), (w.B - 1, w.H - 1), (1, 7)):
        check_head(o, rm, rs, ra_, q, k, v, w.scale, w.causal, rows, True, b, h)
    return counts


def test_long_causal_workload_sampled():
    counts = _sampled_full_size(ATTN_LONG_CAUSAL, torch.float32)
    nqt = ATTN_LONG_CAUSAL.N // 128
    assert int(counts[0]) == ATTN_LONG_CAUSAL.B * ATTN_LONG_CAUSAL.H * nqt * (nqt + 1) // 2


def test_long_wide_workload_forward_sampled():
    counts = _sampled_full_size(ATTN_LONG_WIDE, torch.float32)
    nqt = ATTN_LONG_WIDE.N // 128
    assert int(counts[0]) == ATTN_LONG_WIDE.B * ATTN_LONG_WIDE.H * nqt * nqt
    assert 0 <= int(counts[1]) <= int(counts[0])


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_single_key_gives_V(dtype):
    D = 64
    q, k, v = attention_inputs(2, 3, 150, 1, D, seed=5, dtype=dtype, with_dout=False)
    o, *_ = gpu_fwd(q, k, v, 0.2, False)
    want = v.float().expand(2, 3, 150, D)
    if dtype == torch.float32:
        assert torch.equal(o.cpu(), want)          # phi_max = 1 exactly on the fp32 path
    else:
        # tensor-core path: phi_max comes from an approximate reciprocal (a few ulp), and
        # q ~ 1 raised to the 8th power multiplies that by 8, so phi_max = 1 to ~2e-6
        torch.testing.assert_close(o.cpu(), want, rtol=1e-5, atol=0)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16])
def test_causal_first_row_and_causality_probe(dtype):
    D = 64
    q, k, v = attention_inputs(1, 2, 300, 300, D, seed=6, dtype=dtype, with_dout=False)
    o1, *_ = gpu_fwd(q, k, v, 0.2, True)
    if dtype == torch.float32:
        assert torch.equal(o1[:, :, 0].cpu(), v[:, :, 0].float())
    else:
        torch.testing.assert_close(o1[:, :, 0].cpu(), v[:, :, 0].float(), rtol=1e-5, atol=0)
    t = 140
    k2, v2 = k.clone(), v.clone()
    k2[:, :, t + 1:] = k2[:, :, t + 1:] * -2
    v2[:, :, t + 1:] = v2[:, :, t + 1:] + 3
    o2, *_ = gpu_fwd(q, k2, v2, 0.2, True)
    assert torch.equal(o1[:, :, :t + 1], o2[:, :, :t + 1])
    assert (o1[:, :, t + 1:] - o2[:, :, t + 1:]).abs().max() > 0.1


def test_dead_tiles_are_skipped_and_counted():
    # keys 0..127 align with every query; keys 128.. are pushed far below the support,
    # so every (query tile, key tile >= 1) pair has all u >= 1
    D, N = 128, 512
    q, k, v = attention_inputs(1, 1, N, N, D, seed=8, dtype=torch.float32, with_dout=False)
    base = torch.ones(D) / np.sqrt(D)
    q = (q * 0.1 + 4.0 * base).to(torch.bfloat16)
    kk = k * 0.1
    kk[:, :, :128] += 4.0 * base
    kk[:, :, 128:] -= 4.0 * base
    k = kk.to(torch.bfloat16)
    v = v.to(torch.bfloat16)
    o, rm, rs, ra_, counts = check_all(q, k, v, 1.0, False)
    assert int(counts[0]) == 4 * 4 and int(counts[1]) == 4 * 3


@pytest.mark.parametrize("nq,nk,causal", [(128, 128, False), (300, 300, True), (513, 700, False), (1000, 1000, True),
                                          (700, 513, True)])
def test_cta_pair_and_single_cta_layouts_agree(nq, nk, causal):
    """The D = 128 forward as clusters of two CTAs (products spanning both SMs) and as
    single CTAs: both against the oracle, and against each other to fp32 rounding."""
    q, k, v = attention_inputs(2, 2, nq, nk, 128, seed=nq + 7 * nk, sigma_qk=1.0, dtype=torch.bfloat16,
                               with_dout=False)
    outs = {}
    try:
        for mode in (1, 2):
            ra.debug_fwd_pair(mode)
            outs[mode] = check_all(q, k, v, 128 ** -0.5, causal)
    finally:
        ra.debug_fwd_pair(0)
    single, pair = outs[1], outs[2]
    assert torch.equal(single[3], pair[3])                     # argmax
    for a, b in zip(single[:3], pair[:3]):                      # O, row max, row sum
        np.testing.assert_allclose(a.cpu().numpy(), b.cpu().numpy(), rtol=1e-5, atol=1e-6)
    assert torch.equal(single[4], pair[4])                     # visited / skipped tile pairs


@pytest.mark.parametrize("causal", [False, True])
def test_fp32_path_at_scale_sampled_rows(causal):
    """fp32 inputs at N = 4096, D = 128 (the CUDA-core path): 96 sampled rows of each head
    against the oracle within 2e-5, with the statistics and the argmax."""
    q, k, v = attention_inputs(1, 2, 4096, 4096, 128, seed=21 + int(causal), dtype=torch.float32, with_dout=False)
    o, rm, rs, ra_, _ = gpu_fwd(q, k, v, 128 ** -0.5, causal)
    rows = np.sort(np.random.default_rng(5).choice(4096, size=96, replace=False))
    rows[0], rows[-1] = 0, 4095
    for h in range(2):
        check_head(o, rm, rs, ra_, q, k, v, 128 ** -0.5, causal, rows, False, 0, h)
