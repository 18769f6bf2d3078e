"""Seeded random configurations of the attention forward and backward against the float64
oracle: sizes on both sides of the 128-row tile and of the CTA-pair threshold (N_Q > 256 at
D = 128), 1-row and 1-key cases, causal or not, fp32 or bf16 inputs, and for bf16 random,
block, key-padding and empty-row masks in every broadcast layout.  Tolerances are the other
parity tests' (bf16: max-abs 1e-2, mean-abs 1e-3; fp32: max-abs 2e-5) for outputs of unit
scale, as at the five workloads; some random shapes give much larger values (300 queries
sharing two keys put |dV| near 30, where fp16 P's 2^-11 rounding alone is ~5e-3), so here
the bounds scale with max(1, RMS of the oracle's output).  Argmax agreement by
parity.check_argmax, with the oracle's backward following the GPU's argmax where the two
differ within the fp32 score-error bound."""
import numpy as np
import pytest
import torch

import oracle
import parity
import rational_softmax_attention_gb300 as ra
from rational_softmax_attention_gb300.inputs import attention_inputs

pytestmark = pytest.mark.gpu

SIZES = [1, 2, 5, 17, 63, 64, 65, 127, 128, 129, 200, 255, 256, 257, 300, 383, 385, 511, 513]
N_CASES = 96


def _mask(rng, kind, B, H, nq, nk):
    layout = rng.choice(["shared", "per_batch", "per_head", "full"])
    shape = {"shared": (nq, nk), "per_batch": (B, 1, nq, nk), "per_head": (1, H, nq, nk),
             "full": (B, H, nq, nk)}[layout]
    lead = shape[:-2]
    if kind == "random":
        m = rng.random(shape) < rng.uniform(0.2, 0.8)
    elif kind == "blocks":
        nqt, nkt = -(-nq // 128), -(-nk // 128)
        blk = rng.integers(0, 3, size=lead + (nqt, nkt))   # 0 masked, 1 full, 2 half filled
        dense = np.repeat(np.repeat(blk, 128, axis=-2), 128, axis=-1)[..., :nq, :nk]
        m = (dense == 1) | ((dense == 2) & (rng.random(shape) < 0.5))
    elif kind == "keypad":
        lens = rng.integers(1, nk + 1, size=lead + (1, 1))
        m = np.broadcast_to(np.arange(nk) < lens, shape).copy()
    else:   # "rows": random, with some query rows allowed nothing
        m = rng.random(shape) < 0.6
        m[..., rng.random(nq) < 0.2, :] = False
    return m


def _case(i):
    rng = np.random.default_rng(7000 + i)
    fp32 = rng.random() < 0.25
    D = int(rng.choice([16, 32, 64, 128])) if fp32 else int(rng.choice([64, 128]))
    sizes = [n for n in SIZES if n <= 300] if fp32 else SIZES
    nq, nk = int(rng.choice(sizes)), int(rng.choice(sizes))
    B, H = int(rng.integers(1, 3)), int(rng.integers(1, 4))
    causal = bool(rng.random() < 0.5)
    sigma = float(rng.choice([0.5, 1.0])) if fp32 else float(rng.choice([0.5, 1.0, 3.0]))
    kind = None if fp32 or rng.random() < 0.3 else str(rng.choice(["random", "blocks", "keypad", "rows"]))
    mask = _mask(rng, kind, B, H, nq, nk) if kind else None
    bf16_out = (not fp32) and rng.random() < 0.3   # O and the gradients rounded to bf16 once
    return dict(fp32=fp32, D=D, nq=nq, nk=nk, B=B, H=H, causal=causal, sigma=sigma, kind=kind, mask=mask,
                bf16_out=bf16_out)


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_configuration_matches_oracle(i):
    c = _case(i)
    dtype = torch.float32 if c["fp32"] else torch.bfloat16
    B, H, nq, nk, D, causal = c["B"], c["H"], c["nq"], c["nk"], c["D"], c["causal"]
    scale = D ** -0.5
    what = (f"case {i}: {'fp32' if c['fp32'] else 'bf16'} B{B} H{H} {nq}x{nk} D{D} causal={causal} "
            f"mask={c['kind']} bf16_out={c['bf16_out']}")
    out_dt = torch.bfloat16 if c["bf16_out"] else torch.float32
    q, k, v, do = attention_inputs(B, H, nq, nk, D, seed=9000 + i, sigma_qk=c["sigma"], dtype=dtype)
    qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    pm = None
    full = np.ones((B, H, nq, nk), dtype=bool)
    if c["mask"] is not None:
        pm = ra.pack_attn_mask(torch.from_numpy(np.ascontiguousarray(c["mask"])).cuda(), B, H, nq, nk)
        m = c["mask"]
        while m.ndim < 4:
            m = m[None]
        full = np.broadcast_to(m, (B, H, nq, nk))
    o, rm, rs, ra_, _ = ra.ra_attention_forward(qg, kg, vg, scale=scale, causal=causal, out_dtype=out_dt,
                                                mask=pm)
    # the backward reads O for D_i = dO . O; it takes the fp32 O here, so that bf16 gradients
    # differ from the oracle's only by their own rounding (a bf16 O in D_i is covered by
    # test_bf16_autograd_function_bf16_gradients)
    o32 = o if out_dt == torch.float32 else ra.ra_attention_forward(qg, kg, vg, scale=scale, causal=causal,
                                                                     out_dtype=torch.float32, mask=pm)[0]
    dq, dk, dv = ra.ra_attention_backward(qg, kg, vg, o32, dog, rm, rs, ra_, scale=scale, causal=causal,
                                          grad_dtype=out_dt, mask=pm)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK", what
    def close(got, want, msg):
        sc = max(1.0, float(np.sqrt(np.mean(np.square(want)))) if want.size else 1.0)
        if c["bf16_out"]:   # the bounds plus one bf16 rounding of each value (half an ulp: 2^-9 relative)
            err = np.abs(np.asarray(got) - want)
            assert np.all(np.isfinite(got)), msg
            assert np.all(err <= parity.BF16_MAX_ABS * sc + 2.0 ** -8 * np.abs(want)), msg
            assert err.mean() <= parity.BF16_MEAN_ABS * sc + 2.0 ** -9 * np.abs(want).mean(), msg
        elif c["fp32"]:
            parity.assert_close_fp32(got, want, msg, max_abs=parity.FP32_MAX_ABS * sc)
        else:
            parity.assert_close_bf16(got, want, msg, max_abs=parity.BF16_MAX_ABS * sc, mean_abs=parity.BF16_MEAN_ABS * sc)
    tril = np.tril(np.ones((nq, nk), dtype=bool))
    for b in range(B):
        for h in range(H):
            qd, kd, vd, dod = (t[b, h].double().numpy() for t in (q, k, v, do))
            allowed = full[b, h] & (tril if causal else True)
            S = np.where(allowed, scale * (qd @ kd.T), -np.inf)
            a_gpu = ra_[b, h].cpu().numpy().astype(np.int64)
            nd = parity.check_argmax(S, a_gpu, parity.score_error_bound(qd, kd, scale), what,
                                     m_gpu=parity.f64(rm[b, h]))
            msk = None if c["mask"] is None else full[b, h]
            wo, _, ws, _ = oracle.ra_attention_head_fwd(qd, kd, vd, scale, causal, mask=msk)
            close(parity.f64(o[b, h]), wo, f"{what} O[{b},{h}]")
            np.testing.assert_array_equal(rs[b, h].cpu().numpy() == 0, ws == 0)   # rows with no allowed key
            gq, gk, gv = oracle.ra_attention_head_bwd(qd, kd, vd, dod, scale, causal, argmax=a_gpu if nd else None,
                                                      mask=msk)
            close(parity.f64(dq[b, h]), gq, f"{what} dq[{b},{h}]")
            close(parity.f64(dk[b, h]), gk, f"{what} dk[{b},{h}]")
            close(parity.f64(dv[b, h]), gv, f"{what} dv[{b},{h}]")


@pytest.mark.parametrize("i", range(48))
def test_random_softmax_rows_match_oracle(i):
    """ra_softmax forward and backward on seeded random shapes (both the register-held and
    the generic kernels: columns in and out of multiples of 4 and 8, up to 20000), fp32 and
    bf16, spread 0.5 to 8: fp32 within 2e-5; bf16 forward within half a bf16 ulp (+1e-6) and
    bf16 backward within the bound of test_gpu_softmax (p the float64 probabilities rounded
    to bf16)."""
    from test_gpu_softmax import _assert_bf16_rounding_of, _bwd_bf16_bound
    rng = np.random.default_rng(11000 + i)
    bf16 = bool(rng.random() < 0.5)
    rows = int(rng.integers(1, 7))
    cols = int(rng.choice([1, 2, 3, 7, 8, 31, 64, 100, 1000, 1024, 2050, 4096, 4100, 8192, 8200, 12288, 16384, 20000]))
    sigma = float(rng.choice([0.5, 2.0, 8.0]))
    x = torch.from_numpy(rng.standard_normal((rows, cols)) * sigma).float()
    dy = torch.from_numpy(rng.standard_normal((rows, cols))).float()
    if bf16:
        x, dy = x.to(torch.bfloat16), dy.to(torch.bfloat16)
    xd, dyd = x.double().numpy(), dy.double().numpy()
    want_p, *_ = oracle.ra_softmax(xd)
    want_dx = oracle.ra_softmax_bwd(xd, dyd)
    p = ra.ra_softmax(x.cuda())
    p_in = torch.from_numpy(want_p).to(x.dtype).cuda() if bf16 else p
    dx = ra.ra_softmax_backward(x.cuda(), p_in, dy.cuda())
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    what = f"softmax case {i}: {'bf16' if bf16 else 'fp32'} [{rows}x{cols}] sigma {sigma}"
    if bf16:
        _assert_bf16_rounding_of(parity.f64(p), want_p, what)
        err = np.abs(parity.f64(dx) - want_dx)
        assert np.all(err <= _bwd_bf16_bound(xd, want_p, dyd, want_dx)), what
    else:
        parity.assert_close_fp32(parity.f64(p), want_p, what)
        parity.assert_close_fp32(parity.f64(dx), want_dx, what + " bwd")
