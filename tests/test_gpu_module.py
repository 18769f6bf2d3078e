"""GPU parity of the RaAttention module against the float64 module oracle.

fp32 (attention on the CUDA-core path, projections in fp32 cuBLAS with TF32 off): the
oracle's bound for the attention (2e-5) widened by the fp32 GEMM rounding, 1e-4 max-abs.

bf16 (attention on the tensor-core path): every GEMM output (q, k, v, O and y) is rounded
to bf16 (relative 2^-9), against exact float64 in the oracle.  At this shape |y| stays
below ~4, so the final rounding alone is up to 2^-9 * 4 = 8e-3, and the rounded q, k, v
and O add errors of the same order: max-abs 3e-2, mean-abs 3e-3.
"""
import numpy as np
import pytest
import torch

import oracle
import parity
import rational_softmax_attention_gb300 as ra

pytestmark = pytest.mark.gpu


def _module(dim, heads, causal, dtype, qk_norm=False, qkv_bias=False, seed=0):
    torch.manual_seed(seed)
    m = ra.RaAttention(dim, num_heads=heads, qkv_bias=qkv_bias, qk_norm=qk_norm, causal=causal)
    if qk_norm:   # non-trivial normalisation parameters
        with torch.no_grad():
            for ln in (m.q_norm, m.k_norm):
                ln.weight.uniform_(0.5, 1.5)
                ln.bias.uniform_(-0.2, 0.2)
    return m.to(device="cuda", dtype=dtype)


def _f64(t):
    return None if t is None else t.detach().to("cpu", torch.float64).numpy()


def _oracle_fwd(m, x):
    qn = (_f64(m.q_norm.weight), _f64(m.q_norm.bias)) if m.q_norm is not None else None
    kn = (_f64(m.k_norm.weight), _f64(m.k_norm.bias)) if m.k_norm is not None else None
    return oracle.ra_attention_module_fwd(_f64(x), _f64(m.qkv.weight), _f64(m.qkv.bias), _f64(m.proj.weight),
                                          _f64(m.proj.bias), m.num_heads, causal=m.causal, q_norm=qn, k_norm=kn)


@pytest.fixture(autouse=True)
def _no_tf32():
    old = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = False
    yield
    torch.backends.cuda.matmul.allow_tf32 = old


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("qk_norm,qkv_bias", [(False, False), (True, True)])
def test_module_fp32_matches_oracle(causal, qk_norm, qkv_bias):
    m = _module(128, 4, causal, torch.float32, qk_norm=qk_norm, qkv_bias=qkv_bias, seed=1)
    x = torch.randn(2, 40, 128, generator=torch.Generator().manual_seed(2)).cuda()
    y = m(x)
    torch.cuda.synchronize()
    parity.assert_close_fp32(parity.f64(y), _oracle_fwd(m, x), "RaAttention fp32", max_abs=1e-4)


@pytest.mark.parametrize("qk_norm", [False, True])
def test_module_bf16_pages_shape_matches_oracle(qk_norm):
    """The page's example: dim 768, 12 heads, causal, x [2, 128, 768]."""
    m = _module(768, 12, True, torch.bfloat16, qk_norm=qk_norm, seed=3)
    x = torch.randn(2, 128, 768, generator=torch.Generator().manual_seed(4)).to("cuda", torch.bfloat16)
    y = m(x)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    parity.assert_close_bf16(parity.f64(y), _oracle_fwd(m, x), "RaAttention bf16", max_abs=3e-2, mean_abs=3e-3)


@pytest.mark.parametrize("causal", [False, True])
def test_module_fp32_backward_matches_oracle(causal):
    """Gradients of sum(dy * y) in x and in every weight and bias, against the oracle's
    closed-form module backward (no qk_norm)."""
    m = _module(64, 2, causal, torch.float32, qkv_bias=True, seed=5)
    g = torch.Generator().manual_seed(6)
    x = torch.randn(2, 33, 64, generator=g).cuda().requires_grad_(True)
    dy = torch.randn(2, 33, 64, generator=g)
    m(x).backward(dy.cuda())
    torch.cuda.synchronize()
    want = oracle.ra_attention_module_bwd(_f64(x), _f64(m.qkv.weight), _f64(m.qkv.bias), _f64(m.proj.weight),
                                          _f64(m.proj.bias), m.num_heads, dy.double().numpy(), causal=causal)
    got = [x.grad, m.qkv.weight.grad, m.qkv.bias.grad, m.proj.weight.grad, m.proj.bias.grad]
    for name, gv, wv in zip(["dx", "dW_qkv", "db_qkv", "dW_proj", "db_proj"], got, want):
        parity.assert_close_fp32(parity.f64(gv), wv, f"RaAttention backward {name}", max_abs=1e-4)


def test_module_rejects_dropout():
    with pytest.raises(NotImplementedError):
        ra.RaAttention(64, num_heads=2, proj_drop=0.1)
