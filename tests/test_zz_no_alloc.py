"""The scratch-free backward entry point, checked against the allocating one.

ra_attention_bwd_noalloc is for callers that cannot allocate device memory (their
framework owns the allocator, or cudaMalloc is not allowed on their path); it takes its
workspace from a fixed array inside the library.  Here it is called through the C ABI
twice in a row on the same inputs and must agree with ra_attention_bwd (given a
torch-allocated workspace) within the tolerance of the other backward tests: the bf16
bounds for bf16 inputs, 2e-5 for fp32 inputs.
This file is collected last so that a failure here comes after every other test.
"""
import ctypes

import pytest
import torch

import parity
import rational_softmax_attention_gb300 as ra
from rational_softmax_attention_gb300.inputs import ATTN_MODULE_SHAPE, attention_inputs, workload_inputs

pytestmark = pytest.mark.gpu


def _noalloc_fn():
    L = ra.lib()
    fn = L.ra_attention_bwd_noalloc
    vp, i32, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn.argtypes = [vp] * 11 + [i32, i32, i32, i32, i32, f32, i32, i32, i32, i32, vp]
    fn.restype = i32
    return fn


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("case", ["module_shape", "ragged", "fp32_ragged"])
def test_noalloc_backward_matches_the_allocating_entry_point(case):
    if case == "module_shape":
        w = ATTN_MODULE_SHAPE
        q, k, v, do = workload_inputs(w)
        scale, causal = w.scale, w.causal
    elif case == "ragged":
        q, k, v, do = attention_inputs(1, 3, 200, 300, 128, seed=9, sigma_qk=2.0)
        scale, causal = 128 ** -0.5, False
    else:   # fp32 inputs: the CUDA-core backward, whose per-row arrays come from the same array
        q, k, v, do = attention_inputs(2, 2, 150, 190, 64, seed=10, dtype=torch.float32)
        scale, causal = 0.125, True
    f32 = q.dtype == torch.float32
    qg, kg, vg, dog = q.cuda(), k.cuda(), v.cuda(), do.cuda()
    o, rm, rs, ra_, _ = ra.ra_attention_forward(qg, kg, vg, scale=scale, causal=causal, out_dtype=torch.float32)
    ref = ra.ra_attention_backward(qg, kg, vg, o, dog, rm, rs, ra_, scale=scale, causal=causal)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    fn = _noalloc_fn()
    B, H, NQ, D = q.shape
    NK = k.shape[2]
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        dq, dk, dv = (torch.full_like(r, float("nan")) for r in ref)
        code = fn(_p(qg), _p(kg), _p(vg), _p(o), _p(dog), _p(rm), _p(rs), _p(ra_), _p(dq), _p(dk), _p(dv),
                  B, H, NQ, NK, D, scale, 1 if causal else 0, 0 if f32 else 1, 0, 0, st)
        assert code == 0, ra.lib().ra_status_string(code)
        torch.cuda.synchronize()
        assert ra.device_status() == "RA_OK"
        for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
            if f32:
                parity.assert_close_fp32(parity.f64(got), parity.f64(want), f"{name} (call {call + 1})")
            else:
                parity.assert_close_bf16(parity.f64(got), parity.f64(want), f"{name} (call {call + 1})")


def test_noalloc_rejects_sizes_beyond_its_scratch():
    fn = _noalloc_fn()
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: the size check comes first
    code = fn(*([fake] * 11), 64, 64, 8192, 8192, 128, 0.0, 0, 1, 0, 0, ctypes.c_void_p(0))
    assert code == 2   # RA_ERR_UNSUPPORTED: the fixed scratch is too small for these sizes


def test_noalloc_fp32_inputs_count_only_their_own_workspace():
    """fp32 inputs use the CUDA-core backward, whose workspace is two per-row float arrays
    (256 KB here), so sizes whose bf16 workspace would not fit the array still run."""
    B, H, N, D = 1, 8, 4096, 128
    assert ra.lib().ra_attention_bwd_workspace_size(B, H, N, N, D) > (32 << 20)
    q, k, v, do = (t.cuda() for t in attention_inputs(B, H, N, N, D, seed=12, dtype=torch.float32))
    o, rm, rs, ra_, _ = ra.ra_attention_forward(q, k, v, out_dtype=torch.float32)
    ref = ra.ra_attention_backward(q, k, v, o, do, rm, rs, ra_)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    dq, dk, dv = (torch.full_like(r, float("nan")) for r in ref)
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    code = _noalloc_fn()(_p(q), _p(k), _p(v), _p(o), _p(do), _p(rm), _p(rs), _p(ra_), _p(dq), _p(dk), _p(dv),
                         B, H, N, N, D, 0.0, 0, 0, 0, 0, st)
    assert code == 0, ra.lib().ra_status_string(code)
    torch.cuda.synchronize()
    assert ra.device_status() == "RA_OK"
    for name, got, want in (("dq", dq, ref[0]), ("dk", dk, ref[1]), ("dv", dv, ref[2])):
        parity.assert_close_fp32(parity.f64(got), parity.f64(want), name)
