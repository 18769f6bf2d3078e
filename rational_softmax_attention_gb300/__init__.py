"""Python binding of libraattn: rational-softmax (Ra-family) attention on GB300.

Argument marshalling only.  Every computation runs in the CUDA kernels of
libraattn.so, reached through its C ABI (include/raattn.h) with ctypes; torch
provides device memory and the current stream.  There is no CPU path: when the
library is not built, or the tensors are not on a CUDA device, the calls raise.

Functional API, after the page "Ra-Family: Rational Neural Architecture",
section 3 "Rational Attention & Softmax":
    ra_softmax(x)                                   last-dim rational soft-argmax
    ra_attention(q, k, v, attn_mask=None, is_causal=False, scale=None)   drop-in for SDPA, autograd-aware
plus the explicit forward/backward entry points used by tests and benchmarks.
"""
from __future__ import annotations

import ctypes
import os
import re

import torch

__all__ = [
    "RaError", "lib", "ra_softmax", "ra_softmax_backward", "ra_attention", "ra_attention_forward", "RaAttention",
    "ra_attention_backward", "pack_attn_mask", "device_status", "set_wait_limit_ns", "exported_symbols", "LIB_PATH",
    "debug_kernel_events",
]

PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG_DIR, "libraattn.so")
HEADER_PATH = os.path.join(os.path.dirname(PKG_DIR), "include", "raattn.h")

RA_F32, RA_BF16 = 0, 1
_STATUS = {0: "RA_OK", 1: "RA_ERR_ARG", 2: "RA_ERR_UNSUPPORTED", 3: "RA_ERR_LAUNCH", 4: "RA_ERR_TIMEOUT"}


class RaError(RuntimeError):
    """A libraattn call returned a status other than RA_OK."""

    def __init__(self, fn, code, text):
        super().__init__(f"{fn}: {text} (status {code})")
        self.code = code


_lib = None
_vp, _i64, _i32, _f32, _u64 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float, ctypes.c_uint64

_SIGNATURES = {
    "ra_status_string": ([_i32], ctypes.c_char_p),
    "ra_softmax_fwd": ([_vp, _vp, _i64, _i64, _i32, _vp], _i32),
    "ra_softmax_bwd": ([_vp, _vp, _vp, _vp, _i64, _i64, _i32, _vp], _i32),
    "ra_attention_fwd": ([_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _f32, _i32,
                          _i32, _i32, _vp], _i32),
    "ra_attention_fwd_workspace_size": ([_i32, _i32, _i32, _i32, _i32], ctypes.c_size_t),
    "ra_attention_bwd_workspace_size": ([_i32, _i32, _i32, _i32, _i32], ctypes.c_size_t),
    "ra_attention_bwd": ([_vp] * 12 + [_i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _i32, _i32, _vp], _i32),
    "ra_attention_mask_words": ([_i32], _i32),
    "ra_attention_mask_pack": ([_vp, _i32, _i32, _i32, _vp, _vp, _vp], _i32),
    "ra_attention_fwd_masked": ([_vp] * 9 + [_i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _i32, _vp, _i32, _i32,
                                               _vp], _i32),
    "ra_attention_bwd_masked": ([_vp] * 12 + [_i32, _i32, _i32, _i32, _i32, _f32, _i32, _i32, _i32, _i32, _vp, _vp,
                                                _i32, _i32, _vp], _i32),
    "ra_device_status": ([_vp], _i32),
    "ra_set_wait_limit_ns": ([_u64], None),
    "ra_debug_force_timeout": ([_i32], None),
    "ra_debug_fwd_pair": ([_i32], None),
    "ra_debug_kernel_events": ([ctypes.POINTER(ctypes.c_void_p), _i32], None),
}


def lib():
    """The loaded libraattn (ctypes.CDLL).  Raises if the library has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libraattn.so is not built ({LIB_PATH}); run "
                               "`python -m rational_softmax_attention_gb300.build`")
        handle = ctypes.CDLL(LIB_PATH)
        for name, (args, res) in _SIGNATURES.items():
            fn = getattr(handle, name)
            fn.argtypes = args
            fn.restype = res
        _lib = handle
    return _lib


def exported_symbols():
    """Names of the functions include/raattn.h declares."""
    with open(HEADER_PATH) as f:
        text = f.read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w]*\**\s+\**(ra_\w+)\s*\(", text, re.M)))


def _check(fn, code):
    if code != 0:
        raise RaError(fn, code, lib().ra_status_string(code).decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device):
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _dtype_code(dt):
    if dt == torch.float32:
        return RA_F32
    if dt == torch.bfloat16:
        return RA_BF16
    raise TypeError(f"unsupported dtype {dt}: libraattn takes float32 or bfloat16")


def _require_cuda(*ts):
    for t in ts:
        if t is not None and (not t.is_cuda or not t.is_contiguous()):
            raise ValueError("libraattn takes contiguous CUDA tensors (there is no CPU path)")


def ra_softmax(x):
    """ra_softmax along the last dimension of a float32 or bfloat16 CUDA tensor (same dtype out)."""
    _require_cuda(x)
    y = torch.empty_like(x)
    cols = x.shape[-1]
    rows = x.numel() // cols if cols else 0
    _check("ra_softmax_fwd", lib().ra_softmax_fwd(_ptr(x), _ptr(y), rows, cols, _dtype_code(x.dtype),
                                                   _stream(x.device)))
    return y


def ra_softmax_backward(x, p, dy, out=None):
    """Closed-form gradient of sum(dy * ra_softmax(x)) with respect to x (last dimension).

    out: optional tensor for dx, shaped like x; it may be dy itself (gradient in place)."""
    _require_cuda(x, p, dy)
    if p.dtype != x.dtype or dy.dtype != x.dtype or p.shape != x.shape or dy.shape != x.shape:
        raise ValueError("x, p and dy must share one shape and dtype (float32 or bfloat16)")
    if out is not None:
        _require_cuda(out)
        if out.shape != x.shape or out.dtype != x.dtype or not out.is_contiguous():
            raise ValueError("out must be a contiguous tensor shaped like x")
    dx = torch.empty_like(x) if out is None else out
    cols = x.shape[-1]
    rows = x.numel() // cols
    _check("ra_softmax_bwd", lib().ra_softmax_bwd(_ptr(x), _ptr(p), _ptr(dy), _ptr(dx), rows, cols,
                                                   _dtype_code(x.dtype), _stream(x.device)))
    return dx


def pack_attn_mask(attn_mask, B, H, n_q, n_k):
    """Bit-packs a boolean attn_mask broadcastable to [B, H, N_Q, N_K] (True = the query may
    attend to the key, as in scaled_dot_product_attention) for the masked attention calls.

    Returns (mask_q, mask_k, MB, MH): the packed mask with a row per query and with a row
    per key, and how many batch and head entries it has (1 = shared)."""
    if attn_mask.dtype != torch.bool:
        raise NotImplementedError("only boolean attention masks are supported")
    _require_cuda(attn_mask.contiguous())
    m = attn_mask
    while m.dim() < 4:
        m = m.unsqueeze(0)
    if m.dim() != 4:
        raise ValueError("attn_mask must broadcast to [B, H, N_Q, N_K]")
    MB, MH = m.shape[0], m.shape[1]
    if MB not in (1, B) or MH not in (1, H):
        raise ValueError("attn_mask must broadcast to [B, H, N_Q, N_K]")
    m8 = m.expand(MB, MH, n_q, n_k).contiguous().view(torch.uint8)
    L = lib()
    mask_q = torch.empty((MB * MH, n_q, L.ra_attention_mask_words(n_k)), dtype=torch.int32, device=m.device)
    mask_k = torch.empty((MB * MH, n_k, L.ra_attention_mask_words(n_q)), dtype=torch.int32, device=m.device)
    _check("ra_attention_mask_pack", L.ra_attention_mask_pack(_ptr(m8), MB * MH, n_q, n_k, _ptr(mask_q),
                                                                _ptr(mask_k), _stream(m.device)))
    return mask_q, mask_k, MB, MH


def ra_attention_forward(q, k, v, *, scale=None, causal=False, out_dtype=None, with_stats=True,
                         tile_counts=False, mask=None):
    """O = ra_softmax(scale q k^T [causal] [mask]) v for [B, H, N, D] tensors.

    mask: None, or the tuple pack_attn_mask returns (bf16 inputs only).
    Returns (o, row_m, row_s, row_arg, counts): the statistics are None unless
    with_stats; counts is an int64 CUDA tensor [pairs visited, pairs skipped]
    when tile_counts, else None.
    """
    _require_cuda(q, k, v)
    B, H, NQ, D = q.shape
    NK = k.shape[2]
    out_dtype = out_dtype or q.dtype
    o = torch.empty((B, H, NQ, D), dtype=out_dtype, device=q.device)
    stats = None
    if with_stats:
        stats = (torch.empty((B, H, NQ), dtype=torch.float32, device=q.device),
                 torch.empty((B, H, NQ), dtype=torch.float32, device=q.device),
                 torch.empty((B, H, NQ), dtype=torch.int32, device=q.device))
    counts = torch.empty(2, dtype=torch.int64, device=q.device) if tile_counts else None
    rm, rs, ra = stats if stats else (None, None, None)
    L = lib()
    ws = None
    if q.dtype == torch.bfloat16:
        ws = torch.empty(L.ra_attention_fwd_workspace_size(B, H, NQ, NK, D), dtype=torch.uint8, device=q.device)
    if mask is None:
        _check("ra_attention_fwd", L.ra_attention_fwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(rm), _ptr(rs), _ptr(ra), _ptr(counts), _ptr(ws),
            B, H, NQ, NK, D, float(scale or 0.0), 1 if causal else 0, _dtype_code(q.dtype), _dtype_code(out_dtype),
            _stream(q.device)))
    else:
        mask_q, _, MB, MH = mask
        _check("ra_attention_fwd_masked", L.ra_attention_fwd_masked(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(rm), _ptr(rs), _ptr(ra), _ptr(counts), _ptr(ws),
            B, H, NQ, NK, D, float(scale or 0.0), 1 if causal else 0, _dtype_code(q.dtype), _dtype_code(out_dtype),
            _ptr(mask_q), MB, MH, _stream(q.device)))
    return o, rm, rs, ra, counts


def ra_attention_backward(q, k, v, o, dout, row_m, row_s, row_arg, *, scale=None, causal=False,
                          grad_dtype=torch.float32, workspace=None, mask=None):
    """Gradients (dq, dk, dv) of sum(dout * O) for the forward that produced o and the row
    statistics; mask as given to that forward."""
    _require_cuda(q, k, v, o, dout, row_m, row_s, row_arg)
    B, H, NQ, D = q.shape
    NK = k.shape[2]
    L = lib()
    if workspace is None:
        nbytes = L.ra_attention_bwd_workspace_size(B, H, NQ, NK, D)
        workspace = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=q.device)
    dq = torch.empty((B, H, NQ, D), dtype=grad_dtype, device=q.device)
    dk = torch.empty((B, H, NK, D), dtype=grad_dtype, device=q.device)
    dv = torch.empty((B, H, NK, D), dtype=grad_dtype, device=q.device)
    if mask is None:
        _check("ra_attention_bwd", L.ra_attention_bwd(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(row_m), _ptr(row_s), _ptr(row_arg),
            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), B, H, NQ, NK, D, float(scale or 0.0),
            1 if causal else 0, _dtype_code(q.dtype), _dtype_code(o.dtype), _dtype_code(grad_dtype),
            _stream(q.device)))
    else:
        mask_q, mask_k, MB, MH = mask
        _check("ra_attention_bwd_masked", L.ra_attention_bwd_masked(
            _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(dout), _ptr(row_m), _ptr(row_s), _ptr(row_arg),
            _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace), B, H, NQ, NK, D, float(scale or 0.0),
            1 if causal else 0, _dtype_code(q.dtype), _dtype_code(o.dtype), _dtype_code(grad_dtype),
            _ptr(mask_q), _ptr(mask_k), MB, MH, _stream(q.device)))
    return dq, dk, dv


class _RaAttentionFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale, attn_mask):
        mask = None
        if attn_mask is not None:
            mask = pack_attn_mask(attn_mask, q.shape[0], q.shape[1], q.shape[2], k.shape[2])
        o, rm, rs, ra, _ = ra_attention_forward(q, k, v, scale=scale, causal=causal, out_dtype=q.dtype, mask=mask)
        ctx.save_for_backward(q, k, v, o, rm, rs, ra)
        ctx.causal, ctx.scale, ctx.mask = causal, scale, mask
        return o

    @staticmethod
    def backward(ctx, do):
        q, k, v, o, rm, rs, ra = ctx.saved_tensors
        dq, dk, dv = ra_attention_backward(q, k, v, o, do.contiguous().to(q.dtype), rm, rs, ra,
                                           scale=ctx.scale, causal=ctx.causal, grad_dtype=q.dtype, mask=ctx.mask)
        return dq, dk, dv, None, None, None


def ra_attention(q, k, v, attn_mask=None, is_causal=False, scale=None):
    """Rational-softmax attention, a drop-in for scaled_dot_product_attention (no dropout).

    attn_mask: optional boolean mask broadcastable to [B, H, N_Q, N_K], True where the query
    may attend to the key (bf16 inputs only); combined with is_causal."""
    return _RaAttentionFn.apply(q.contiguous(), k.contiguous(), v.contiguous(), bool(is_causal), scale, attn_mask)


class RaAttention(torch.nn.Module):
    """Multi-head attention with ra_softmax (page "Ra-Family: Rational Neural Architecture",
    section 3, "ra_attention & RaAttention").

    x [B, N, dim] -> one projection to q, k, v of every head ([B, heads, N, dim/heads])
    -> optional layer normalisation of q and k over the head dimension (qk_norm)
    -> ra_attention (this library's kernels, with autograd) -> heads merged -> output
    projection.  The two projections are plain library GEMMs (torch Linear, cuBLAS).
    Dropout is not part of this path: attn_drop and proj_drop must be 0.
    """

    def __init__(self, dim, num_heads=8, qkv_bias=False, qk_norm=False, attn_drop=0.0, proj_drop=0.0,
                 causal=False, device=None, dtype=None):
        super().__init__()
        if dim % num_heads != 0:
            raise ValueError("dim must be a multiple of num_heads")
        if attn_drop != 0.0 or proj_drop != 0.0:
            raise NotImplementedError("dropout is not supported (attn_drop and proj_drop must be 0)")
        self.num_heads = num_heads
        self.head_dim = dim // num_heads
        self.causal = bool(causal)
        kw = {"device": device, "dtype": dtype}
        self.qkv = torch.nn.Linear(dim, 3 * dim, bias=qkv_bias, **kw)
        self.q_norm = torch.nn.LayerNorm(self.head_dim, eps=1e-5, **kw) if qk_norm else None
        self.k_norm = torch.nn.LayerNorm(self.head_dim, eps=1e-5, **kw) if qk_norm else None
        self.proj = torch.nn.Linear(dim, dim, **kw)

    def forward(self, x):
        B, N, C = x.shape
        q, k, v = self.qkv(x).reshape(B, N, 3, self.num_heads, self.head_dim).permute(2, 0, 3, 1, 4).unbind(0)
        if self.q_norm is not None:
            q, k = self.q_norm(q), self.k_norm(k)
        o = ra_attention(q, k, v, is_causal=self.causal)
        return self.proj(o.transpose(1, 2).reshape(B, N, C))


def device_status(stream=None):
    """Synchronise and return the device-side status name ('RA_OK', 'RA_ERR_TIMEOUT', ...), clearing it."""
    s = stream if stream is not None else torch.cuda.current_stream()
    return _STATUS.get(lib().ra_device_status(ctypes.c_void_p(s.cuda_stream)), "unknown")


def set_wait_limit_ns(ns):
    """Limit on every device-side wait of later launches (0 restores the 2 s default)."""
    lib().ra_set_wait_limit_ns(int(ns))


def debug_force_timeout(on):
    """Test knob: make later tensor-core launches take their timeout and wind-down path."""
    lib().ra_debug_force_timeout(1 if on else 0)


def debug_fwd_pair(mode):
    """Layout of later bf16 D = 128 forward calls: 0 automatic (CTA pairs when N_Q > 256),
    1 single CTAs, 2 CTA pairs."""
    lib().ra_debug_fwd_pair(int(mode))


def debug_kernel_events(events):
    """Measurement knob: later bf16 attention calls record these torch.cuda.Event objects
    (up to four, created with enable_timing=True) at their kernel boundaries; None turns it
    off.  Forward: [before the V conversion, before the attention kernel, after it];
    backward: [before the conversion, before dQ, before dK/dV, after dK/dV]."""
    if not events:
        lib().ra_debug_kernel_events(None, 0)
        return
    stream = torch.cuda.current_stream()
    handles = []
    for e in events:
        if e.cuda_event == 0:      # torch creates the CUDA event on its first record
            e.record(stream)
        handles.append(e.cuda_event)
    arr = (ctypes.c_void_p * len(handles))(*handles)
    lib().ra_debug_kernel_events(arr, len(handles))
