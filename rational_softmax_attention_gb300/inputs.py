"""Seeded synthetic inputs shared by the tests, the smoke check and the benchmark.

This module holds random draws and shapes only -- none of the method's
arithmetic -- so that the CUDA path and the float64 oracle can be fed the very
same (already rounded) values without either importing the other.

Recipe: one CPU torch.Generator seeded with `seed`; torch.randn draws in the
order Q, K, V, dO (attention) or x (ra_softmax), in float32, each multiplied by
its standard deviation, then cast to the stated dtype.  The oracle reads the
rounded values converted to float64.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch


def attention_inputs(B, H, N_Q, N_K, D, *, seed, sigma_qk=1.0, sigma_v=1.0, sigma_do=1.0,
                     dtype=torch.bfloat16, with_dout=True):
    """Q, K [B,H,N,D] ~ N(0, sigma_qk^2); V ~ N(0, sigma_v^2); dO ~ N(0, sigma_do^2)."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    q = torch.randn((B, H, N_Q, D), generator=g, dtype=torch.float32) * sigma_qk
    k = torch.randn((B, H, N_K, D), generator=g, dtype=torch.float32) * sigma_qk
    v = torch.randn((B, H, N_K, D), generator=g, dtype=torch.float32) * sigma_v
    out = [q.to(dtype), k.to(dtype), v.to(dtype)]
    if with_dout:
        do = torch.randn((B, H, N_Q, D), generator=g, dtype=torch.float32) * sigma_do
        out.append(do.to(dtype))
    return tuple(out)


def softmax_inputs(rows, cols, *, seed, sigma=1.0, dtype=torch.float32):
    """Logits x [rows, cols] ~ N(0, sigma^2)."""
    g = torch.Generator("cpu").manual_seed(int(seed))
    x = torch.randn((rows, cols), generator=g, dtype=torch.float32) * sigma
    return x.to(dtype)


@dataclass(frozen=True)
class AttentionWorkload:
    name: str
    B: int
    H: int
    N: int
    D: int
    dtype: torch.dtype
    sigma_qk: float
    scale: float
    causal: bool
    backward: bool
    seed: int = 0


@dataclass(frozen=True)
class SoftmaxWorkload:
    name: str
    rows: int
    cols: int
    sigma: float
    seed: int = 1


# The five workloads the library is specified and measured on.
ATTN_TINY_FP32 = AttentionWorkload("attn_fwd_fp32_b1h2n128d64", 1, 2, 128, 64, torch.float32,
                                   1.0, 1.0 / 8.0, False, False)
RA_SOFTMAX_LONG_ROWS = SoftmaxWorkload("ra_softmax_fp32_16384x8192", 16384, 8192, 4.0)
ATTN_MODULE_SHAPE = AttentionWorkload("attn_fwdbwd_bf16_b2h12n128d64_causal", 2, 12, 128, 64,
                                      torch.bfloat16, 1.0, 1.0 / 8.0, True, True)
ATTN_LONG_CAUSAL = AttentionWorkload("attn_fwd_bf16_b4h16n8192d128_causal", 4, 16, 8192, 128,
                                     torch.bfloat16, 1.0, 128 ** -0.5, True, False)
ATTN_LONG_WIDE = AttentionWorkload("attn_fwdbwd_bf16_b4h16n8192d128_sigma3", 4, 16, 8192, 128,
                                   torch.bfloat16, 3.0, 128 ** -0.5, False, True)

WORKLOADS = {w.name: w for w in (ATTN_TINY_FP32, RA_SOFTMAX_LONG_ROWS, ATTN_MODULE_SHAPE,
                                 ATTN_LONG_CAUSAL, ATTN_LONG_WIDE)}


def workload_inputs(w: AttentionWorkload):
    """Q, K, V (and dO when the workload has a backward) of an attention workload."""
    return attention_inputs(w.B, w.H, w.N, w.N, w.D, seed=w.seed, sigma_qk=w.sigma_qk,
                            dtype=w.dtype, with_dout=w.backward)
