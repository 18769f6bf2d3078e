"""The tolerance of the bf16 ra_softmax backward test is neither vacuous nor too tight.

A float32 emulation of the bf16 path (p rounded to bf16, fp32 arithmetic, dx rounded once)
stays inside the bound derived in test_gpu_softmax._bwd_bf16_bound on random rows; the same
emulation with a plausible mistake (the (1 - u^2) factor dropped, the argmax correction
dropped, D taken from dy alone) leaves it.  No GPU: everything here runs on the host."""
import sys
import os

import numpy as np
import pytest
import torch

import oracle

sys.path.insert(0, os.path.dirname(__file__))
from test_gpu_softmax import _bwd_bf16_bound  # noqa: E402


def _bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16).double().numpy()


def _emulate(x, p_hat, dy, mistake=None):
    x32, p32, g32 = (a.astype(np.float32) for a in (x, p_hat, dy))
    m = x32.max(axis=-1, keepdims=True)
    a = x32.argmax(axis=-1)
    d = (p32 * g32).sum(axis=-1, keepdims=True, dtype=np.float32)
    if mistake == "no_D":
        d = np.zeros_like(d)
    delta = m - x32
    den = (16.0 - delta) * (16.0 + delta) / np.float32(256.0)
    if mistake == "no_denominator":
        den = np.ones_like(den)
    e = np.where(delta < 16.0, p32 * (g32 - d) / np.where(delta < 16.0, den, 1.0), 0.0).astype(np.float32)
    rows = np.arange(x.shape[0])
    e[rows, a] = 0.0
    r = e.sum(axis=-1, dtype=np.float32)
    if mistake != "no_argmax":
        e[rows, a] = -r
    return _bf16(e)


def _case(seed, rows=6, cols=2048):
    rng = np.random.default_rng(seed)
    x = _bf16(rng.standard_normal((rows, cols)) * 4.0)
    dy = _bf16(rng.standard_normal((rows, cols)))
    p64, *_ = oracle.ra_softmax(x)
    return x, dy, p64, _bf16(p64)


@pytest.mark.parametrize("seed", range(4))
def test_emulated_bf16_path_stays_inside_the_bound(seed):
    x, dy, p64, p_hat = _case(seed)
    want = oracle.ra_softmax_bwd(x, dy)
    assert np.all(np.abs(_emulate(x, p_hat, dy) - want) <= _bwd_bf16_bound(x, p64, dy, want))


@pytest.mark.parametrize("mistake", ["no_denominator", "no_argmax", "no_D"])
def test_plausible_mistakes_leave_the_bound(mistake):
    x, dy, p64, p_hat = _case(7)
    want = oracle.ra_softmax_bwd(x, dy)
    assert np.any(np.abs(_emulate(x, p_hat, dy, mistake) - want) > _bwd_bf16_bound(x, p64, dy, want))
