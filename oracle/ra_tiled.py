"""Tiled two-pass float64 CPU restatement of ra_attention, written separately.

TEST INFRASTRUCTURE, NOT PRODUCT CODE (same import rule as ra_oracle.py).

Page "Ra-Family: Rational Neural Architecture", section 3, ra_attention:
the result is computed "without materializing the [B, H, N_Q, N_K] attention
matrix", by a "2-pass" tiled kernel.  Because phi depends on the row maximum
in a way that does not factor (phi(Delta + c) is not phi(Delta) times a
function of c), the first pass can only find the row maximum; the second pass
evaluates phi tile by tile and accumulates sum(phi) and phi V.

This file shares no code with ra_oracle.py on purpose: the test that compares
the two (materialised against tiled) is a pin on both.  Pure-Python tile loops:
small inputs only.
"""
from __future__ import annotations

import math

import numpy as np


def _phi_scalar(delta):
    # Compact-support Cayley weight: ((16 - Delta)/(16 + Delta))^8 for Delta < 16,
    # which equals ((1-u)/(1+u))^8 with u = Delta/16; exactly 0 beyond.
    if delta >= 16.0:
        return 0.0
    return ((16.0 - delta) / (16.0 + delta)) ** 8


def ra_attention_tiled_head(q, k, v, scale, causal, bm=4, bn=4):
    """One head, query tiles of bm rows, key tiles of bn columns, two sweeps per query tile."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n_q, n_k = q.shape[0], k.shape[0]
    out = np.zeros((n_q, v.shape[1]))
    row_max = np.zeros(n_q)
    row_sum = np.zeros(n_q)
    row_arg = np.full(n_q, -1, dtype=np.int64)
    for i0 in range(0, n_q, bm):
        i1 = min(i0 + bm, n_q)
        # sweep 1: running maximum (strictly greater updates keep the lowest index)
        best = [-math.inf] * (i1 - i0)
        arg = [-1] * (i1 - i0)
        for j0 in range(0, n_k, bn):
            j1 = min(j0 + bn, n_k)
            tile = scale * (q[i0:i1] @ k[j0:j1].T)
            for r in range(i1 - i0):
                for c in range(j1 - j0):
                    if causal and (j0 + c) > (i0 + r):
                        continue
                    if tile[r, c] > best[r]:
                        best[r] = tile[r, c]
                        arg[r] = j0 + c
        # sweep 2: phi, running sum and phi-weighted values
        acc = np.zeros((i1 - i0, v.shape[1]))
        tot = [0.0] * (i1 - i0)
        for j0 in range(0, n_k, bn):
            j1 = min(j0 + bn, n_k)
            tile = scale * (q[i0:i1] @ k[j0:j1].T)
            w = np.zeros((i1 - i0, j1 - j0))
            for r in range(i1 - i0):
                if arg[r] < 0:
                    continue
                for c in range(j1 - j0):
                    if causal and (j0 + c) > (i0 + r):
                        continue
                    w[r, c] = _phi_scalar(best[r] - tile[r, c])
                    tot[r] += w[r, c]
            if not w.any():
                continue  # every entry outside the support: the V tile is not needed
            acc += w @ v[j0:j1]
        for r in range(i1 - i0):
            if arg[r] >= 0:
                out[i0 + r] = acc[r] / tot[r]
                row_max[i0 + r] = best[r]
                row_sum[i0 + r] = tot[r]
                row_arg[i0 + r] = arg[r]
    return out, row_max, row_sum, row_arg
