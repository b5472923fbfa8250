"""Test-harness helpers: input layouts built from the oracle's plan.

Rank k's gradient buffer of a reduce bucket holds, for each bucket entry
(param, e_lo, e_hi, buf_off), the elements e_lo..e_hi-1 of that rank's full
gradient of the parameter at buf_off.  The helpers below place synthetic
values into that layout; the arithmetic of the step stays in `oracle`.
"""
from __future__ import annotations

import numpy as np

from oracle import plan as oplan
from synth import philox


def full_grads_from_pool(plan, seed, sigma, n_ranks, outlier_frac=0.0):
    """Per-rank full gradients (uint16, model input layout), rank k's drawn
    at pool indices k*input_elems + i."""
    n = plan.input_elems
    G = []
    for k in range(n_ranks):
        idx = np.arange(k * n, (k + 1) * n, dtype=np.uint64)
        G.append(philox.grad_bf16(seed, 0, idx, sigma, outlier_frac))
    return G


def bucket_buffers(plan, G):
    """bufs[b][k]: rank k's gradient buffer of bucket b from full gradients
    G[k] (uint16, model input layout).  Gap elements between entries are
    filled with a NaN pattern, which must never be read."""
    out = []
    for b, ents in enumerate(plan.reduce_buckets):
        L = plan.bucket_buf_elems[b]
        row = []
        for k in range(plan.n_ranks):
            buf = np.full(L, 0x7FC1, dtype=np.uint16)
            for e in ents:
                p = plan.params[e.param]
                n = e.e_hi - e.e_lo
                buf[e.buf_off:e.buf_off + n] = G[k][p.input_off + e.e_lo:p.input_off + e.e_hi]
            row.append(buf)
        out.append(row)
    return out


def random_numels(rng, n, lo=0, hi=300):
    return [int(x) for x in rng.integers(lo, hi + 1, size=n)]


def build(numel, N, **kw):
    return oplan.build_partition(numel, N, **kw)
