"""float32 <-> bfloat16 conversions of the oracle.

bfloat16 keeps the sign, the 8 exponent bits and the top 7 fraction bits of
an IEEE-754 binary32 value.  The method stores parameters and gradients in
16 bits ([Core flow] §1 table: parameters and gradients in fp16, optimizer
state in fp32; the workloads use bfloat16).

f32_to_bf16 rounds to nearest, ties to even, from the IEEE-754 definition:
the result is one of the two bf16 neighbours of x (the truncation t, or the
next value away from zero t+1 in bit terms); the discarded 16 bits r decide:
r > 0x8000 rounds away, r < 0x8000 truncates, r == 0x8000 picks the even
one.  Stepping t+1 past the largest finite value yields infinity, as the
definition requires.  A NaN stays a NaN (quiet bit set).
"""
from __future__ import annotations

import numpy as np


def bf16_to_f32(u16) -> np.ndarray:
    """Exact widening: the bf16 bits become the upper half of a float32."""
    u = np.asarray(u16, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def f32_to_bf16(x) -> np.ndarray:
    """Round float32 values to bfloat16 bit patterns (uint16), nearest-even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    t = u >> np.uint32(16)                 # truncated bf16 bits
    r = u & np.uint32(0xFFFF)              # discarded bits
    half = np.uint32(0x8000)
    up = (r > half) | ((r == half) & ((t & np.uint32(1)) == np.uint32(1)))
    out = np.where(up, t + np.uint32(1), t)
    nan = np.isnan(x)
    out = np.where(nan, (u >> np.uint32(16)) | np.uint32(0x0040), out)
    return out.astype(np.uint16)
