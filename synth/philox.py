"""Philox4x32-10 and the value mappings of the synthetic inputs (numpy).

Philox4x32-10 is written from its published definition (Salmon, Moraes, Dror,
Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11): a 4x32-bit
counter and a 2x32-bit key, ten rounds of two 32x32->64 multiplies
(multipliers 0xD2511F53, 0xCD9E8D57) with the key bumped by the Weyl
constants 0x9E3779B9, 0xBB67AE85 between rounds.

Counter layout used everywhere in this project:
    ctr = (index & 0xffffffff, index >> 32, sub, stream),  key = (seed lo, seed hi)
`index` is the element index of the value drawn, `sub` a sub-stream id (0 in
all workloads) and `stream` one of the STREAM_* tags below.

Value mappings (identical in synth/csrc/synth_gen.cu):
  normal  : the 8 16-bit halves h_i of one Philox output are summed exactly
            (Irwin-Hall of 8), z = 2*sum - 8*65535 is an exact integer in
            [-524280, 524280], and the value is float32(z) * c with
            c = float32(sigma / (65536 * sqrt(8/3))), one round-to-nearest
            multiply.  Mean 0, standard deviation ~sigma.
  outlier : a second Philox output (stream STREAM_OUTLIER) whose first word
            is below floor(frac * 2^32) marks the element; its value is then
            multiplied by float32(scale).
  bf16    : gradients are stored as bfloat16 by keeping the upper 16 bits of
            the float32 value (truncation; a generator convention, chosen so
            that no rounding rule of the method is involved in making inputs).
  fp16    : fp16 gradients are floor(z / 512) * 2^e (an integer of at most
            11 bits times a power of two: exactly representable in binary16,
            so again no rounding is involved); outliers multiply by 2^o.
"""
from __future__ import annotations

import math

import numpy as np

STREAM_GRAD = 1
STREAM_OUTLIER = 2
STREAM_WEIGHT = 3
STREAM_SHAPE = 4

_M0 = np.uint64(0xD2511F53)
_M1 = np.uint64(0xCD9E8D57)
_W0 = 0x9E3779B9
_W1 = 0xBB67AE85
_LO = np.uint64(0xFFFFFFFF)
_SH = np.uint64(32)


def philox4x32_10(c0, c1, c2, c3, k0: int, k1: int):
    """Ten Philox rounds on uint32 counter arrays; returns four uint32 arrays."""
    c0 = np.asarray(c0, dtype=np.uint32)
    c1 = np.asarray(c1, dtype=np.uint32)
    c2 = np.asarray(c2, dtype=np.uint32)
    c3 = np.asarray(c3, dtype=np.uint32)
    k0 = int(k0) & 0xFFFFFFFF
    k1 = int(k1) & 0xFFFFFFFF
    for _ in range(10):
        p0 = c0.astype(np.uint64) * _M0
        p1 = c2.astype(np.uint64) * _M1
        hi0 = (p0 >> _SH).astype(np.uint32)
        lo0 = (p0 & _LO).astype(np.uint32)
        hi1 = (p1 >> _SH).astype(np.uint32)
        lo1 = (p1 & _LO).astype(np.uint32)
        c0, c1, c2, c3 = (hi1 ^ c1 ^ np.uint32(k0), lo1,
                          hi0 ^ c3 ^ np.uint32(k1), lo0)
        k0 = (k0 + _W0) & 0xFFFFFFFF
        k1 = (k1 + _W1) & 0xFFFFFFFF
    return c0, c1, c2, c3


def _words(seed: int, stream: int, sub: int, idx):
    idx = np.asarray(idx, dtype=np.uint64)
    lo = (idx & _LO).astype(np.uint32)
    hi = (idx >> _SH).astype(np.uint32)
    return philox4x32_10(lo, hi,
                         np.full(idx.shape, sub, dtype=np.uint32),
                         np.full(idx.shape, stream, dtype=np.uint32),
                         seed & 0xFFFFFFFF, (seed >> 32) & 0xFFFFFFFF)


def normal_scale(sigma: float) -> np.float32:
    """The float32 constant c of the normal mapping for a target sigma."""
    return np.float32(sigma / (65536.0 * math.sqrt(8.0 / 3.0)))


def outlier_threshold(frac: float) -> int:
    return int(math.floor(frac * 4294967296.0))


def normal_f32(seed: int, stream: int, sub: int, idx, sigma: float) -> np.ndarray:
    """Approximately N(0, sigma^2) float32 values at element indices `idx`."""
    w = _words(seed, stream, sub, idx)
    s = np.zeros(np.shape(idx), dtype=np.int64)
    for x in w:
        x = x.astype(np.int64)
        s += (x & 0xFFFF) + (x >> 16)
    z = (2 * s - 8 * 65535).astype(np.float32)
    return z * normal_scale(sigma)


def grad_bf16(seed: int, sub: int, idx, sigma: float,
              outlier_frac: float = 0.0, outlier_scale: float = 100.0) -> np.ndarray:
    """Gradient values as raw bfloat16 bit patterns (uint16) at indices `idx`."""
    v = normal_f32(seed, STREAM_GRAD, sub, idx, sigma)
    if outlier_frac > 0.0:
        u = _words(seed, STREAM_OUTLIER, sub, idx)[0]
        hit = u < np.uint32(outlier_threshold(outlier_frac))
        v = np.where(hit, v * np.float32(outlier_scale), v).astype(np.float32)
    return (v.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def weight_f32(seed: int, idx, sigma: float) -> np.ndarray:
    """Initial full-parameter values (float32) at model-flat indices `idx`."""
    return normal_f32(seed, STREAM_WEIGHT, 0, idx, sigma)


def uniform_u32(seed: int, stream: int, sub: int, idx) -> np.ndarray:
    """First Philox output word at indices `idx` (uniform on [0, 2^32))."""
    return _words(seed, stream, sub, idx)[0]


def grad_fp16(seed: int, sub: int, idx, log2_scale: int, outlier_frac: float = 0.0,
              outlier_log2: int = 0) -> np.ndarray:
    """fp16 gradient values as raw binary16 bit patterns (uint16): the
    Irwin-Hall integer z of the normal mapping, floor(z / 512) in
    [-1024, 1023], times 2^log2_scale (times 2^outlier_log2 for outliers;
    large outliers overflow to inf on purpose)."""
    w = _words(seed, STREAM_GRAD, sub, idx)
    s = np.zeros(np.shape(idx), dtype=np.int64)
    for x in w:
        x = x.astype(np.int64)
        s += (x & 0xFFFF) + (x >> 16)
    k = (2 * s - 8 * 65535) // 512
    e = np.full(np.shape(idx), log2_scale, dtype=np.int64)
    if outlier_frac > 0.0:
        u = _words(seed, STREAM_OUTLIER, sub, idx)[0]
        e = np.where(u < np.uint32(outlier_threshold(outlier_frac)), e + outlier_log2, e)
    v = np.ldexp(k.astype(np.float32), e.astype(np.int32)).astype(np.float32)
    with np.errstate(over="ignore"):
        return v.astype(np.float16).view(np.uint16)
