"""float32 <-> IEEE binary16 conversions of the oracle (fp16 mode).

The pages' accounting stores parameters and gradients in fp16 ([Core flow]
§1 table); the fp16 mode of the step keeps them as binary16 bit patterns
(uint16).  Widening is exact; narrowing rounds to nearest, ties to even,
with overflow to infinity (numpy's float16 cast, an IEEE conversion)."""
from __future__ import annotations

import numpy as np


def fp16_to_f32(u16) -> np.ndarray:
    return np.ascontiguousarray(u16, dtype=np.uint16).view(np.float16).astype(np.float32)


def f32_to_fp16(x) -> np.ndarray:
    with np.errstate(over="ignore"):
        return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)
