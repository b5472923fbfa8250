"""Device-side fills with the same values as synth.philox (libzs_synth.so)."""
from __future__ import annotations

import ctypes as C
import os

from . import philox

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libzs_synth.so")
_lib = None


def _load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"{LIB_PATH} is missing: run the build first")
        lib = C.CDLL(LIB_PATH)
        lib.zsg_fill_grad_bf16.restype = C.c_int
        lib.zsg_fill_grad_bf16.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_uint64,
                                           C.c_uint32, C.c_float, C.c_uint32, C.c_float,
                                           C.c_void_p]
        lib.zsg_fill_grad_fp16.restype = C.c_int
        lib.zsg_fill_grad_fp16.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_uint64,
                                           C.c_uint32, C.c_int, C.c_uint32, C.c_int, C.c_void_p]
        lib.zsg_busy.restype = C.c_int
        lib.zsg_busy.argtypes = [C.c_int64, C.c_int, C.c_int, C.c_void_p, C.c_void_p]
        lib.zsg_fill_normal_f32.restype = C.c_int
        lib.zsg_fill_normal_f32.argtypes = [C.c_void_p, C.c_int64, C.c_int64, C.c_uint64,
                                            C.c_uint32, C.c_uint32, C.c_float, C.c_void_p]
        _lib = lib
    return _lib


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def fill_grad_bf16(t, start: int, seed: int, sigma: float, outlier_frac: float = 0.0,
                   outlier_scale: float = 100.0, sub: int = 0, stream=None) -> None:
    """t (2-byte CUDA tensor)[i] = philox.grad_bf16(seed, sub, start + i, ...)."""
    thr = philox.outlier_threshold(outlier_frac) if outlier_frac > 0 else 0
    err = _load().zsg_fill_grad_bf16(t.data_ptr(), int(start), t.numel(), int(seed), sub,
                                     float(philox.normal_scale(sigma)), thr, float(outlier_scale),
                                     _stream(stream))
    if err:
        raise RuntimeError(f"zsg_fill_grad_bf16: CUDA error {err}")


def fill_weight_f32(t, start: int, seed: int, sigma: float, stream=None) -> None:
    """t (float32 CUDA tensor)[i] = philox.weight_f32(seed, start + i, sigma)."""
    err = _load().zsg_fill_normal_f32(t.data_ptr(), int(start), t.numel(), int(seed), 0,
                                      philox.STREAM_WEIGHT, float(philox.normal_scale(sigma)),
                                      _stream(stream))
    if err:
        raise RuntimeError(f"zsg_fill_normal_f32: CUDA error {err}")


def fill_grad_fp16(t, start: int, seed: int, log2_scale: int, outlier_frac: float = 0.0,
                   outlier_log2: int = 0, sub: int = 0, stream=None) -> None:
    """t (2-byte CUDA tensor)[i] = philox.grad_fp16(seed, sub, start + i, ...)."""
    thr = philox.outlier_threshold(outlier_frac) if outlier_frac > 0 else 0
    err = _load().zsg_fill_grad_fp16(t.data_ptr(), int(start), t.numel(), int(seed), sub,
                                     int(log2_scale), thr, int(outlier_log2), _stream(stream))
    if err:
        raise RuntimeError(f"zsg_fill_grad_fp16: CUDA error {err}")


def busy(iters: int, blocks: int, sink, stream=None, threads: int = 256) -> None:
    """Stand-in compute: `blocks` CTAs of `threads` threads, `iters` FMAs each."""
    err = _load().zsg_busy(int(iters), int(blocks), int(threads), sink.data_ptr(),
                           _stream(stream))
    if err:
        raise RuntimeError(f"zsg_busy: CUDA error {err}")
