"""Python binding of libzs (include/zs.h): the ZeRO-3 per-step shard data
path on one GB300, N virtual ranks in one HBM.

Argument marshalling only.  Every step of the path runs in libzs's CUDA
kernels; this module converts Python values (ints, torch tensors, streams)
to the C arguments and raises ZsError on a non-zero status.  Importing it
fails loudly when libzs.so is missing: there is no fallback.

Functions keep the C names: zs_build_partition, zs_plan_upload,
zs_partition, zs_reduce_scatter, zs_grad_norm, zs_adam_step,
zs_all_gather_coalesced, zs_shard_step, plus the plan queries.
"""
from __future__ import annotations

import ctypes as C
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libzs.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build it first "
        "(python -c 'import __graft_entry__ as g; g.build()'); libzs has no CPU fallback")
_lib = C.CDLL(LIB_PATH)

ZS_OK, ZS_EINVAL, ZS_ENOMEM, ZS_ECUDA, ZS_ESTATE, ZS_ETIMEOUT = 0, -1, -2, -3, -4, -5
ZS_MAX_RANKS = 256
ZS_SKIP_NONFINITE = 1
ZS_DTYPE_BF16, ZS_DTYPE_FP16 = 0, 1
ZS_NOALLOC_NORM_MAX_SCRATCH = 1 << 20
TILE_DTYPE = [("dst", "<i8"), ("src", "<i8"), ("flat", "<i8"), ("win", "<i8"),
              ("len", "<i4"), ("valid", "<i4"), ("flat_len", "<i4"), ("bucket", "<i4")]


class ZsError(RuntimeError):
    def __init__(self, status: int, fn: str, msg: str):
        super().__init__(f"{fn} failed ({status}): {msg}")
        self.status = status


class zs_config(C.Structure):
    _fields_ = [("n_ranks", C.c_int32), ("dtype", C.c_int32),
                ("param_persistence_threshold", C.c_int64), ("reduce_bucket_size", C.c_int64),
                ("prefetch_bucket_size", C.c_int64), ("sub_group_size", C.c_int64),
                ("shard_group_size", C.c_int32), ("reserved", C.c_int32)]


class zs_adam_hparams(C.Structure):
    _fields_ = [("lr", C.c_float), ("beta1", C.c_float), ("beta2", C.c_float),
                ("eps", C.c_float), ("weight_decay", C.c_float), ("adamw", C.c_int32),
                ("bias_correction", C.c_int32)]


class zs_plan_info_t(C.Structure):
    _fields_ = [(n, C.c_int32) for n in ("n_ranks", "n_params", "n_reduce_buckets",
                                         "n_gather_buckets", "n_sub_groups", "dtype",
                                         "shard_group_size", "reserved")] + \
               [(n, C.c_int64) for n in ("psi", "shard_elems", "shard_elems_logical",
                                         "persist_elems", "persist_elems_logical", "flat_elems",
                                         "padding_elems", "max_bucket_buf_elems",
                                         "max_gather_elems", "bytes_per_rank", "n_tiles",
                                         "device_table_bytes", "norm_scratch_elems")]


class zs_param_info_t(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("numel", "ds_id", "partition_size", "padding",
                                         "shard_offset", "persist_offset", "flat_offset",
                                         "input_offset")] + \
               [(n, C.c_int32) for n in ("persistent", "position", "sub_group", "gather_bucket",
                                         "first_reduce_bucket", "n_reduce_buckets")]


class zs_bucket_info_t(C.Structure):
    _fields_ = [("n_entries", C.c_int32), ("reserved", C.c_int32), ("buf_elems", C.c_int64),
                ("grad_elems", C.c_int64), ("first_tile", C.c_int64), ("n_tiles", C.c_int64)]


class zs_gather_bucket_info_t(C.Structure):
    _fields_ = [("n_params", C.c_int32), ("reserved", C.c_int32), ("flat_offset", C.c_int64),
                ("flat_elems", C.c_int64)]


class zs_sub_group_info_t(C.Structure):
    _fields_ = [("n_params", C.c_int32), ("reserved", C.c_int32), ("shard_lo", C.c_int64),
                ("shard_hi", C.c_int64), ("persist_lo", C.c_int64), ("persist_hi", C.c_int64)]


class zs_loss_scaler(C.Structure):
    _fields_ = [("d_scale", C.c_void_p), ("d_good_steps", C.c_void_p), ("scale_factor", C.c_float),
                ("min_scale", C.c_float), ("scale_window", C.c_int32), ("reserved", C.c_int32)]


class zs_shard_state(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in ("grad_shards", "param_shards", "master", "exp_avg",
                                          "exp_avg_sq", "persist_grads", "persist_params",
                                          "p_master", "p_exp_avg", "p_exp_avg_sq")]


class zs_sched_config(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("prefetch_bucket_size", "max_live_parameters",
                                         "max_reuse_distance", "arena_elems",
                                         "gather_ctas", "log_limit")]


class zs_sched_stats_t(C.Structure):
    _fields_ = [(n, C.c_int64) for n in ("passes", "gathers", "params_gathered", "elems_gathered",
                                         "elems_prefetched", "fetch_misses", "max_live_elems",
                                         "max_arena_elems", "invalidations")]


class zs_sched_event(C.Structure):
    _fields_ = [("kind", C.c_int32), ("module_pos", C.c_int32), ("op", C.c_int32),
                ("param", C.c_int32), ("offset", C.c_int64), ("aux", C.c_int64)]


_P = C.c_void_p
_i32, _i64, _f32 = C.c_int32, C.c_int64, C.c_float


def _sig(name, res, args):
    f = getattr(_lib, name)
    f.restype = res
    f.argtypes = args
    return f


_sig("zs_last_error", C.c_char_p, [])
_sig("zs_version", C.c_char_p, [])
_sig("zs_default_config", None, [C.POINTER(zs_config), _i32])
_sig("zs_build_partition", _i32, [C.POINTER(zs_config), _i32, C.POINTER(_i64), C.POINTER(_i64),
                                  C.POINTER(_P)])
_sig("zs_free_plan", None, [_P])
_sig("zs_plan_info", _i32, [_P, C.POINTER(zs_plan_info_t)])
_sig("zs_param_info", _i32, [_P, _i32, C.POINTER(zs_param_info_t)])
_sig("zs_param_at", _i32, [_P, _i32, C.POINTER(_i32)])
_sig("zs_bucket_info", _i32, [_P, _i32, C.POINTER(zs_bucket_info_t)])
_sig("zs_bucket_entry", _i32, [_P, _i32, _i32, C.POINTER(_i32), C.POINTER(_i64), C.POINTER(_i64),
                               C.POINTER(_i64)])
_sig("zs_gather_bucket_info", _i32, [_P, _i32, C.POINTER(zs_gather_bucket_info_t)])
_sig("zs_gather_bucket_param", _i32, [_P, _i32, _i32, C.POINTER(_i32)])
_sig("zs_sub_group_info", _i32, [_P, _i32, C.POINTER(zs_sub_group_info_t)])
_sig("zs_plan_table", _i32, [_P, _P, _i64])
_sig("zs_plan_upload", _i32, [_P, _P, _i64, _P])
_sig("zs_partition", _i32, [_P, _P, C.POINTER(zs_shard_state), _P])
_sig("zs_reduce_scatter", _i32, [_P, _i32, C.POINTER(_P), _P, _P, _P, _P])
_sig("zs_grad_norm", _i32, [_P, _P, _P, _P, _i32, _f32, _P, _P, _P, _P])
_sig("zs_adam_step", _i32, [_P, _i32, C.POINTER(zs_adam_hparams), _i64, _P, _P,
                            C.POINTER(zs_shard_state), _P])
_sig("zs_all_gather_coalesced", _i32, [_P, _i32, C.POINTER(_i32), _P, _P, _i64, C.POINTER(_i64), _P])
_sig("zs_device_wait_timeouts", _i32, [C.POINTER(_i32), _i32])
_sig("zs_test_wait_timeout", _i32, [_i64, _P])
_sig("zs_reduce_scatter_all", _i32, [_P, _P, _P, _P, _P, _P])
_sig("zs_reduce_scatter_range", _i32, [_P, _i32, _i32, _P, _P, _P, _P, _P])
_sig("zs_adam_gather", _i32, [_P, C.POINTER(zs_adam_hparams), _i64, _P, _P,
                              C.POINTER(zs_shard_state), _P, _P])
_sig("zs_grad_norm_noalloc", _i32, [_P, _P, _P, _f32, _P, _P, _P, _P])
_sig("zs_unscale_and_clip", _i32, [_P, _P, _P, _P, _i32, _f32, C.POINTER(zs_loss_scaler), _P,
                                   _P, _P, _P])
_sig("zs_shard_step_scaled", _i32, [_P, _P, C.POINTER(zs_shard_state), _P,
                                    C.POINTER(zs_adam_hparams), _i64, _f32,
                                    C.POINTER(zs_loss_scaler), _P, _P, _P, _P, _P])
_sig("zs_sched_create", _i32, [_P, _i32, C.POINTER(_i32), C.POINTER(_i32),
                               C.POINTER(zs_sched_config), _P, C.POINTER(_P)])
_sig("zs_sched_destroy", None, [_P])
_sig("zs_sched_fetch", _i32, [_P, _i32, _P, _P, _P])
_sig("zs_sched_release", _i32, [_P, _i32, _P])
_sig("zs_sched_end_pass", _i32, [_P, _P])
_sig("zs_sched_param_offset", _i32, [_P, _i32, C.POINTER(_i64)])
_sig("zs_sched_stats", _i32, [_P, C.POINTER(zs_sched_stats_t)])
_sig("zs_sched_log", _i32, [_P, C.POINTER(zs_sched_event), _i64, C.POINTER(_i64)])
_sig("zs_shard_step", _i32, [_P, _P, C.POINTER(zs_shard_state), _P, C.POINTER(zs_adam_hparams),
                             _i64, _f32, _P, _P, _P, _P, _P])


def _check(status: int, fn: str) -> None:
    if status != ZS_OK:
        raise ZsError(status, fn, _lib.zs_last_error().decode(errors="replace"))


def _ptr(x):
    """Device/host address of a tensor, an int, or None (NULL)."""
    if x is None:
        return None
    if hasattr(x, "data_ptr"):
        return x.data_ptr()
    return int(x)


def _stream(s):
    if s is None:
        try:
            import torch
            return torch.cuda.current_stream().cuda_stream if torch.cuda.is_available() else None
        except Exception:  # torch without CUDA
            return None
    if hasattr(s, "cuda_stream"):
        return s.cuda_stream
    return int(s)


def _struct(cls, d):
    if isinstance(d, cls):
        return d
    obj = cls()
    for k, v in d.items():
        setattr(obj, k, v)
    return obj


def zs_version() -> str:
    return _lib.zs_version().decode()


def zs_last_error() -> str:
    return _lib.zs_last_error().decode(errors="replace")


def zs_default_config(n_ranks: int) -> zs_config:
    c = zs_config()
    _lib.zs_default_config(C.byref(c), n_ranks)
    return c


class Plan:
    """Owner of a zs_plan* (freed with the object)."""

    def __init__(self, handle: int):
        self._h = handle
        self._table = None   # device buffer the plan was uploaded to (kept alive)

    @property
    def handle(self):
        return self._h

    def __del__(self):
        if getattr(self, "_h", None):
            _lib.zs_free_plan(self._h)
            self._h = None

    def info(self) -> dict:
        return zs_plan_info(self)


def _h(plan):
    return plan.handle if isinstance(plan, Plan) else plan


def zs_build_partition(config, numel, ds_id=None) -> Plan:
    cfg = config if isinstance(config, zs_config) else _struct(zs_config, dict(config))
    n = len(numel)
    arr = (_i64 * max(n, 1))(*[int(x) for x in numel])
    ids = None
    if ds_id is not None:
        ids = (_i64 * max(n, 1))(*[int(x) for x in ds_id])
    out = _P()
    _check(_lib.zs_build_partition(C.byref(cfg), n, arr, ids, C.byref(out)), "zs_build_partition")
    return Plan(out.value)


def zs_free_plan(plan: Plan) -> None:
    if plan._h:
        _lib.zs_free_plan(plan._h)
        plan._h = None


def _to_dict(s):
    return {name: getattr(s, name) for name, _ in s._fields_ if name != "reserved"}


def zs_plan_info(plan) -> dict:
    o = zs_plan_info_t()
    _check(_lib.zs_plan_info(_h(plan), C.byref(o)), "zs_plan_info")
    return _to_dict(o)


def zs_param_info(plan, i: int) -> dict:
    o = zs_param_info_t()
    _check(_lib.zs_param_info(_h(plan), i, C.byref(o)), "zs_param_info")
    return _to_dict(o)


def zs_param_at(plan, position: int) -> int:
    o = _i32()
    _check(_lib.zs_param_at(_h(plan), position, C.byref(o)), "zs_param_at")
    return o.value


def zs_bucket_info(plan, b: int) -> dict:
    o = zs_bucket_info_t()
    _check(_lib.zs_bucket_info(_h(plan), b, C.byref(o)), "zs_bucket_info")
    return _to_dict(o)


def zs_bucket_entry(plan, b: int, q: int):
    p, lo, hi, off = _i32(), _i64(), _i64(), _i64()
    _check(_lib.zs_bucket_entry(_h(plan), b, q, C.byref(p), C.byref(lo), C.byref(hi), C.byref(off)),
           "zs_bucket_entry")
    return p.value, lo.value, hi.value, off.value


def zs_gather_bucket_info(plan, g: int) -> dict:
    o = zs_gather_bucket_info_t()
    _check(_lib.zs_gather_bucket_info(_h(plan), g, C.byref(o)), "zs_gather_bucket_info")
    return _to_dict(o)


def zs_gather_bucket_param(plan, g: int, i: int) -> int:
    o = _i32()
    _check(_lib.zs_gather_bucket_param(_h(plan), g, i, C.byref(o)), "zs_gather_bucket_param")
    return o.value


def zs_sub_group_info(plan, s: int) -> dict:
    o = zs_sub_group_info_t()
    _check(_lib.zs_sub_group_info(_h(plan), s, C.byref(o)), "zs_sub_group_info")
    return _to_dict(o)


def zs_plan_table(plan):
    """Host copy of the work table as a numpy structured array."""
    import numpy as np
    info = zs_plan_info(plan)
    arr = np.zeros(info["n_tiles"], dtype=TILE_DTYPE)
    _check(_lib.zs_plan_table(_h(plan), arr.ctypes.data if arr.size else None, arr.nbytes),
           "zs_plan_table")
    return arr


def zs_plan_launch_order(plan):
    """The reduce-scatter's launch order (int32 per tile: launch position i
    works on tile order[i]), the part of the device table after the tiles."""
    import numpy as np
    info = zs_plan_info(plan)
    n = info["n_tiles"]
    buf = np.zeros(info["device_table_bytes"], dtype=np.uint8)
    _check(_lib.zs_plan_table(_h(plan), buf.ctypes.data if buf.size else None, buf.nbytes),
           "zs_plan_table")
    rec = np.dtype(TILE_DTYPE).itemsize
    return buf[rec * n:(rec + 4) * n].view(np.int32).copy()


def zs_plan_upload(plan, d_table, nbytes: int, stream=None) -> None:
    _check(_lib.zs_plan_upload(_h(plan), _ptr(d_table), int(nbytes), _stream(stream)),
           "zs_plan_upload")
    if isinstance(plan, Plan):
        plan._table = d_table


def make_state(**kw) -> zs_shard_state:
    """zs_shard_state from tensors / addresses given by field name."""
    st = zs_shard_state()
    for name, _ in zs_shard_state._fields_:
        setattr(st, name, _ptr(kw.get(name)))
    return st


def zs_partition(plan, full_params, state: zs_shard_state, stream=None) -> None:
    _check(_lib.zs_partition(_h(plan), _ptr(full_params), C.byref(state), _stream(stream)),
           "zs_partition")


def zs_reduce_scatter(plan, bucket: int, rank_grads, grad_shards, persist_grads,
                      norm_scratch=None, stream=None) -> None:
    ptrs = (_P * max(len(rank_grads), 1))(*[_ptr(x) for x in rank_grads])
    _check(_lib.zs_reduce_scatter(_h(plan), bucket, ptrs, _ptr(grad_shards), _ptr(persist_grads),
                                  _ptr(norm_scratch), _stream(stream)), "zs_reduce_scatter")


def zs_grad_norm(plan, grad_shards, persist_grads, norm_scratch, recompute: bool, max_norm: float,
                 d_norm, d_clip_coef, d_flags, stream=None) -> None:
    _check(_lib.zs_grad_norm(_h(plan), _ptr(grad_shards), _ptr(persist_grads), _ptr(norm_scratch),
                             1 if recompute else 0, float(max_norm), _ptr(d_norm),
                             _ptr(d_clip_coef), _ptr(d_flags), _stream(stream)), "zs_grad_norm")


def _hp(hp) -> zs_adam_hparams:
    if isinstance(hp, zs_adam_hparams):
        return hp
    d = dict(hp)
    return zs_adam_hparams(float(d["lr"]), float(d["beta1"]), float(d["beta2"]), float(d["eps"]),
                           float(d["weight_decay"]), int(d.get("adamw", 1)),
                           int(d.get("bias_correction", 1)))


def zs_adam_step(plan, sub_group: int, hp, step: int, d_clip_coef, d_flags,
                 state: zs_shard_state, stream=None) -> None:
    h = _hp(hp)
    _check(_lib.zs_adam_step(_h(plan), sub_group, C.byref(h), int(step), _ptr(d_clip_coef),
                             _ptr(d_flags), C.byref(state), _stream(stream)), "zs_adam_step")


def zs_all_gather_coalesced(plan, params, param_shards, flat_out, flat_capacity: int,
                            stream=None) -> list:
    n = len(params)
    arr = (_i32 * max(n, 1))(*[int(x) for x in params])
    views = (_i64 * max(n, 1))()
    _check(_lib.zs_all_gather_coalesced(_h(plan), n, arr, _ptr(param_shards), _ptr(flat_out),
                                        int(flat_capacity), views, _stream(stream)),
           "zs_all_gather_coalesced")
    return [views[i] for i in range(n)]


def zs_device_wait_timeouts(reset: bool = False) -> int:
    """Bounded device waits that gave up on the current device (synchronous)."""
    c = _i32()
    st = _lib.zs_device_wait_timeouts(C.byref(c), int(bool(reset)))
    if st != ZS_ETIMEOUT:
        _check(st, "zs_device_wait_timeouts")
    return c.value


def zs_test_wait_timeout(limit_ns: int, stream=None) -> None:
    """Enqueue one bounded wait that runs out after limit_ns (test hook)."""
    _check(_lib.zs_test_wait_timeout(int(limit_ns), _stream(stream)), "zs_test_wait_timeout")


def zs_shard_step(plan, d_rank_grads, state: zs_shard_state, norm_scratch, hp, step: int,
                  max_norm: float, d_norm, d_clip_coef, d_flags, flat_out, stream=None) -> None:
    h = _hp(hp)
    _check(_lib.zs_shard_step(_h(plan), _ptr(d_rank_grads), C.byref(state), _ptr(norm_scratch),
                              C.byref(h), int(step), float(max_norm), _ptr(d_norm),
                              _ptr(d_clip_coef), _ptr(d_flags), _ptr(flat_out), _stream(stream)),
           "zs_shard_step")


def zs_reduce_scatter_all(plan, d_rank_grads, grad_shards, persist_grads, norm_scratch,
                          stream=None) -> None:
    _check(_lib.zs_reduce_scatter_all(_h(plan), _ptr(d_rank_grads), _ptr(grad_shards),
                                      _ptr(persist_grads), _ptr(norm_scratch), _stream(stream)),
           "zs_reduce_scatter_all")


def zs_reduce_scatter_range(plan, first_bucket: int, n_buckets: int, d_rank_grads, grad_shards,
                            persist_grads, norm_scratch, stream=None) -> None:
    _check(_lib.zs_reduce_scatter_range(_h(plan), int(first_bucket), int(n_buckets),
                                        _ptr(d_rank_grads), _ptr(grad_shards), _ptr(persist_grads),
                                        _ptr(norm_scratch), _stream(stream)),
           "zs_reduce_scatter_range")


def zs_adam_gather(plan, hp, step: int, d_clip_coef, d_flags, state: zs_shard_state, flat_out,
                   stream=None) -> None:
    h = _hp(hp)
    _check(_lib.zs_adam_gather(_h(plan), C.byref(h), int(step), _ptr(d_clip_coef), _ptr(d_flags),
                               C.byref(state), _ptr(flat_out), _stream(stream)), "zs_adam_gather")


def zs_grad_norm_noalloc(plan, grad_shards, persist_grads, max_norm: float, d_norm, d_clip_coef,
                         d_flags, stream=None) -> None:
    """zs_grad_norm(recompute=1) with the library's built-in scratch array,
    for callers that cannot allocate device memory."""
    _check(_lib.zs_grad_norm_noalloc(_h(plan), _ptr(grad_shards), _ptr(persist_grads),
                                     float(max_norm), _ptr(d_norm), _ptr(d_clip_coef),
                                     _ptr(d_flags), _stream(stream)), "zs_grad_norm_noalloc")


def make_loss_scaler(d_scale, d_good_steps=None, scale_factor=2.0, min_scale=1.0,
                     scale_window=1000) -> zs_loss_scaler:
    """zs_loss_scaler from device tensors / addresses (float32 scale, int32 count)."""
    return zs_loss_scaler(_ptr(d_scale), _ptr(d_good_steps), float(scale_factor),
                          float(min_scale), int(scale_window), 0)


def zs_unscale_and_clip(plan, grad_shards, persist_grads, norm_scratch, recompute: bool,
                        max_norm: float, scaler: zs_loss_scaler, d_norm, d_clip_coef, d_flags,
                        stream=None) -> None:
    _check(_lib.zs_unscale_and_clip(_h(plan), _ptr(grad_shards), _ptr(persist_grads),
                                    _ptr(norm_scratch), 1 if recompute else 0, float(max_norm),
                                    C.byref(scaler), _ptr(d_norm), _ptr(d_clip_coef),
                                    _ptr(d_flags), _stream(stream)), "zs_unscale_and_clip")


def zs_shard_step_scaled(plan, d_rank_grads, state: zs_shard_state, norm_scratch, hp, step: int,
                         max_norm: float, scaler: zs_loss_scaler, d_norm, d_clip_coef, d_flags,
                         flat_out, stream=None) -> None:
    h = _hp(hp)
    _check(_lib.zs_shard_step_scaled(_h(plan), _ptr(d_rank_grads), C.byref(state),
                                     _ptr(norm_scratch), C.byref(h), int(step), float(max_norm),
                                     C.byref(scaler), _ptr(d_norm), _ptr(d_clip_coef),
                                     _ptr(d_flags), _ptr(flat_out), _stream(stream)),
           "zs_shard_step_scaled")


class Sched:
    """Owner of a zs_sched* (destroyed with the object); keeps the plan alive."""

    def __init__(self, handle, plan, arena):
        self._h, self._plan, self._arena = handle, plan, arena

    @property
    def handle(self):
        return self._h

    def __del__(self):
        if getattr(self, "_h", None):
            _lib.zs_sched_destroy(self._h)
            self._h = None


def zs_sched_create(plan, modules, cfg, d_arena=None) -> Sched:
    """modules: list of lists of parameter indices; cfg: dict or zs_sched_config."""
    c = cfg if isinstance(cfg, zs_sched_config) else _struct(zs_sched_config, dict(cfg))
    offs, flat = [0], []
    for m in modules:
        flat += [int(p) for p in m]
        offs.append(len(flat))
    o = (_i32 * len(offs))(*offs)
    f = (_i32 * max(len(flat), 1))(*flat)
    out = _P()
    _check(_lib.zs_sched_create(_h(plan), len(modules), o, f, C.byref(c), _ptr(d_arena),
                                C.byref(out)), "zs_sched_create")
    return Sched(out.value, plan, d_arena)


def zs_sched_fetch(sched, module: int, param_shards=None, compute_stream=None,
                   gather_stream=None) -> None:
    _check(_lib.zs_sched_fetch(sched.handle, module, _ptr(param_shards),
                               _stream(compute_stream) if sched._arena is not None else None,
                               _stream(gather_stream) if sched._arena is not None else None),
           "zs_sched_fetch")


def zs_sched_release(sched, module: int, compute_stream=None) -> None:
    _check(_lib.zs_sched_release(sched.handle, module,
                                 _stream(compute_stream) if sched._arena is not None else None),
           "zs_sched_release")


def zs_sched_end_pass(sched, compute_stream=None) -> None:
    _check(_lib.zs_sched_end_pass(sched.handle,
                                  _stream(compute_stream) if sched._arena is not None else None),
           "zs_sched_end_pass")


def zs_sched_param_offset(sched, param: int) -> int:
    o = _i64()
    _check(_lib.zs_sched_param_offset(sched.handle, param, C.byref(o)), "zs_sched_param_offset")
    return o.value


def zs_sched_stats(sched) -> dict:
    o = zs_sched_stats_t()
    _check(_lib.zs_sched_stats(sched.handle, C.byref(o)), "zs_sched_stats")
    return {n: getattr(o, n) for n, _ in o._fields_}


def zs_sched_log(sched) -> list:
    n = _i64()
    _check(_lib.zs_sched_log(sched.handle, None, 0, C.byref(n)), "zs_sched_log")
    buf = (zs_sched_event * max(n.value, 1))()
    _check(_lib.zs_sched_log(sched.handle, buf, n.value, C.byref(n)), "zs_sched_log")
    return [(e.kind, e.module_pos, e.op, e.param, e.offset, e.aux) for e in buf[:n.value]]
