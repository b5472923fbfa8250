"""GPU test harness: one plan on the device next to the oracle's plan.

Every output buffer sits between two guard regions filled with a canary
pattern; `check_canaries` verifies after each call that no kernel wrote
outside its buffer (the bounds check these tests use in place of a memory
sanitizer).  Inputs come from the shared generator `synth` only (the CPU
implementation, or the GPU one for larger inputs, which
test_gpu_parity.test_generator_gpu_matches_cpu pins to the CPU one).

Tolerances (the parity targets of the method, written out):
  reduce-scatter, partition, gather : bit-exact
  gradient norm                     : |a - b| <= 1e-5 |b|
  fp32 master / exp_avg / exp_avg_sq: bit-exact whenever the device's clip
        coefficient has the oracle's bits (the same float32 operations in the
        same order; the device accumulates the norm without rounding error, so
        its coefficient is the oracle's in practice); otherwise, per element,
        |a - b| <= 1e-6 max(|b|, |prev|), prev the oracle's value of the same
        element before the step (the floor for values that cancel towards 0)
  16-bit parameters                 : bit-exact with the same coefficient,
        else within 1 ulp of the oracle's value
"""
from __future__ import annotations

import numpy as np
import torch

import zero_sharded_optimizer_bucket_gb300 as zs
from oracle import plan as oplan
from oracle import step as ostep
from oracle.bf16 import bf16_to_f32
from synth import gpu as sgpu
from synth import philox

GUARD = 64                     # elements on each side (16-byte multiple for 2- and 4-byte types)
CANARY16 = -21555              # 0xABCD as int16
CANARY32 = float(np.frombuffer(np.uint32(0x7FBADBAD).tobytes(), np.float32)[0])


class Guarded:
    """A device buffer of n elements with canary guards on both sides."""

    def __init__(self, n, dtype, device, fill=0):
        self.n = int(n)
        self.full = torch.empty(self.n + 2 * GUARD, dtype=dtype, device=device)
        if dtype == torch.float32:
            self.full.view(torch.int32).fill_(0x7FBADBAD)
        elif dtype == torch.float64:
            self.full.view(torch.int64).fill_(0x7FF0BADBADBADBAD)
        else:
            self.full.fill_(CANARY16)
        self.t = self.full[GUARD:GUARD + self.n]
        self.t.zero_() if fill == 0 else self.t.fill_(fill)

    def ptr(self):
        return self.t.data_ptr()

    def guards_ok(self):
        a, b = self.full[:GUARD], self.full[GUARD + self.n:]
        if self.full.dtype == torch.float32:
            a, b = a.view(torch.int32), b.view(torch.int32)
            return bool((a == 0x7FBADBAD).all() and (b == 0x7FBADBAD).all())
        if self.full.dtype == torch.float64:
            a, b = a.view(torch.int64), b.view(torch.int64)
            return bool((a == 0x7FF0BADBADBADBAD).all() and (b == 0x7FF0BADBADBADBAD).all())
        return bool((a == CANARY16).all() and (b == CANARY16).all())

    def u16(self):
        return self.t.cpu().numpy().view(np.uint16)

    def np(self):
        return self.t.cpu().numpy()


class DevicePlan:
    def __init__(self, numel, N, threshold=100_000, B=5_000_000, G=50_000_000, U=10**9,
                 ds_id=None, seed=1234, sigma=1e-2, outlier=0.0, device="cuda:0", dtype="bf16",
                 log2_scale=-4, outlier_log2=0, group=0):
        self.dev = torch.device(device)
        self.numel, self.N, self.seed, self.sigma, self.outlier = numel, N, seed, sigma, outlier
        self.dtype, self.log2_scale, self.outlier_log2 = dtype, log2_scale, outlier_log2
        self.op = oplan.build_partition(numel, N, threshold=threshold, reduce_bucket_size=B,
                                        prefetch_bucket_size=G, sub_group_size=U, ds_id=ds_id,
                                        dtype=dtype, shard_group_size=group or None)
        cfg = zs.zs_default_config(N)
        cfg.dtype = zs.ZS_DTYPE_FP16 if dtype == "fp16" else zs.ZS_DTYPE_BF16
        cfg.shard_group_size = group
        cfg.param_persistence_threshold = threshold
        cfg.reduce_bucket_size = B
        cfg.prefetch_bucket_size = G
        cfg.sub_group_size = U
        self.plan = zs.zs_build_partition(cfg, numel, ds_id)
        self.info = zs.zs_plan_info(self.plan)
        assert self.info["shard_elems"] == self.op.S and self.info["persist_elems"] == self.op.Pn_alloc
        S, P = self.op.S, self.op.Pn_alloc
        N = self.op.group          # rows of shard space: a group's shard owners
        d = self.dev
        self.table = torch.empty(max(self.info["device_table_bytes"], 16), dtype=torch.uint8, device=d)
        zs.zs_plan_upload(self.plan, self.table, self.table.numel())
        self.bufs = {
            "grad_shards": Guarded(N * S, torch.int16, d), "param_shards": Guarded(N * S, torch.int16, d),
            "master": Guarded(N * S, torch.float32, d), "exp_avg": Guarded(N * S, torch.float32, d),
            "exp_avg_sq": Guarded(N * S, torch.float32, d), "persist_grads": Guarded(P, torch.int16, d),
            "persist_params": Guarded(P, torch.int16, d), "p_master": Guarded(P, torch.float32, d),
            "p_exp_avg": Guarded(P, torch.float32, d), "p_exp_avg_sq": Guarded(P, torch.float32, d),
        }
        self.state = zs.make_state(**{k: v.ptr() for k, v in self.bufs.items()})
        self.scratch = Guarded(self.info["norm_scratch_elems"], torch.float64, d)
        self.d_norm = Guarded(1, torch.float32, d)
        self.d_coef = Guarded(1, torch.float32, d)
        self.d_flags = Guarded(1, torch.int32, d)
        self.flat = Guarded(self.op.flat_elems, torch.int16, d)
        self.grad_bufs = None
        self.dev_grads = None

    # ------------------------------------------------------------ inputs --
    def init_weights(self):
        W = philox.weight_f32(self.seed, np.arange(self.op.input_elems, dtype=np.uint64), 0.02)
        Wd = torch.from_numpy(W).to(self.dev)
        zs.zs_partition(self.plan, Wd, self.state)
        self.ost = ostep.partition(self.op, W)
        torch.cuda.synchronize()

    def set_grads(self, step_seed, use_gpu_generator=False):
        """Rank gradient buffers of every bucket, drawn at consecutive pool
        indices (bucket-major, rank-minor)."""
        op, N = self.op, self.N
        total = sum(N * L for L in op.bucket_buf_elems)
        if use_gpu_generator:
            pool = torch.empty(max(total, 8), dtype=torch.int16, device=self.dev)
            if self.dtype == "fp16":
                sgpu.fill_grad_fp16(pool, 0, step_seed, self.log2_scale, self.outlier,
                                    self.outlier_log2)
            else:
                sgpu.fill_grad_bf16(pool, 0, step_seed, self.sigma, self.outlier)
            host = pool.cpu().numpy().view(np.uint16)
        else:
            idx = np.arange(total, dtype=np.uint64)
            if not total:
                host = np.zeros(0, np.uint16)
            elif self.dtype == "fp16":
                host = philox.grad_fp16(step_seed, 0, idx, self.log2_scale, self.outlier,
                                        self.outlier_log2)
            else:
                host = philox.grad_bf16(step_seed, 0, idx, self.sigma, self.outlier)
            pool = torch.from_numpy(host.view(np.int16).copy()).to(self.dev)
        self.grad_bufs, self.ptrs, run = [], [], 0
        for L in op.bucket_buf_elems:
            row, prow = [], []
            for k in range(N):
                row.append(host[run:run + L])
                prow.append(pool.data_ptr() + 2 * run)
                run += L
            self.grad_bufs.append(row)
            self.ptrs.append(prow)
        self.pool = pool
        flat_ptrs = [p for row in self.ptrs for p in row]
        self.ptr_table = torch.tensor(flat_ptrs or [0], dtype=torch.int64, device=self.dev)

    # ------------------------------------------------------------- calls --
    def reduce_scatter_all_buckets(self, with_scratch=True):
        for b in range(len(self.op.reduce_buckets)):
            zs.zs_reduce_scatter(self.plan, b, self.ptrs[b], self.bufs["grad_shards"].ptr(),
                                 self.bufs["persist_grads"].ptr(),
                                 self.scratch.ptr() if with_scratch else None)

    def grad_norm(self, max_norm, recompute):
        zs.zs_grad_norm(self.plan, self.bufs["grad_shards"].ptr(), self.bufs["persist_grads"].ptr(),
                        self.scratch.ptr(), recompute, max_norm, self.d_norm.ptr(),
                        self.d_coef.ptr(), self.d_flags.ptr())

    def adam(self, hp, step, sub_group=-1):
        zs.zs_adam_step(self.plan, sub_group, hp, step, self.d_coef.ptr(), self.d_flags.ptr(),
                        self.state)

    def shard_step(self, hp, step, max_norm):
        zs.zs_shard_step(self.plan, self.ptr_table, self.state, self.scratch.ptr(), hp, step,
                         max_norm, self.d_norm.ptr(), self.d_coef.ptr(), self.d_flags.ptr(),
                         self.flat.ptr())

    def gather_model_unfused(self, out: Guarded):
        """zs_all_gather_coalesced of every gather bucket into its place."""
        for g in self.op.gather_buckets:
            base = out.ptr() + 2 * g.flat_off
            views = zs.zs_all_gather_coalesced(self.plan, g.params, self.bufs["param_shards"].ptr(),
                                               base, g.flat_elems)
            assert views == [self.op.params[i].flat_off - g.flat_off for i in g.params]

    # ------------------------------------------------------------ checks --
    def check_canaries(self):
        torch.cuda.synchronize()
        for name, b in list(self.bufs.items()) + [("scratch", self.scratch), ("flat", self.flat),
                                                   ("norm", self.d_norm), ("coef", self.d_coef),
                                                   ("flags", self.d_flags)]:
            assert b.guards_ok(), f"write outside {name}"

    def snapshot(self):
        torch.cuda.synchronize()
        N, S = self.op.group, self.op.S
        out = {}
        for k, b in self.bufs.items():
            a = b.u16() if b.t.dtype == torch.int16 else b.np()
            out[k] = a.reshape(N, S) if b.n == N * S and k in ("grad_shards", "param_shards", "master",
                                                                "exp_avg", "exp_avg_sq") else a
        return out


# ------------------------------------------------------------ compare -----
STATE = ("master", "exp_avg", "exp_avg_sq", "p_master", "p_exp_avg", "p_exp_avg_sq")


def oracle_state(ost):
    """A copy of the oracle's fp32 state: the previous values of the
    per-element bound of the next step."""
    return {k: getattr(ost, k).copy() for k in STATE}


def same_bits(a, b) -> bool:
    return np.float32(a).tobytes() == np.float32(b).tobytes()


def assert_f32_close(a, b, what, prev=None, rtol=1e-6):
    """|a - b| <= rtol * max(|b|, |prev|) per element (exact equality where
    both are 0); prints and returns the worst relative error."""
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if a.size == 0:
        return 0.0
    scale = np.abs(b) if prev is None else np.maximum(np.abs(b), np.abs(np.asarray(prev, np.float64)))
    err = np.abs(a - b)
    bad = ~(err <= rtol * scale)
    with np.errstate(divide="ignore", invalid="ignore"):
        rel = np.where(scale > 0, err / scale, np.where(err > 0, np.inf, 0.0))
    worst = float(np.max(rel))
    print(f"{what}: worst relative error {worst:.3e} over {a.size} elements")
    assert not bad.any(), (f"{what}: {int(bad.sum())} of {a.size} outside 1e-6 relative; "
                           f"worst {worst:.3e}")
    return worst


def assert_state(got, ost, prev, what, exact, keys=STATE):
    """The device's fp32 state (dict of arrays) against the oracle's: bit for
    bit when both used the same clip coefficient (exact), else within the
    per-element bound against the oracle's previous values prev."""
    for k in keys:
        ref = getattr(ost, k) if not isinstance(ost, dict) else ost[k]
        if exact:
            same = np.array_equal(np.asarray(got[k]).view(np.uint32), np.asarray(ref).view(np.uint32))
            assert same, f"{what}: {k} not bit-identical to the oracle"
        else:
            assert_f32_close(got[k], ref, f"{what}: {k}", prev[k])
    if exact:
        print(f"{what}: {', '.join(keys)} bit-identical to the oracle")


def assert_16bit(a_u16, b_u16, what, dtype, exact):
    """16-bit parameters: bits with the oracle's coefficient, else 1 ulp."""
    if exact:
        assert np.array_equal(np.asarray(a_u16, np.uint16), np.asarray(b_u16, np.uint16)), \
            f"{what}: not bit-identical to the oracle"
    elif dtype == "fp16":
        assert_fp16_within_ulp(a_u16, b_u16, what)
    else:
        assert_bf16_within_ulp(a_u16, b_u16, what)


def bf16_ulp(x_u16):
    v = np.abs(bf16_to_f32(x_u16).astype(np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -133)))
    return np.maximum(2.0 ** (e - 7), 2.0 ** -133)


def fp16_ulp(x_u16):
    v = np.abs(np.asarray(x_u16, np.uint16).view(np.float16).astype(np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -24)))
    return np.maximum(2.0 ** (e - 10), 2.0 ** -24)


def assert_fp16_within_ulp(a_u16, b_u16, what):
    a = np.asarray(a_u16, np.uint16).view(np.float16).astype(np.float64)
    b = np.asarray(b_u16, np.uint16).view(np.float16).astype(np.float64)
    bad = np.abs(a - b) > fp16_ulp(b_u16) * (1 + 1e-9)
    assert not bad.any(), f"{what}: {int(bad.sum())} values more than 1 fp16 ulp away"


def assert_bf16_within_ulp(a_u16, b_u16, what):
    a = bf16_to_f32(a_u16).astype(np.float64)
    b = bf16_to_f32(b_u16).astype(np.float64)
    bad = np.abs(a - b) > bf16_ulp(b_u16) * (1 + 1e-9)
    assert not bad.any(), f"{what}: {int(bad.sum())} values more than 1 bf16 ulp away"
