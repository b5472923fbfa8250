"""A1 data movement, A2 reduce-scatter, A3 norm/clip, A4 Adam(W)+cast,
A5 all_gather_coalesced: the oracle's arithmetic.

Floating point is numpy float32, one IEEE operation per step below, in the
order written; the gradient norm is float64 with an exactly rounded sum
(math.fsum).  Buffers are numpy arrays in the layouts of `oracle.plan`:
    grad_shards, param_shards  uint16  [N][S]   (bfloat16 or, when the plan's
                                                 dtype is fp16, binary16 bits)
    master, exp_avg, exp_avg_sq float32 [N][S]
    persist_* likewise, [Pn_alloc]
"""
from __future__ import annotations

import math
from dataclasses import dataclass
from fractions import Fraction

import numpy as np

from .bf16 import bf16_to_f32, f32_to_bf16
from .fp16 import f32_to_fp16, fp16_to_f32
from .plan import Plan


def to_f32(u16, dtype: str = "bf16") -> np.ndarray:
    return bf16_to_f32(u16) if dtype == "bf16" else fp16_to_f32(u16)


def from_f32(x, dtype: str = "bf16") -> np.ndarray:
    return f32_to_bf16(x) if dtype == "bf16" else f32_to_fp16(x)

F32 = np.float32


@dataclass
class State:
    master: np.ndarray
    exp_avg: np.ndarray
    exp_avg_sq: np.ndarray
    param_shards: np.ndarray
    grad_shards: np.ndarray
    p_master: np.ndarray
    p_exp_avg: np.ndarray
    p_exp_avg_sq: np.ndarray
    persist_params: np.ndarray
    persist_grads: np.ndarray


def new_state(plan: Plan) -> State:
    N, S, P = plan.group, plan.S, plan.Pn_alloc
    z32 = lambda *s: np.zeros(s, dtype=np.float32)
    z16 = lambda *s: np.zeros(s, dtype=np.uint16)
    return State(z32(N, S), z32(N, S), z32(N, S), z16(N, S), z16(N, S),
                 z32(P), z32(P), z32(P), z16(P), z16(P))


# ---------------------------------------------------------------- A1 -----
def partition(plan: Plan, W: np.ndarray) -> State:
    """Copy each rank's range [r*ps, (r+1)*ps) of every full parameter into
    its fp32 master shard, zero beyond numel ([ZeRO-3 chapter] §3.1 item 1:
    _partition_param copies the rank's element range into ds_tensor; §6.1:
    one fp32 master partition per rank).  Persistent parameters are copied
    whole ([ZeRO-3 chapter] §5.3).  Moments start at zero; the 16-bit shard
    is the rounded master."""
    W = np.asarray(W, dtype=np.float32)
    st = new_state(plan)
    N = plan.group
    for p in plan.params:
        if p.persistent:
            st.p_master[p.persist_off:p.persist_off + p.numel] = \
                W[p.input_off:p.input_off + p.numel]
            continue
        if p.ps == 0:
            continue
        e = np.arange(N * p.ps)
        valid = e < p.numel
        vals = np.zeros(e.shape, dtype=np.float32)
        vals[valid] = W[p.input_off + e[valid]]
        st.master[e // p.ps, p.shard_off + e % p.ps] = vals
    st.param_shards = from_f32(st.master, plan.dtype)
    st.persist_params = from_f32(st.p_master, plan.dtype)
    return st


# ---------------------------------------------------------------- A2 -----
def reduce_mean_bf16(vals: np.ndarray) -> np.ndarray:
    """Mean over ranks of bf16 gradients, element-wise: s = 0; for k = 0..N-1:
    s = s + float(g_k) (float32, rank order); result bf16(s / N).
    The average of [Grok blog] §3 (Backward: sum, average, scatter) and the
    avg-scatter of [ZeRO-3 chapter] §6.2."""
    vals = np.asarray(vals, dtype=np.uint16)
    N = vals.shape[0]
    s = np.zeros(vals.shape[1:], dtype=np.float32)
    for k in range(N):
        s = s + bf16_to_f32(vals[k])
    return f32_to_bf16(s / F32(N))


def reduce_mean_fp16(vals: np.ndarray) -> np.ndarray:
    """The same mean for fp16 gradients: float32 sum in rank order, s / N,
    rounded to fp16 (an overflow becomes inf, which the norm then reports)."""
    vals = np.asarray(vals, dtype=np.uint16)
    N = vals.shape[0]
    s = np.zeros(vals.shape[1:], dtype=np.float32)
    for k in range(N):
        s = s + fp16_to_f32(vals[k])
    return f32_to_fp16(s / F32(N))


def reduce_mean(vals, dtype: str = "bf16") -> np.ndarray:
    return reduce_mean_bf16(vals) if dtype == "bf16" else reduce_mean_fp16(vals)


def reduce_mean_groups(vals, G: int, dtype: str = "bf16") -> np.ndarray:
    """HSDP mean ([Core flow] §4: reduce-scatter inside each replica group,
    all-reduce across groups): each group's G ranks are summed in rank order
    from 0 (float32), the group sums are added in group order from 0, and
    the total is divided by the number of ranks N and rounded to 16 bits.
    With one group this is the flat mean, bit for bit (0 + s == s)."""
    vals = np.asarray(vals, dtype=np.uint16)
    N = vals.shape[0]
    if G == N:
        return reduce_mean(vals, dtype)
    total = np.zeros(vals.shape[1:], dtype=np.float32)
    for g in range(N // G):
        inner = np.zeros(vals.shape[1:], dtype=np.float32)
        for j in range(G):
            inner = inner + to_f32(vals[g * G + j], dtype)
        total = total + inner
    return from_f32(total / F32(N), dtype)


def reduce_scatter(plan: Plan, bucket: int, rank_bufs, st: State) -> None:
    """Reduce bucket `bucket` of all N ranks and keep each rank's slice
    ([ZeRO-3 chapter] §6.2: all_reduce of the bucket then each rank keeps its
    range, or reduce_scatter to the owners; both give this result).
    rank_bufs[k] is rank k's gradient buffer of the bucket (uint16)."""
    N, G = plan.n_ranks, plan.group
    assert len(rank_bufs) == N
    for ent in plan.reduce_buckets[bucket]:
        p = plan.params[ent.param]
        if p.persistent:
            L = ent.e_hi - ent.e_lo
            vals = np.stack([np.asarray(b[ent.buf_off:ent.buf_off + L]) for b in rank_bufs])
            st.persist_grads[p.persist_off + ent.e_lo:p.persist_off + ent.e_hi] = \
                reduce_mean_groups(vals, G, plan.dtype)
            continue
        # the bucket holding the parameter's last element also owns the
        # padding elements numel .. N*ps-1 (gradient zero)
        hi = G * p.ps if ent.e_hi == p.numel else ent.e_hi
        if hi <= ent.e_lo:
            continue
        e = np.arange(ent.e_lo, hi)
        valid = e < p.numel
        vals = np.zeros((N, e.size), dtype=np.uint16)
        src = ent.buf_off + (e[valid] - ent.e_lo)
        for k in range(N):
            vals[k, valid] = np.asarray(rank_bufs[k])[src]
        st.grad_shards[e // p.ps, p.shard_off + e % p.ps] = reduce_mean_groups(vals, G, plan.dtype)


# ---------------------------------------------------------------- A3 -----
CLIP_EPS = F32(1e-6)


def grad_norm(plan: Plan, st: State, max_norm: float):
    """Global L2 norm over every rank's shard and the persistent gradients
    (each element once), and the clip coefficient.  The norm must be the
    global one, not a rank's own ([Core flow] 坑 1: per-rank clipping
    silently diverges; [ZeRO-3 chapter] §6.3: unscale_and_clip_grads takes
    global_norm).  norm = float32(sqrt(sum g^2)) with the sum exact in
    float64; coef = min(1, max_norm / (norm + 1e-6)) in float32 (1 when
    max_norm <= 0); a non-finite norm sets skip (coef reported as 1).
    This is unscale_and_clip with loss scale 1."""
    return unscale_and_clip(plan, st, max_norm, 1.0)


def unscale_and_clip(plan: Plan, st: State, max_norm: float, scale: float):
    """unscale_and_clip_grads of [ZeRO-3 chapter] §6.3: the stored gradients
    are the gradients of the loss times `scale` (the loss scale, 1 for bf16).
    norm = float32(sqrt(sum g^2)) / scale is the norm of the true gradients;
    clip = min(1, max_norm / (norm + 1e-6)) (1 when max_norm <= 0);
    coef = clip / scale is the factor the optimizer applies to the stored
    gradients (float32 operations).  A non-finite norm (an overflow) sets
    skip, with coef reported as 1."""
    sq = np.concatenate([to_f32(st.grad_shards, plan.dtype).ravel(),
                         to_f32(st.persist_grads, plan.dtype).ravel()]).astype(np.float64)
    sq = sq * sq
    if np.all(np.isfinite(sq)):
        total = math.fsum(sq.tolist())
    else:
        total = float(np.sum(sq))
    return clip_from_sumsq(total, max_norm, scale)


def clip_from_sumsq(total: float, max_norm: float, scale: float = 1.0):
    """The finish of unscale_and_clip from the sum of squares of the stored
    gradients (float64): (norm, coef, skip) as documented there."""
    S = F32(scale)
    norm = F32(np.sqrt(np.float64(total))) / S
    skip = not bool(np.isfinite(norm))
    if skip:
        return norm, F32(1.0), True
    clip = F32(1.0)
    if max_norm > 0:
        c = F32(max_norm) / (norm + CLIP_EPS)
        clip = c if c < F32(1.0) else F32(1.0)
    return norm, clip / S, False


# ------------------------------------------------ A3, bucket by bucket ---
# The global norm of a model too large to hold the oracle's whole state:
# the reduced gradients are formed one reduce bucket at a time, as the pages'
# backward pass produces them ([ZeRO-3 chapter] §6.2, IPG bucket), and only
# the multiset of their values is kept: how many times each 16-bit |x| bit
# pattern occurs.  The sum of squares is then sum over patterns of
# count * value^2, evaluated exactly in rationals and rounded once, which is
# the same correctly rounded float64 as the fsum of unscale_and_clip.
def bucket_sq_counts(plan: Plan, bucket: int, rank_bufs) -> np.ndarray:
    """Occurrences (int64, 2^15 bins indexed by the bits of |x|) of the
    reduced gradient values that reduce_scatter writes for bucket `bucket`:
    each element of each of the bucket's entries once, the rank mean taken
    as reduce_scatter takes it (reduce_mean_groups).  Padding elements are
    zero and left out.  rank_bufs[k] is rank k's gradient buffer of the
    bucket."""
    counts = np.zeros(1 << 15, dtype=np.int64)
    assert len(rank_bufs) == plan.n_ranks
    for ent in plan.reduce_buckets[bucket]:
        L = ent.e_hi - ent.e_lo
        if L <= 0:
            continue
        vals = np.stack([np.asarray(b[ent.buf_off:ent.buf_off + L]) for b in rank_bufs])
        red = reduce_mean_groups(vals, plan.group, plan.dtype)
        counts += np.bincount(red & np.uint16(0x7FFF), minlength=1 << 15)
    return counts


def sumsq_from_counts(counts, dtype: str = "bf16") -> float:
    """sum over bit patterns of count * value^2, exact (Fraction), rounded
    once to float64; inf when an infinite value occurs, nan when a NaN
    does."""
    counts = np.asarray(counts, dtype=np.int64)
    nz = np.nonzero(counts)[0]
    vals = to_f32(nz.astype(np.uint16), dtype)
    if np.any(np.isnan(vals)):
        return float("nan")
    if np.any(np.isinf(vals)):
        return float("inf")
    total = Fraction(0)
    for c, v in zip(counts[nz].tolist(), vals.tolist()):
        total += c * Fraction(v) ** 2
    return float(total)


def grad_norm_streamed(plan: Plan, bucket_bufs, max_norm: float, scale: float = 1.0):
    """unscale_and_clip computed bucket by bucket: bucket_bufs yields
    (bucket, rank_bufs) for every reduce bucket once, in any order (the
    counts add up).  Returns (norm, coef, skip)."""
    counts = np.zeros(1 << 15, dtype=np.int64)
    seen = set()
    for b, rank_bufs in bucket_bufs:
        if b in seen:
            raise ValueError(f"bucket {b} given twice")
        seen.add(b)
        counts += bucket_sq_counts(plan, b, rank_bufs)
    if len(seen) != len(plan.reduce_buckets):
        raise ValueError("every reduce bucket must be given once")
    return clip_from_sumsq(sumsq_from_counts(counts, plan.dtype), max_norm, scale)


@dataclass
class LossScaler:
    """Dynamic loss scale (the scale the caller multiplies the loss by for
    fp16 gradients).  After a step whose gradients overflowed (skip): scale
    = max(scale / factor, min_scale) and the count of good steps restarts;
    after `window` consecutive good steps: scale = scale * factor.  The
    pages name the unscale step ([ZeRO-3 chapter] §6.3) but not the
    schedule; this is DeepSpeed's documented dynamic schedule without
    hysteresis, in float32."""
    scale: float = 65536.0
    good: int = 0
    factor: float = 2.0
    min_scale: float = 1.0
    window: int = 1000

    def update(self, overflow: bool) -> None:
        if overflow:
            self.scale = float(max(F32(self.scale) / F32(self.factor), F32(self.min_scale)))
            self.good = 0
        else:
            self.good += 1
            if self.good >= self.window:
                self.scale = float(F32(self.scale) * F32(self.factor))
                self.good = 0


# ---------------------------------------------------------------- A4 -----
@dataclass
class AdamConsts:
    lr: np.float32
    b1: np.float32
    b2: np.float32
    omb1: np.float32
    omb2: np.float32
    eps: np.float32
    wd: np.float32
    lr_wd: np.float32
    bc1: np.float32
    bc2: np.float32
    adamw: bool


def adam_consts(hp: dict, step: int) -> AdamConsts:
    """Scalars of step t (t >= 1): hyper-parameters as float32; 1-beta,
    lr*wd and the bias corrections 1-beta^t evaluated in float64 and rounded
    once to float32."""
    if step < 1:
        raise ValueError("step must be >= 1")
    lr, b1, b2 = F32(hp["lr"]), F32(hp["beta1"]), F32(hp["beta2"])
    eps, wd = F32(hp["eps"]), F32(hp["weight_decay"])
    if hp.get("bias_correction", 1):
        bc1 = F32(1.0 - float(b1) ** step)
        bc2 = F32(1.0 - float(b2) ** step)
    else:
        bc1 = bc2 = F32(1.0)
    return AdamConsts(lr, b1, b2, F32(1.0 - float(b1)), F32(1.0 - float(b2)), eps, wd,
                      F32(float(lr) * float(wd)), bc1, bc2, bool(hp.get("adamw", 1)))


def adam_update(p, m, v, gs_bf16, coef, c: AdamConsts, dtype: str = "bf16"):
    """One Adam(W) update of fp32 master p and moments m, v from the reduced
    bf16 gradient; returns (p, m, v, bf16(p)).  The optimizer sees only the
    rank's fp32 partition ([ZeRO-3 chapter] §6.3) and writes back the 16-bit
    shard (_reassign_or_swap_out_partitioned_parameters, §6.3); 12 bytes of
    fp32 state per element ([Core flow] §1).  The pages do not state the
    update itself; this is AdamW with decoupled decay (or L2 decay folded
    into the gradient when adamw is off), bias correction and eps outside
    the square root:
        g  = float(gs) * coef
        p  = p - (lr*wd) * p            [AdamW]   |  g = g + wd * p   [L2]
        m  = b1*m + (1-b1)*g
        v  = b2*v + (1-b2)*(g*g)
        p  = p - lr * ((m/bc1) / (sqrt(v/bc2) + eps))
    """
    F = lambda a: np.asarray(a, dtype=np.float32)
    p, m, v = F(p), F(m), F(v)
    g = to_f32(gs_bf16, dtype) * F32(coef)
    if c.adamw:
        p = p - c.lr_wd * p
    else:
        g = g + c.wd * p
    m = c.b1 * m + c.omb1 * g
    v = c.b2 * v + c.omb2 * (g * g)
    mh = m / c.bc1
    vh = v / c.bc2
    den = np.sqrt(vh) + c.eps
    p = p - c.lr * (mh / den)
    return p, m, v, from_f32(p, dtype)


def adam_step(plan: Plan, sub_group: int, hp: dict, step: int, coef, skip: bool,
              st: State) -> None:
    """Update sub-group `sub_group` (-1: all) on every rank's shard and on the
    persistent parameters it contains ([ZeRO-3 chapter] §6.3: the step loops
    over sub-groups: clip, optimizer step, write back the 16-bit shard).
    Nothing changes when skip is set (non-finite gradient norm)."""
    if skip:
        return
    c = adam_consts(hp, step)
    groups = plan.sub_groups if sub_group == -1 else [plan.sub_groups[sub_group]]
    for g in groups:
        a, b = g.s_lo, g.s_hi
        if b > a:
            p, m, v, pb = adam_update(st.master[:, a:b], st.exp_avg[:, a:b],
                                      st.exp_avg_sq[:, a:b], st.grad_shards[:, a:b], coef, c,
                                      plan.dtype)
            st.master[:, a:b], st.exp_avg[:, a:b], st.exp_avg_sq[:, a:b] = p, m, v
            st.param_shards[:, a:b] = pb
        a, b = g.p_lo, g.p_hi
        if b > a:
            p, m, v, pb = adam_update(st.p_master[a:b], st.p_exp_avg[a:b],
                                      st.p_exp_avg_sq[a:b], st.persist_grads[a:b], coef, c,
                                      plan.dtype)
            st.p_master[a:b], st.p_exp_avg[a:b], st.p_exp_avg_sq[a:b] = p, m, v
            st.persist_params[a:b] = pb


# ---------------------------------------------------------------- A5 -----
def all_gather_coalesced(plan: Plan, params, param_shards: np.ndarray):
    """Gather a list of parameters into one flat buffer: sort by ds_id, lay
    the parameters back to back, each as its N shards in rank order, and
    return the flat buffer and each listed parameter's view offset (-1 for a
    persistent parameter, which is already whole) ([ZeRO-3 chapter] §5.2:
    all_gather_coalesced sorts by ds_id, packs one flat buffer, one
    collective, per-parameter views; §7: a wrong order is silently wrong)."""
    params = [int(i) for i in params]
    if len(set(params)) != len(params):
        raise ValueError("duplicate parameter in gather list")
    N = plan.group
    srt = sorted(params, key=lambda i: plan.params[i].ds_id)
    offs, off = {}, 0
    for i in srt:
        p = plan.params[i]
        if p.persistent:
            offs[i] = -1
        else:
            offs[i] = off
            off += N * p.ps
    flat = np.zeros(off, dtype=np.uint16)
    for i in srt:
        p = plan.params[i]
        if p.persistent:
            continue
        for r in range(N):
            flat[offs[i] + r * p.ps:offs[i] + (r + 1) * p.ps] = \
                param_shards[r, p.shard_off:p.shard_off + p.ps]
    return flat, [offs[i] for i in params]


def gather_model(plan: Plan, param_shards: np.ndarray) -> np.ndarray:
    """All gather buckets back to back: the model flat space."""
    parts = [all_gather_coalesced(plan, g.params, param_shards)[0]
             for g in plan.gather_buckets]
    return np.concatenate(parts) if parts else np.zeros(0, dtype=np.uint16)


# ------------------------------------------------------------ the step ---
def shard_step(plan: Plan, st: State, bucket_bufs, hp: dict, step: int,
               max_norm: float, scaler: LossScaler = None):
    """One step of the path: reduce-scatter every bucket, global norm and
    clip coefficient (unscaled by the loss scale when a scaler is given,
    which is then updated), Adam(W) over every sub-group, then the gathers
    the next forward pass performs.  bucket_bufs[b][k] is rank k's gradient
    buffer of bucket b."""
    for b in range(len(plan.reduce_buckets)):
        reduce_scatter(plan, b, bucket_bufs[b], st)
    if scaler is None:
        norm, coef, skip = grad_norm(plan, st, max_norm)
    else:
        norm, coef, skip = unscale_and_clip(plan, st, max_norm, scaler.scale)
        scaler.update(skip)
    adam_step(plan, -1, hp, step, coef, skip, st)
    return norm, coef, skip, gather_model(plan, st.param_shards)
