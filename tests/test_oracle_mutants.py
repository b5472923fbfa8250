"""Plant plausible mistakes in the oracle (on the CPU) and check that a pin
catches each one: evidence that the pins constrain every part of it."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import bf16 as obf16
from oracle import plan as oplan
from oracle import step as ostep
from tests import test_oracle_pins as pins

F32 = np.float32


def _rm_divisor(vals):
    vals = np.asarray(vals, dtype=np.uint16)
    s = np.zeros(vals.shape[1:], dtype=np.float32)
    for k in range(vals.shape[0]):
        s = s + ostep.bf16_to_f32(vals[k])
    return ostep.f32_to_bf16(s / F32(max(vals.shape[0] - 1, 1)))


def _rm_drop_last(vals):
    vals = np.asarray(vals, dtype=np.uint16)
    s = np.zeros(vals.shape[1:], dtype=np.float32)
    for k in range(vals.shape[0] - 1):
        s = s + ostep.bf16_to_f32(vals[k])
    return ostep.f32_to_bf16(s / F32(vals.shape[0]))


def _bf16_truncate(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _adam_eps_inside(p, m, v, gs, coef, c):
    p, m, v = (np.asarray(a, dtype=np.float32) for a in (p, m, v))
    g = ostep.bf16_to_f32(gs) * F32(coef)
    p = p - c.lr_wd * p
    m = c.b1 * m + c.omb1 * g
    v = c.b2 * v + c.omb2 * (g * g)
    den = np.sqrt(v / c.bc2 + c.eps)
    p = p - c.lr * ((m / c.bc1) / den)
    return p, m, v, ostep.f32_to_bf16(p)


def _adam_no_bias_correction(p, m, v, gs, coef, c):
    import dataclasses
    return _orig_adam(p, m, v, gs, coef, dataclasses.replace(c, bc1=F32(1), bc2=F32(1)))


def _norm_persistent_twice(plan, st, max_norm):
    st2 = ostep.State(**{k: getattr(st, k) for k in st.__dataclass_fields__})
    st2.persist_grads = np.concatenate([st.persist_grads, st.persist_grads])
    return _orig_norm(plan, st2, max_norm)


def _norm_no_min(plan, st, max_norm):
    norm, coef, skip = _orig_norm(plan, st, max_norm)
    if not skip and max_norm > 0:
        coef = F32(max_norm) / (norm + ostep.CLIP_EPS)
    return norm, coef, skip


def _gather_unsorted(plan, params, shards):
    N = plan.n_ranks
    offs, off = {}, 0
    for i in params:
        p = plan.params[i]
        offs[i] = -1 if p.persistent else off
        off += 0 if p.persistent else N * p.ps
    flat = np.zeros(off, dtype=np.uint16)
    for i in params:
        p = plan.params[i]
        if not p.persistent:
            for r in range(N):
                flat[offs[i] + r * p.ps:offs[i] + (r + 1) * p.ps] = \
                    shards[r, p.shard_off:p.shard_off + p.ps]
    return flat, [offs[i] for i in params]


_orig_norm = ostep.grad_norm
_orig_adam = ostep.adam_update


def _floor_ps_build(*a, **k):
    plan = _orig_build(*a, **k)
    for p in plan.params:
        if not p.persistent and p.numel:
            p.ps = max(p.numel // plan.n_ranks, 1)
    return plan


_orig_build = oplan.build_partition
_orig_unscale = ostep.unscale_and_clip


def _unscale_forgets_scale(plan, st, max_norm, scale):
    norm, coef, skip = _orig_unscale(plan, st, max_norm, scale)
    return norm, (coef * np.float32(scale) if not skip else coef), skip


_orig_counts = ostep.bucket_sq_counts


def _counts_skip_persistent(plan, bucket, rank_bufs):
    kept = [e for e in plan.reduce_buckets[bucket] if not plan.params[e.param].persistent]
    import dataclasses
    plan2 = dataclasses.replace(plan, reduce_buckets=[
        kept if b == bucket else ents for b, ents in enumerate(plan.reduce_buckets)])
    return _orig_counts(plan2, bucket, rank_bufs)


def _sumsq_float32(counts, dtype="bf16"):
    counts = np.asarray(counts)
    vals = ostep.to_f32(np.arange(1 << 15, dtype=np.uint16), dtype)
    tot = np.float32(0)
    for i in np.nonzero(counts)[0]:
        tot = tot + np.float32(counts[i]) * vals[i] * vals[i]
    return float(tot)


class _GreedyScaler(ostep.LossScaler):
    def update(self, overflow):
        if overflow:
            self.scale = max(self.scale / self.factor, self.min_scale)
        else:
            self.scale = self.scale * self.factor


def _fp16_pin_unscale():
    from tests import test_oracle_fp16 as f16
    f16.test_fp16_step_matches_textbook_adamw_on_unscaled_gradients()


def _fp16_pin_schedule():
    from tests import test_oracle_fp16 as f16
    f16.test_loss_scaler_schedule_by_hand()

MUTANTS = [
    ("divide by N-1", ostep, "reduce_mean_bf16", _rm_divisor,
     lambda: pins.test_rs_exact_small_values(4)),
    ("drop the last rank", ostep, "reduce_mean_bf16", _rm_drop_last,
     lambda: pins.test_rs_exact_small_values(8)),
    ("truncate instead of round", obf16, "f32_to_bf16", _bf16_truncate,
     pins.test_bf16_rne_matches_torch),
    ("eps inside the square root", ostep, "adam_update", _adam_eps_inside,
     lambda: pins.test_adam_matches_torch(1)),
    ("no bias correction", ostep, "adam_update", _adam_no_bias_correction,
     pins.test_adam_closed_form_constant_gradient),
    ("persistent counted twice", ostep, "grad_norm", _norm_persistent_twice,
     pins.test_norm_sharded_equals_unsharded),
    ("clip coefficient not capped at 1", ostep, "grad_norm", _norm_no_min,
     pins.test_clip_matches_torch),
    ("gather ignores ds_id order", ostep, "all_gather_coalesced", _gather_unsorted,
     pins.test_gather_order_independent_and_views),
    ("partition size rounded down", oplan, "build_partition", _floor_ps_build,
     lambda: pins.test_partition_bruteforce(3)),
    ("coefficient not unscaled", ostep, "unscale_and_clip", _unscale_forgets_scale,
     _fp16_pin_unscale),
    ("loss scale grows every good step", ostep, "LossScaler", _GreedyScaler,
     _fp16_pin_schedule),
    ("streamed norm leaves out persistent parameters", ostep, "bucket_sq_counts",
     _counts_skip_persistent, lambda: pins.test_streamed_norm_equals_whole_state_norm("tiny_thr100")),
    ("streamed sum of squares in float32", ostep, "sumsq_from_counts", _sumsq_float32,
     pins.test_sumsq_from_counts_is_exact),
]


@pytest.mark.parametrize("name,mod,attr,bad,pin", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_pin_catches_planted_mistake(monkeypatch, name, mod, attr, bad, pin):
    monkeypatch.setattr(mod, attr, bad)
    if mod is obf16:
        monkeypatch.setattr(pins, "f32_to_bf16", bad)
    if mod is oplan:
        monkeypatch.setattr(pins.oplan, "build_partition", bad)
    with pytest.raises((AssertionError, IndexError, ValueError)):
        pin()
