"""Pins of the oracle's HSDP mode (shard_group_size G < N): reduction to
ZeRO-3 when G = N and to the flat rank-order mean when G = 1 (DDP), exact
means on exactly summable inputs, identical-gradient invariance, the
16Ψ/G accounting, a hand-worked case where the group order matters, and the
1-ulp bound between grouped and flat orders."""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import plan as oplan
from oracle import step as ostep
from oracle.bf16 import bf16_to_f32, f32_to_bf16
from synth import philox
from tests import helpers

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, adamw=1,
          bias_correction=1)


def _run(numel, N, G, steps=2, seed=3):
    plan = oplan.build_partition(numel, N, threshold=20, reduce_bucket_size=700,
                                 shard_group_size=G)
    st = ostep.partition(plan, philox.weight_f32(seed, np.arange(plan.input_elems, dtype=np.uint64), 0.02))
    outs = []
    for t in range(1, steps + 1):
        G_ = helpers.full_grads_from_pool(plan, seed * 10 + t, 1e-2, N)
        bufs = helpers.bucket_buffers(plan, G_)
        norm, coef, skip, flat = ostep.shard_step(plan, st, bufs, HP, t, 1.0)
        outs.append((norm, flat.copy()))
    return plan, st, outs


def _full(plan, flat, st):
    parts = []
    for p in plan.params:
        if p.persistent:
            parts.append(st.persist_params[p.persist_off:p.persist_off + p.numel])
        else:
            parts.append(flat[p.flat_off:p.flat_off + p.numel])
    return np.concatenate(parts)


NUMEL = [300, 17, 1024, 5, 999, 2048, 1]


def test_group_equal_to_n_is_zero3():
    p1, s1, o1 = _run(NUMEL, 8, None)
    p2, s2, o2 = _run(NUMEL, 8, 8)
    assert p1.S == p2.S and p1.flat_elems == p2.flat_elems and p2.group == 8
    for (n1, f1), (n2, f2) in zip(o1, o2):
        assert n1 == n2 and np.array_equal(f1, f2)
    assert np.array_equal(s1.master, s2.master)


def test_group_of_one_is_ddp_flat_mean():
    """G = 1: every rank holds every parameter whole (ps = numel, no
    padding) and the grouped sum is the flat rank-order sum, so the result
    equals ZeRO-3 over the same N ranks, parameter by parameter."""
    p1, s1, o1 = _run(NUMEL, 6, None)
    p2, s2, o2 = _run(NUMEL, 6, 1)
    assert all(p.ps == p.numel and p.pad == 0 for p in p2.params if not p.persistent)
    for (n1, f1), (n2, f2) in zip(o1, o2):
        assert n1 == n2
        assert np.array_equal(_full(p1, f1, s1), _full(p2, f2, s2))


@pytest.mark.parametrize("N,G", [(4, 2), (8, 2), (8, 4), (12, 3), (16, 4), (64, 8)])
def test_exact_mean_on_exactly_summable_inputs(N, G):
    rng = np.random.default_rng(N * 100 + G)
    vals = rng.integers(-96, 97, size=(N, 77))
    Gr = [f32_to_bf16((vals[k] * 2.0 ** -10).astype(np.float32)) for k in range(N)]
    plan = oplan.build_partition([77], N, threshold=0, shard_group_size=G)
    st = ostep.new_state(plan)
    ostep.reduce_scatter(plan, 0, helpers.bucket_buffers(plan, Gr)[0], st)
    flat = ostep.gather_model(plan, st.grad_shards)
    for i in range(77):
        exact = Fraction(int(vals[:, i].sum()), 1024 * N)
        ref = torch.tensor([float(np.float32(float(exact)))]).to(torch.bfloat16).view(torch.int16).item()
        assert int(flat[i]) == (ref & 0xFFFF)
    # identical rank gradients give the gradient back
    g = philox.grad_bf16(2, 0, np.arange(77, dtype=np.uint64), 1e-2)
    st = ostep.new_state(plan)
    ostep.reduce_scatter(plan, 0, helpers.bucket_buffers(plan, [g] * N)[0], st)
    assert np.array_equal(ostep.gather_model(plan, st.grad_shards)[:77], g)


def test_accounting_16_psi_over_g():
    for N, G in [(8, 2), (16, 4), (64, 8)]:
        numel = [G * k for k in (3, 1000, 12345)]
        plan = oplan.build_partition(numel, N, threshold=0, shard_group_size=G)
        assert plan.bytes_per_rank() * G == 16 * sum(numel)


def test_group_order_by_hand():
    """Ranks hold 2^24, 1, 1, -2^24 (exact in bf16).  Flat order:
    2^24 + 1 = 2^24 (rounded), + 1 = 2^24, - 2^24 = 0: mean 0.  Groups of
    two: (2^24 + 1) = 2^24 and (1 - 2^24) = -16777215 exactly, summed: 1,
    mean 0.25."""
    vals = np.array([[2.0 ** 24], [1.0], [1.0], [-(2.0 ** 24)]], dtype=np.float32)
    u = f32_to_bf16(vals)
    assert float(bf16_to_f32(ostep.reduce_mean_groups(u, 4)[0])) == 0.0
    assert float(bf16_to_f32(ostep.reduce_mean_groups(u, 2)[0])) == 0.25


def test_grouped_and_flat_within_one_bf16_ulp():
    rng = np.random.default_rng(1)
    # a wide exponent spread, so that float32 sums round and the order shows
    x = rng.standard_normal((16, 20000)) * 10.0 ** rng.uniform(-4, 4, (16, 20000))
    u = f32_to_bf16(x.astype(np.float32))
    a = bf16_to_f32(ostep.reduce_mean_groups(u, 4)).astype(np.float64)
    b = bf16_to_f32(ostep.reduce_mean_groups(u, 16)).astype(np.float64)
    ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(b), 2.0 ** -126))) - 7)
    assert np.all(np.abs(a - b) <= ulp)
    assert np.any(a != b)        # the order is visible in the last bit somewhere


def test_bad_group_size():
    with pytest.raises(ValueError):
        oplan.build_partition([10], 8, shard_group_size=3)
