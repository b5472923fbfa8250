"""Pins of the oracle's fp16 mode: binary16 casts against torch, the rank
mean on exact inputs, unscale-and-clip against numpy / torch on the unscaled
gradients, the dynamic loss-scale schedule on a hand-worked sequence, and a
whole fp16 step against torch.optim.AdamW on the unscaled gradients."""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import plan as oplan
from oracle import step as ostep
from oracle.fp16 import f32_to_fp16, fp16_to_f32
from synth import philox
from tests import helpers

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, adamw=1,
          bias_correction=1)


def torch_half_bits(x):
    return torch.from_numpy(np.asarray(x, np.float32)).half().view(torch.int16).numpy().view(np.uint16)


def test_fp16_casts_match_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100_000).astype(np.float32) * 10.0 ** rng.integers(-9, 6, 100_000),
                        np.array([65504, 65519.99, 65520, 1e6, -7e4, 2.0 ** -24, 2.0 ** -25,
                                  3 * 2.0 ** -26, 0.0, -0.0, np.inf, -np.inf], np.float32)]).astype(np.float32)
    assert np.array_equal(f32_to_fp16(x), torch_half_bits(x))
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = fp16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.float16).float().numpy()
    assert np.array_equal(ours.view(np.uint32)[~np.isnan(ref)], ref.view(np.uint32)[~np.isnan(ref)])
    assert np.all(np.isnan(ours[np.isnan(ref)]))


def test_fp16_generator_values_are_exact():
    g = philox.grad_fp16(3, 0, np.arange(50_000, dtype=np.uint64), -4, 0.01, 20)
    v = fp16_to_f32(g)
    finite = np.isfinite(v)
    assert finite.mean() < 1.0                   # some outliers overflow on purpose
    k = v[finite] * 16.0
    assert np.all(k[np.abs(k) < 2048] == np.round(k[np.abs(k) < 2048]))


@pytest.mark.parametrize("N", [2, 3, 4, 7, 16, 64])
def test_fp16_rank_mean_exact(N):
    rng = np.random.default_rng(N)
    vals = rng.integers(-300, 301, size=(N, 129))
    G = [f32_to_fp16((vals[k] * 2.0 ** -6).astype(np.float32)) for k in range(N)]
    plan = oplan.build_partition([129], N, threshold=0, dtype="fp16")
    st = ostep.new_state(plan)
    ostep.reduce_scatter(plan, 0, helpers.bucket_buffers(plan, G)[0], st)
    flat = ostep.gather_model(plan, st.grad_shards)
    for i in range(129):
        exact = Fraction(int(vals[:, i].sum()), 64 * N)
        assert int(flat[i]) == int(torch_half_bits(np.array([np.float32(float(exact))]))[0])
    # identical rank gradients give the gradient back
    g = philox.grad_fp16(5, 0, np.arange(129, dtype=np.uint64), -3)
    st = ostep.new_state(plan)
    ostep.reduce_scatter(plan, 0, helpers.bucket_buffers(plan, [g] * N)[0], st)
    assert np.array_equal(ostep.gather_model(plan, st.grad_shards)[:129], g)


def _fp16_setup(scale_log2=10, N=5):
    rng = np.random.default_rng(2)
    numel = [int(x) for x in rng.integers(1, 600, size=12)]
    plan = oplan.build_partition(numel, N, threshold=20, reduce_bucket_size=500, dtype="fp16")
    G = [philox.grad_fp16(10 + k, 0, np.arange(plan.input_elems, dtype=np.uint64), scale_log2 - 12)
         for k in range(N)]
    st = ostep.partition(plan, philox.weight_f32(1, np.arange(plan.input_elems, dtype=np.uint64), 0.02))
    bufs = helpers.bucket_buffers(plan, G)
    for b in range(len(plan.reduce_buckets)):
        ostep.reduce_scatter(plan, b, bufs[b], st)
    return plan, st, bufs, G


def test_unscale_and_clip_against_unscaled_gradients():
    plan, st, _, G = _fp16_setup()
    S = 1024.0
    mean = []
    for p in plan.params:
        s = np.zeros(p.numel, np.float32)
        for k in range(plan.n_ranks):
            s = s + fp16_to_f32(G[k][p.input_off:p.input_off + p.numel])
        mean.append(fp16_to_f32(f32_to_fp16(s / np.float32(plan.n_ranks))) / np.float32(S))
    true = np.concatenate(mean).astype(np.float64)
    for max_norm in (1e-4, 1.0, 0.0):
        norm, coef, skip = ostep.unscale_and_clip(plan, st, max_norm, S)
        assert not skip
        assert abs(float(norm) - np.linalg.norm(true)) <= 1e-6 * np.linalg.norm(true)
        ts = [torch.from_numpy(m.copy()).requires_grad_() for m in mean]
        for t, m in zip(ts, mean):
            t.grad = torch.from_numpy(m.copy())
        if max_norm > 0:
            torch.nn.utils.clip_grad_norm_(ts, max_norm)
        for t, m, p in zip(ts, mean, plan.params):
            stored = m * np.float32(S)       # the stored (scaled) gradient, exact
            assert np.allclose(stored * coef, t.grad.numpy(), rtol=2e-6, atol=0)
    # scale 1 is the plain gradient norm
    assert ostep.unscale_and_clip(plan, st, 1.0, 1.0) == ostep.grad_norm(plan, st, 1.0)


def test_loss_scaler_schedule_by_hand():
    sc = ostep.LossScaler(scale=2.0 ** 16, factor=2.0, min_scale=2.0 ** 14, window=3)
    seq = [False, False, False, True, False, True, True, True, False, False, False]
    want = [2 ** 16, 2 ** 16, 2 ** 17, 2 ** 16, 2 ** 16, 2 ** 15, 2 ** 14, 2 ** 14, 2 ** 14,
            2 ** 14, 2 ** 15]
    got = []
    for ov in seq:
        sc.update(ov)
        got.append(sc.scale)
    assert got == [float(x) for x in want]


def test_fp16_step_matches_textbook_adamw_on_unscaled_gradients():
    """N = 1, scale 2^10: the stored fp16 gradient is exactly S times a value
    g, and coef = 1/S restores g exactly, so the step is AdamW on g."""
    n, S = 3000, 1024.0
    plan = oplan.build_partition([n], 1, threshold=0, dtype="fp16")
    W = philox.weight_f32(4, np.arange(n, dtype=np.uint64), 0.02)
    st = ostep.partition(plan, W)
    f = lambda x: float(np.float32(x))
    tp = torch.from_numpy(fp16_to_f32(f32_to_fp16(W)).copy()).requires_grad_()
    st.master[:] = tp.detach().numpy()          # start both from the fp16-rounded weights
    opt = torch.optim.AdamW([tp], lr=f(1e-3), betas=(f(0.9), f(0.999)), eps=f(1e-8),
                            weight_decay=f(0.01), foreach=False)
    scaler = ostep.LossScaler(scale=S, window=10 ** 9)
    for t in range(1, 4):
        g = philox.grad_fp16(20 + t, 0, np.arange(n, dtype=np.uint64), -2)   # scaled gradient
        bufs = helpers.bucket_buffers(plan, [g])
        ostep.shard_step(plan, st, bufs, HP, t, 0.0, scaler)
        tp.grad = torch.from_numpy(fp16_to_f32(g) / np.float32(S))
        opt.step()
        # Adam's update hardly depends on the gradient's scale, its moments do
        tst = opt.state[tp]
        for ours, ref in [(st.master[0, :n], tp.detach().numpy()),
                          (st.exp_avg[0, :n], tst["exp_avg"].numpy()),
                          (st.exp_avg_sq[0, :n], tst["exp_avg_sq"].numpy())]:
            assert np.allclose(ours, ref, rtol=1e-6, atol=1e-6 * np.abs(ref).max())


def test_fp16_overflow_skips_and_halves_the_scale():
    plan, st, bufs, G = _fp16_setup()
    bufs[0][1][0] = 0x7C00                      # +inf in rank 1's first gradient
    before = st.master.copy()
    scaler = ostep.LossScaler(scale=1024.0, window=5)
    norm, coef, skip, _ = ostep.shard_step(plan, st, bufs, HP, 1, 1.0, scaler)
    assert skip and scaler.scale == 512.0 and scaler.good == 0
    assert np.array_equal(before, st.master)
