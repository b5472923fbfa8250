"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: the pages'
worked example and accounting (tests/golden), closed forms, invariants,
brute force on tiny inputs, or a library routine (torch's bfloat16 cast,
torch.optim.AdamW / Adam, torch.nn.utils.clip_grad_norm_, numpy.linalg.norm).
"""
from __future__ import annotations

import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

from oracle import plan as oplan
from oracle import step as ostep
from oracle.bf16 import bf16_to_f32, f32_to_bf16
from synth import philox
from tests import helpers

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, adamw=1,
          bias_correction=1)


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def torch_bf16_bits(x):
    t = torch.from_numpy(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------- bf16 ------
def test_bf16_rne_matches_torch():
    rng = np.random.default_rng(1)
    u = rng.integers(0, 2**32, size=200_000, dtype=np.uint64).astype(np.uint32)
    # ties with odd and even truncations, values next to ties, max finite
    special = []
    for t in [0x3F80, 0x3F81, 0x7F7F, 0x0001, 0x8001, 0xBF80, 0x0000, 0x7F7E]:
        for r in [0x7FFF, 0x8000, 0x8001, 0xFFFF, 0x0000]:
            special.append((t << 16) | r)
    special += [0x7F800000, 0xFF800000, 0x00000001, 0x80000001, 0x007FFFFF]
    u = np.concatenate([u, np.array(special, dtype=np.uint32)])
    x = u.view(np.float32)
    finite = ~np.isnan(x)
    ours = f32_to_bf16(x)
    ref = torch_bf16_bits(x)
    assert np.array_equal(ours[finite], ref[finite])
    assert np.all(np.isnan(bf16_to_f32(ours[~finite])))


def test_bf16_widen_exact_all_patterns():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = bf16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    same = (ours.view(np.uint32) == ref.view(np.uint32)) | (np.isnan(ours) & np.isnan(ref))
    assert same.all()


# ------------------------------------------------ worked example ---------
def test_worked_example():
    ex = golden("worked_example.json")
    N = ex["n_ranks"]
    plan = oplan.build_partition([len(ex["weights"])], N, threshold=0)
    W = np.array(ex["weights"], dtype=np.float32)
    st = ostep.partition(plan, W)
    # GPU r holds unit r+1
    for r in range(N):
        assert list(st.master[r, :plan.params[0].ps]) == ex["rank_holds"][r]
    # memory: one unit per rank instead of four
    assert plan.params[0].ps == ex["memory_units_per_rank_after_partition"]
    assert plan.params[0].numel == ex["memory_units_baseline"]
    # identical full gradients on every rank; reduce-scatter average
    g = f32_to_bf16(np.array(ex["full_grads_every_rank"], dtype=np.float32))
    bufs = helpers.bucket_buffers(plan, [g] * N)
    ostep.reduce_scatter(plan, 0, bufs[0], st)
    assert bf16_to_f32(st.grad_shards[0, 0]) == ex["rank0_reduced_grad"]
    for r in range(N):
        assert bf16_to_f32(st.grad_shards[r, 0]) == ex["full_grads_every_rank"][r]
    # all_gather(partition(x)) gives the weights back
    flat, views = ostep.all_gather_coalesced(plan, [0], st.param_shards)
    assert list(bf16_to_f32(flat)) == ex["weights"] and views == [0]
    # the global norm of the averaged gradient
    norm, coef, skip = ostep.grad_norm(plan, st, 1.0)
    assert not skip
    assert abs(float(norm) - math.sqrt(7.5)) <= 1e-6 * math.sqrt(7.5)
    assert abs(float(coef) - 1.0 / (math.sqrt(7.5) + 1e-6)) <= 1e-6
    # one local AdamW step with the workload hyper-parameters (no clipping):
    # at t=1, m^ = g and v^ = g^2, so p <- p(1 - lr*wd) - lr*g/(|g| + eps)
    ostep.adam_step(plan, -1, HP, 1, np.float32(1.0), False, st)
    for r, w in enumerate(ex["weights"]):
        gr = ex["full_grads_every_rank"][r]
        expect = w * (1 - 1e-3 * 0.01) - 1e-3 * gr / (abs(gr) + 1e-8)
        assert abs(float(st.master[r, 0]) - expect) <= 1e-6 * abs(expect)
    # master moves (0.99899, ...), the bf16 shard does not: 1, 2, 3, 4
    assert [float(bf16_to_f32(st.param_shards[r, 0])) for r in range(N)] == ex["weights"]


# ---------------------------------------------------------- plan ---------
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 6, 7, 8, 9, 16, 64])
def test_partition_bruteforce(N):
    """ps is the smallest equal split covering the tensor; (rank, offset) is
    a bijection onto [0, N*ps); partition then gather is the identity."""
    numel = list(range(0, 201))
    plan = oplan.build_partition(numel, N, threshold=0)
    for p in plan.params:
        n = p.numel
        assert p.ps * N >= n and (p.ps == 0 or (p.ps - 1) * N < n)
        assert p.pad == N * p.ps - n
        seen = set()
        for e in range(N * p.ps):
            r, col = oplan.owner(plan, p.index, e)
            assert 0 <= r < N and p.shard_off <= col < p.shard_off + p.ps
            seen.add((r, col))
        assert len(seen) == N * p.ps
    assert plan.padding_elems == sum(N * -(-n // N) - n for n in numel)
    W = philox.weight_f32(7, np.arange(plan.input_elems, dtype=np.uint64), 0.02)
    st = ostep.partition(plan, W)
    flat = ostep.gather_model(plan, st.param_shards)
    for p in plan.params:
        got = flat[p.flat_off:p.flat_off + p.numel]
        assert np.array_equal(got, f32_to_bf16(W[p.input_off:p.input_off + p.numel]))
        assert np.all(flat[p.flat_off + p.numel:p.flat_off + N * p.ps] == 0)


def _layout_checks(plan):
    N = plan.n_ranks
    prev_end = 0
    for i in plan.order:
        p = plan.params[i]
        assert p.persistent == (p.numel < plan.threshold)
        if not p.persistent:
            assert p.shard_off % 8 == 0 and p.shard_off >= prev_end
            prev_end = p.shard_off + p.ps
    assert plan.S % 8 == 0 and plan.S >= prev_end
    # input and flat offsets are plain running sums in ds_id order
    w = f = 0
    for i in plan.order:
        p = plan.params[i]
        assert p.input_off == w
        w += p.numel
        if not p.persistent:
            assert p.flat_off == f
            f += N * p.ps
    assert plan.flat_elems == f and plan.input_elems == w


def _bucket_checks(plan):
    B = plan.reduce_bucket_size
    covered = {i: [] for i in range(len(plan.params))}
    seq = []
    for b, ents in enumerate(plan.reduce_buckets):
        total = sum(e.e_hi - e.e_lo for e in ents)
        assert total <= B
        off = 0
        for e in ents:
            assert e.buf_off == off and e.buf_off % 8 == 0
            off += (e.e_hi - e.e_lo + 7) // 8 * 8
            covered[e.param].append((e.e_lo, e.e_hi))
            seq.append(e.param)
        assert plan.bucket_buf_elems[b] == off
        if len(ents) > 1:
            assert all(e.e_lo == 0 and e.e_hi == plan.params[e.param].numel for e in ents)
    for i, ranges in covered.items():
        n = plan.params[i].numel
        ranges.sort()
        assert ranges[0][0] == 0 and ranges[-1][1] == n
        for (a, b), (c, d) in zip(ranges, ranges[1:]):
            assert b == c
        if n > B:
            assert [b - a for a, b in ranges[:-1]] == [B] * (len(ranges) - 1)
    # bucket order follows ds_id order
    order_pos = {i: k for k, i in enumerate(plan.order)}
    assert [order_pos[i] for i in seq] == sorted(order_pos[i] for i in seq)
    # greedy maximality: a closed bucket could not take the next parameter
    for b in range(len(plan.reduce_buckets) - 1):
        ents, nxt = plan.reduce_buckets[b], plan.reduce_buckets[b + 1]
        n_next = plan.params[nxt[0].param].numel
        if n_next > B or plan.params[ents[-1].param].numel > B:
            continue
        assert sum(e.e_hi - e.e_lo for e in ents) + n_next > B


def _gather_and_subgroup_checks(plan):
    N, G, U = plan.n_ranks, plan.prefetch_bucket_size, plan.sub_group_size
    part = [i for i in plan.order if not plan.params[i].persistent]
    assert [i for g in plan.gather_buckets for i in g.params] == part
    for k, g in enumerate(plan.gather_buckets):
        size = sum(N * plan.params[i].ps for i in g.params)
        assert g.flat_elems == size and g.flat_off == plan.params[g.params[0]].flat_off
        assert size <= G or len(g.params) == 1
        if k + 1 < len(plan.gather_buckets):
            nxt = plan.gather_buckets[k + 1].params[0]
            assert size + N * plan.params[nxt].ps > G
    assert [i for s in plan.sub_groups for i in s.params] == list(plan.order)
    w = lambda i: plan.params[i].numel if plan.params[i].persistent else plan.params[i].ps
    for k, s in enumerate(plan.sub_groups):
        tot = sum(w(i) for i in s.params)
        assert tot <= U or len(s.params) == 1
        if k + 1 < len(plan.sub_groups):
            assert tot + w(plan.sub_groups[k + 1].params[0]) > U
    # sub-group column ranges tile the shard row and the persistent space
    assert plan.sub_groups == [] or plan.sub_groups[0].s_lo == 0
    for a, b in zip(plan.sub_groups, plan.sub_groups[1:]):
        assert a.s_hi == b.s_lo and a.p_hi == b.p_lo
    if plan.sub_groups:
        assert plan.sub_groups[-1].s_hi == plan.S and plan.sub_groups[-1].p_hi == plan.Pn_alloc


@pytest.mark.parametrize("seed", range(12))
def test_plan_invariants_random(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(0, 40))
    numel = [int(x) for x in rng.integers(0, 3000, size=n)]
    N = int(rng.choice([1, 2, 3, 4, 7, 8, 16, 64]))
    ds = [int(x) for x in rng.permutation(n) * 3 + 5]
    plan = oplan.build_partition(numel, N, threshold=int(rng.integers(0, 200)),
                                 reduce_bucket_size=int(rng.integers(1, 4000)),
                                 prefetch_bucket_size=int(rng.integers(1, 20000)),
                                 sub_group_size=int(rng.integers(1, 3000)), ds_id=ds)
    _layout_checks(plan)
    _bucket_checks(plan)
    _gather_and_subgroup_checks(plan)


def test_plan_defaults_and_workloads():
    from synth import workloads as wl
    w5 = wl.llama3_8b()
    plan = oplan.build_partition(w5.numel, w5.n_ranks, **{k: v for k, v in w5.config().items()
                                                          if k != "n_ranks" and k != "param_persistence_threshold"},
                                 threshold=w5.persistence_threshold)
    _bucket_checks(plan)
    _gather_and_subgroup_checks(plan)
    # the two 128256x4096 matrices are gathered alone; one sub-group
    assert len(plan.sub_groups) == 1
    assert sum(1 for g in plan.gather_buckets if len(g.params) == 1 and
               plan.params[g.params[0]].numel == 128256 * 4096) == 2
    # Llama-3-8B: norms (4096) persistent at threshold 1e5
    assert plan.Pn == 65 * 4096
    # the 16-layer workload is one sub-group under per-rank counting
    w4 = wl.llama3_layers()
    p4 = oplan.build_partition(w4.numel, w4.n_ranks)
    assert len(p4.sub_groups) == 1


def test_accounting_16_psi_over_n():
    acc = golden("accounting.json")
    # 16 bytes per element a rank holds: 2 (param) + 2 (grad) + 12 (state)
    assert acc["bytes_per_param"] == 2 + 2 + 12
    # unsharded 7.5B model: N = 1, nothing persistent (one flat parameter)
    plan = oplan.build_partition([acc["psi"]], 1, threshold=0)
    assert plan.bytes_per_rank() == acc["total_bytes"]
    assert 2 * plan.S_logical == acc["param_bytes"] == acc["grad_bytes"]
    assert 12 * plan.S_logical == acc["optimizer_bytes"]
    # 16 Psi / N when N divides every numel
    for N in [2, 4, 8, 16, 64]:
        numel = [N * k for k in (3, 1000, 12345, 7)]
        plan = oplan.build_partition(numel, N, threshold=0)
        assert plan.bytes_per_rank() * N == 16 * sum(numel)
        assert plan.padding_elems == 0
    # persistent parameters stay whole on every rank: 16 numel bytes each
    plan = oplan.build_partition([100, 5000], 4, threshold=1000)
    assert plan.bytes_per_rank() == 16 * 100 + 16 * 1250


def test_comm_volume_ratio():
    acc = golden("accounting.json")
    numel = [4096 * 4096, 1024 * 4096, 14336 * 4096]
    N = 8
    plan = oplan.build_partition(numel, N, threshold=0)
    psi = sum(numel)
    gathered = sum(g.flat_elems for g in plan.gather_buckets)   # one all-gather
    reduced = sum(e.e_hi - e.e_lo for b in plan.reduce_buckets for e in b)
    zero3 = 2 * gathered + reduced          # forward AG + backward AG + RS
    ddp = 2 * reduced                       # all-reduce = reduce-scatter + all-gather
    assert zero3 / psi == acc["comm_units_zero3"] and ddp / psi == acc["comm_units_ddp"]


# ---------------------------------------------------- reduce-scatter -----
@pytest.mark.parametrize("N", [1, 2, 3, 4, 5, 7, 8, 16, 64])
def test_rs_identical_grads_n_independent(N):
    """With identical rank gradients the mean is the gradient itself, bit
    for bit: k*g is exact in float32 for a bf16 g and k < 2^16."""
    numel = [37, 1000, 5, 64]
    plan = oplan.build_partition(numel, N, threshold=0, reduce_bucket_size=300)
    g = philox.grad_bf16(3, 0, np.arange(plan.input_elems, dtype=np.uint64), 1e-2, 0.05)
    bufs = helpers.bucket_buffers(plan, [g] * N)
    st = ostep.new_state(plan)
    for b in range(len(plan.reduce_buckets)):
        ostep.reduce_scatter(plan, b, bufs[b], st)
    full = ostep.gather_model(plan, st.grad_shards)
    for p in plan.params:
        assert np.array_equal(full[p.flat_off:p.flat_off + p.numel],
                              g[p.input_off:p.input_off + p.numel])


def _fraction_to_bf16(q: Fraction) -> int:
    """Round an exact rational to float32 (nearest-even), then to bf16
    (nearest-even), through torch's casts: the rounding points of the
    method (s / N in float32, then the bf16 cast)."""
    x32 = np.float32(float(q))      # q = sum/N with small N: never a double-rounding tie
    return int(torch_bf16_bits(np.array([x32]))[0])


@pytest.mark.parametrize("N", [2, 3, 4, 5, 6, 7, 8, 12, 16, 64])
def test_rs_exact_small_values(N):
    """Gradients that are small multiples of 2^-10 sum exactly in float32,
    so the result must be the exact mean rounded once to float32 and once
    to bf16; a dropped rank, a wrong divisor or a shifted index fails."""
    rng = np.random.default_rng(N)
    n = 257
    vals = rng.integers(-96, 97, size=(N, n))
    G = [f32_to_bf16((vals[k] * 2.0 ** -10).astype(np.float32)) for k in range(N)]
    plan = oplan.build_partition([n], N, threshold=0)
    bufs = helpers.bucket_buffers(plan, G)
    st = ostep.new_state(plan)
    ostep.reduce_scatter(plan, 0, bufs[0], st)
    flat = ostep.gather_model(plan, st.grad_shards)
    for i in range(n):
        exact = Fraction(int(vals[:, i].sum()), 1024 * N)
        assert int(flat[i]) == _fraction_to_bf16(exact), i


def test_rs_then_gather_equals_allreduce_mean():
    """reduce-scatter followed by all-gather gives the all-reduce mean of
    the full gradients, for buckets with chunks, several parameters and
    persistent parameters."""
    rng = np.random.default_rng(5)
    numel = [int(x) for x in rng.integers(1, 900, size=25)] + [2500, 3]
    N = 7
    plan = oplan.build_partition(numel, N, threshold=40, reduce_bucket_size=700,
                                 ds_id=list(rng.permutation(len(numel))))
    G = helpers.full_grads_from_pool(plan, 11, 1e-3, N)
    bufs = helpers.bucket_buffers(plan, G)
    st = ostep.new_state(plan)
    for b in range(len(plan.reduce_buckets)):
        ostep.reduce_scatter(plan, b, bufs[b], st)
    flat = ostep.gather_model(plan, st.grad_shards)
    # all-reduce mean over the unpartitioned tensors, one parameter at a time
    for p in plan.params:
        full = np.stack([G[k][p.input_off:p.input_off + p.numel] for k in range(N)])
        s = np.zeros(p.numel, dtype=np.float32)
        for k in range(N):
            s = s + torch.from_numpy(full[k].view(np.int16).copy()).view(torch.bfloat16).float().numpy()
        mean = torch_bf16_bits(s / np.float32(N))
        if p.persistent:
            got = st.persist_grads[p.persist_off:p.persist_off + p.numel]
        else:
            got = flat[p.flat_off:p.flat_off + p.numel]
        assert np.array_equal(got, mean), p.index


# ------------------------------------------------------------- norm ------
def _setup_random(seed=9, N=5, thr=30, B=600):
    rng = np.random.default_rng(seed)
    numel = [int(x) for x in rng.integers(1, 700, size=20)]
    plan = oplan.build_partition(numel, N, threshold=thr, reduce_bucket_size=B)
    G = helpers.full_grads_from_pool(plan, seed, 1e-2, N, outlier_frac=0.02)
    bufs = helpers.bucket_buffers(plan, G)
    st = ostep.partition(plan, philox.weight_f32(seed, np.arange(plan.input_elems,
                                                                 dtype=np.uint64), 0.02))
    for b in range(len(plan.reduce_buckets)):
        ostep.reduce_scatter(plan, b, bufs[b], st)
    full_mean = []
    for p in plan.params:
        s = np.zeros(p.numel, dtype=np.float32)
        for k in range(N):
            s = s + bf16_to_f32(G[k][p.input_off:p.input_off + p.numel])
        full_mean.append(bf16_to_f32(torch_bf16_bits(s / np.float32(N))))
    return plan, st, full_mean, G, bufs


def test_norm_sharded_equals_unsharded():
    plan, st, full_mean, _, _ = _setup_random()
    norm, coef, skip = ostep.grad_norm(plan, st, 1.0)
    ref = np.linalg.norm(np.concatenate(full_mean).astype(np.float64))
    assert not skip
    assert abs(float(norm) - ref) <= 1e-7 * ref
    # a rank-local norm differs from the global one ([Core flow] 坑 1)
    local = np.linalg.norm(bf16_to_f32(st.grad_shards[0]).astype(np.float64))
    assert abs(local - ref) > 1e-3 * ref


def test_clip_matches_torch():
    plan, st, full_mean, _, _ = _setup_random(seed=4)
    for max_norm in [0.05, 1.0, 1e9]:
        norm, coef, skip = ostep.grad_norm(plan, st, max_norm)
        ts = [torch.from_numpy(x.copy()).requires_grad_() for x in full_mean]
        for t, x in zip(ts, full_mean):
            t.grad = torch.from_numpy(x.copy())
        tn = torch.nn.utils.clip_grad_norm_(ts, max_norm)
        assert abs(float(tn) - float(norm)) <= 1e-6 * float(norm)
        for t, x in zip(ts, full_mean):
            ours = x * coef
            assert np.allclose(ours, t.grad.numpy(), rtol=2e-6, atol=0)


def test_norm_nonfinite_sets_skip():
    plan, st, _, _, _ = _setup_random(seed=2)
    st.grad_shards[1, 3] = 0x7F80          # +inf
    norm, coef, skip = ostep.grad_norm(plan, st, 1.0)
    assert skip and coef == 1.0
    before = st.master.copy()
    ostep.adam_step(plan, -1, HP, 1, coef, skip, st)
    assert np.array_equal(before, st.master)


# ------------------------------------------------ norm, streamed ---------
def _streamed(plan, bufs, max_norm, scale=1.0, order=None):
    order = range(len(bufs)) if order is None else order
    return ostep.grad_norm_streamed(plan, ((b, bufs[b]) for b in order), max_norm, scale)


def test_streamed_norm_worked_example():
    """[Grok blog] 具体例子: identical full gradients [0.5, 1, 1.5, 2] on the
    4 GPUs; the global norm of their mean is sqrt(7.5)."""
    ex = golden("worked_example.json")
    N = ex["n_ranks"]
    plan = oplan.build_partition([len(ex["weights"])], N, threshold=0)
    g = f32_to_bf16(np.array(ex["full_grads_every_rank"], dtype=np.float32))
    bufs = helpers.bucket_buffers(plan, [g] * N)
    norm, coef, skip = _streamed(plan, bufs, 1.0)
    assert not skip
    assert float(norm) == float(np.float32(math.sqrt(7.5)))
    assert abs(float(coef) - 1.0 / (math.sqrt(7.5) + 1e-6)) <= 1e-6


def test_streamed_norm_equals_unsharded_norm():
    """Bucket by bucket, the norm is that of the unpartitioned all-reduce
    mean (numpy.linalg.norm), for any order of the buckets."""
    plan, st, full_mean, G, bufs = _setup_random(seed=6)
    ref = np.linalg.norm(np.concatenate(full_mean).astype(np.float64))
    rng = np.random.default_rng(1)
    for order in (None, list(rng.permutation(len(bufs)))):
        norm, coef, skip = _streamed(plan, bufs, 1.0, order=order)
        assert not skip
        assert abs(float(norm) - ref) <= 1e-7 * ref


@pytest.mark.parametrize("kind", ["tiny_thr100", "ragged_chunks", "hsdp", "fp16", "many_small"])
def test_streamed_norm_equals_whole_state_norm(kind):
    """The same correctly rounded sum of squares as the norm over the
    reduce-scattered state: equal bits, clip coefficient included."""
    from synth import workloads
    rng = np.random.default_rng(3)
    dtype, scale, group = "bf16", 1.0, None
    if kind == "tiny_thr100":
        numel, N, kw = workloads.tiny().numel, 4, dict(threshold=100)
    elif kind == "ragged_chunks":
        numel = [int(x) for x in rng.integers(0, 3000, size=25)] + [2501, 1]
        N, kw = 7, dict(threshold=50, reduce_bucket_size=333)
    elif kind == "hsdp":
        numel = [int(x) for x in rng.integers(0, 3000, size=25)]
        N, kw, group = 12, dict(threshold=50, reduce_bucket_size=900), 3
    elif kind == "fp16":
        numel = [int(x) for x in rng.integers(0, 3000, size=25)]
        N, kw, dtype, scale = 16, dict(threshold=50, reduce_bucket_size=900), "fp16", 1024.0
    else:
        # the smaller tensors of the many-small list at N = 64: heavy padding
        numel = [x for x in workloads.many_small(200).numel if x < 20_000][:20]
        N, kw = 64, dict(threshold=2000, reduce_bucket_size=30_000)
    plan = oplan.build_partition(numel, N, dtype=dtype, shard_group_size=group, **kw)
    n = plan.input_elems
    if dtype == "fp16":
        G = [philox.grad_fp16(5, 0, np.arange(k * n, (k + 1) * n, dtype=np.uint64), -3)
             for k in range(N)]
    else:
        G = helpers.full_grads_from_pool(plan, 5, 1e-2, N, outlier_frac=0.01)
    bufs = helpers.bucket_buffers(plan, G)
    st = ostep.new_state(plan)
    for b in range(len(plan.reduce_buckets)):
        ostep.reduce_scatter(plan, b, bufs[b], st)
    for max_norm in (1.0, 0.0):
        a = ostep.unscale_and_clip(plan, st, max_norm, scale)
        b = _streamed(plan, bufs, max_norm, scale, order=list(rng.permutation(len(bufs))))
        assert a[2] == b[2] is False
        assert np.float32(a[0]).tobytes() == np.float32(b[0]).tobytes()
        assert np.float32(a[1]).tobytes() == np.float32(b[1]).tobytes()


def test_sumsq_from_counts_is_exact():
    """1 + 2^20 * (2^-30)^2 = 1 + 2^-40 needs 41 bits: exact in float64,
    lost by a float32 sum."""
    counts = np.zeros(1 << 15, dtype=np.int64)
    one = int(f32_to_bf16(np.array([1.0], np.float32))[0])
    tiny = int(f32_to_bf16(np.array([2.0 ** -30], np.float32))[0])
    counts[one] = 1
    counts[tiny] = 1 << 20
    assert ostep.sumsq_from_counts(counts) == 1.0 + 2.0 ** -40
    assert ostep.sumsq_from_counts(np.zeros(1 << 15, np.int64)) == 0.0


def test_streamed_norm_nonfinite_and_every_bucket_once():
    plan, st, full_mean, G, bufs = _setup_random(seed=8)
    bad = [[b.copy() for b in row] for row in bufs]
    e = plan.reduce_buckets[1][0]
    bad[1][2][e.buf_off] = 0x7F80          # +inf in rank 2's gradient
    norm, coef, skip = _streamed(plan, bad, 1.0)
    assert skip and coef == 1.0
    with pytest.raises(ValueError):
        _streamed(plan, bufs, 1.0, order=[0] + list(range(len(bufs))))
    with pytest.raises(ValueError):
        _streamed(plan, bufs, 1.0, order=list(range(1, len(bufs))))


# ------------------------------------------------------------- adam ------
@pytest.mark.parametrize("adamw", [1, 0])
def test_adam_matches_torch(adamw):
    """N = 1, coef = 1: the shard update is the textbook optimizer."""
    rng = np.random.default_rng(adamw)
    n = 4000
    p0 = (rng.standard_normal(n) * 0.02).astype(np.float32)
    hp = dict(HP, adamw=adamw)
    tp = torch.from_numpy(p0.copy()).requires_grad_()
    # the library's hyper-parameters are float32: hand torch the same values
    f = lambda x: float(np.float32(x))
    opt = (torch.optim.AdamW if adamw else torch.optim.Adam)(
        [tp], lr=f(hp["lr"]), betas=(f(hp["beta1"]), f(hp["beta2"])), eps=f(hp["eps"]),
        weight_decay=f(hp["weight_decay"]), foreach=False)
    p, m, v = p0.copy(), np.zeros(n, np.float32), np.zeros(n, np.float32)
    for t in range(1, 6):
        g = f32_to_bf16((rng.standard_normal(n) * 1e-3).astype(np.float32))
        tp.grad = torch.from_numpy(bf16_to_f32(g).copy())
        opt.step()
        p, m, v, _ = ostep.adam_update(p, m, v, g, np.float32(1.0), ostep.adam_consts(hp, t))
        st = opt.state[tp]
        # torch updates m with lerp (m + (1-b1)(g-m)) and divides by
        # sqrt(bc2) outside the square root: other rounding sequences of the
        # same formula, so the bound is relative to the array's scale
        for ours, ref in [(m, st["exp_avg"].numpy()), (v, st["exp_avg_sq"].numpy()),
                          (p, tp.detach().numpy())]:
            assert np.allclose(ours, ref, rtol=1e-6, atol=1e-6 * np.abs(ref).max())


def test_adam_closed_form_constant_gradient():
    """Constant g: m_t = (1-b1^t) g and v_t = (1-b2^t) g^2, so the bias
    corrected moments are g and g^2 and every step is
    p <- p (1 - lr wd) - lr g / (|g| + eps)."""
    g = np.array([1e-3, -2e-2, 0.5, -3.0, 1e-5], dtype=np.float32)
    gb = f32_to_bf16(g)
    gv = bf16_to_f32(gb).astype(np.float64)
    p = np.array([0.05, -0.3, 1.0, 2.0, -5.0], dtype=np.float32)   # no zero crossing
    ref = p.astype(np.float64)
    m = np.zeros(5, np.float32)
    v = np.zeros(5, np.float32)
    for t in range(1, 31):
        p, m, v, _ = ostep.adam_update(p, m, v, gb, np.float32(1.0), ostep.adam_consts(HP, t))
        ref = ref * (1 - 1e-3 * 0.01) - 1e-3 * gv / (np.abs(gv) + 1e-8)
        assert np.allclose(p, ref, rtol=2e-6, atol=0)


def test_adam_step1_invariant_to_gradient_scale():
    """At t = 1 the update is lr*sign(g) (for |g| >> eps), whatever the clip
    coefficient: clipping only matters from the second step on."""
    g = f32_to_bf16(np.array([1e-2, -3e-3, 0.25], dtype=np.float32))
    p = np.array([0.1, 0.2, -0.3], dtype=np.float32)
    z = np.zeros(3, np.float32)
    c = ostep.adam_consts(HP, 1)
    a = ostep.adam_update(p, z, z, g, np.float32(1.0), c)[0]
    b = ostep.adam_update(p, z, z, g, np.float32(0.125), c)[0]
    assert np.allclose(a, b, rtol=1e-6, atol=0)


def test_padding_stays_zero():
    plan, st, _, G, bufs = _setup_random(seed=12, N=8, thr=0)
    for t in range(1, 4):
        for b in range(len(plan.reduce_buckets)):
            ostep.reduce_scatter(plan, b, bufs[b], st)
        norm, coef, skip = ostep.grad_norm(plan, st, 1.0)
        ostep.adam_step(plan, -1, HP, t, coef, skip, st)
    mask = np.ones((plan.n_ranks, plan.S), dtype=bool)
    for p in plan.params:
        if p.persistent:
            continue
        for r in range(plan.n_ranks):
            n_valid = max(0, min(p.ps, p.numel - r * p.ps))
            mask[r, p.shard_off:p.shard_off + n_valid] = False
    for arr in [st.master, st.exp_avg, st.exp_avg_sq]:
        assert np.all(arr[mask] == 0)
    for arr in [st.param_shards, st.grad_shards]:
        assert np.all(arr[mask] == 0)


# ----------------------------------------------------------- gather ------
def test_gather_order_independent_and_views():
    rng = np.random.default_rng(3)
    numel = [int(x) for x in rng.integers(1, 500, size=15)]
    N = 6
    plan = oplan.build_partition(numel, N, threshold=60, ds_id=list(rng.permutation(15) * 2))
    W = philox.weight_f32(1, np.arange(plan.input_elems, dtype=np.uint64), 0.02)
    st = ostep.partition(plan, W)
    req = [int(x) for x in rng.permutation(15)[:11]]
    flat, views = ostep.all_gather_coalesced(plan, req, st.param_shards)
    flat2, views2 = ostep.all_gather_coalesced(plan, list(reversed(req)), st.param_shards)
    assert np.array_equal(flat, flat2) and views2 == list(reversed(views))
    for i, off in zip(req, views):
        p = plan.params[i]
        if p.persistent:
            assert off == -1
        else:
            assert np.array_equal(flat[off:off + p.numel],
                                  f32_to_bf16(W[p.input_off:p.input_off + p.numel]))
    # the packing follows ds_id order
    part = sorted([i for i in req if not plan.params[i].persistent],
                  key=lambda i: plan.params[i].ds_id)
    offs = [views[req.index(i)] for i in part]
    assert offs == sorted(offs)
    with pytest.raises(ValueError):
        ostep.all_gather_coalesced(plan, [1, 1], st.param_shards)


# --------------------------------------------------------- whole step ----
def test_step_n_independent_with_identical_grads():
    """Identical rank gradients: the gathered parameters after several steps
    do not depend on the number of ranks."""
    numel = [300, 17, 1024, 5, 999]
    results = []
    for N in [1, 4, 8, 64]:
        plan = oplan.build_partition(numel, N, threshold=10, reduce_bucket_size=500)
        W = philox.weight_f32(5, np.arange(plan.input_elems, dtype=np.uint64), 0.02)
        st = ostep.partition(plan, W)
        for t in range(1, 4):
            g = philox.grad_bf16(100 + t, 0, np.arange(plan.input_elems, dtype=np.uint64), 1e-2)
            bufs = helpers.bucket_buffers(plan, [g] * N)
            _, _, _, flat = ostep.shard_step(plan, st, bufs, HP, t, 1.0)
        full = []
        for p in plan.params:
            if p.persistent:
                full.append(st.persist_params[p.persist_off:p.persist_off + p.numel])
            else:
                full.append(flat[p.flat_off:p.flat_off + p.numel])
        results.append(np.concatenate(full))
    for r in results[1:]:
        assert np.array_equal(r, results[0])


def test_bucket_and_subgroup_sizes_do_not_change_results():
    numel = [300, 17, 1024, 5, 999, 2048]
    N = 4
    outs = []
    for B, U in [(5_000_000, 10**9), (100, 50), (1000, 300), (7, 1)]:
        plan = oplan.build_partition(numel, N, threshold=10, reduce_bucket_size=B,
                                     sub_group_size=U)
        W = philox.weight_f32(8, np.arange(plan.input_elems, dtype=np.uint64), 0.02)
        G = helpers.full_grads_from_pool(plan, 21, 1e-2, N)
        st = ostep.partition(plan, W)
        bufs = helpers.bucket_buffers(plan, G)
        norm, _, _, flat = ostep.shard_step(plan, st, bufs, HP, 1, 0.01)
        outs.append((norm, flat, st.master.copy()))
    for o in outs[1:]:
        assert o[0] == outs[0][0]
        assert np.array_equal(o[1], outs[0][1]) and np.array_equal(o[2], outs[0][2])
