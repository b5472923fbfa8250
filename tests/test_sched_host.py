"""The gather scheduler on the host: the C++ scheduler (plan-only mode, no
device work) and the oracle's statement of the rules make the same
decisions, record for record, on random models, passes, orders and
configurations; invariants of the rules hold."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import plan as oplan
from oracle import sched as osched

zs = pytest.importorskip("zero_sharded_optimizer_bucket_gb300")


def _oracle_records(log):
    out = []
    for e in log:
        if e[0] == "gather":
            _, op, pos, items, waits = e
            out += [(1, pos, op, p, off, waits) for p, off in items]
        elif e[0] == "wait":
            _, pos, ops = e
            out += [(2, pos, op, -1, 0, 0) for op in ops] or [(2, pos, -1, -1, 0, 0)]
        else:
            _, pos, rel, ps = e
            out += [(3, pos, -1, p, 0, rel) for p in ps] or [(3, pos, -1, -1, 0, rel)]
    return out


def _model(rng, n_params, n_modules):
    numel = [int(x) for x in rng.integers(1, 3000, size=n_params)]
    mods = []
    for _ in range(n_modules):
        k = int(rng.integers(0, 5))
        mods.append([int(x) for x in rng.integers(0, n_params, size=k)])
    return numel, mods


def _run_both(plan_o, plan_c, mods, cfg, passes):
    """Drive both schedulers in lockstep; an arena failure of the oracle must
    be a ZS_ENOMEM of the library at the same fetch.  Returns (o, c, failed)."""
    o = osched.Scheduler(plan_o, mods, osched.SchedConfig(**cfg))
    c = zs.zs_sched_create(plan_c, mods, cfg)
    for order in passes:
        for m in order:
            try:
                o.fetch(m)
            except osched.ArenaFull:
                with pytest.raises(zs.ZsError) as ei:
                    zs.zs_sched_fetch(c, m)
                assert ei.value.status == zs.ZS_ENOMEM
                return o, c, True
            zs.zs_sched_fetch(c, m)
            o.release(m)
            zs.zs_sched_release(c, m)
        o.end_pass()
        zs.zs_sched_end_pass(c)
    return o, c, False


@pytest.mark.parametrize("seed", range(30))
def test_cpp_scheduler_equals_oracle(seed):
    rng = np.random.default_rng(seed)
    n_params, n_modules = int(rng.integers(3, 40)), int(rng.integers(1, 25))
    numel, mods = _model(rng, n_params, n_modules)
    N = int(rng.choice([1, 2, 4, 8]))
    thr = int(rng.integers(0, 300))
    plan_o = oplan.build_partition(numel, N, threshold=thr)
    cfg_c = zs.zs_default_config(N)
    cfg_c.param_persistence_threshold = thr
    plan_c = zs.zs_build_partition(cfg_c, numel)
    largest = max([sum(N * plan_o.params[p].ps for p in set(m)) for m in mods] + [1])
    cfg = dict(prefetch_bucket_size=int(rng.integers(1, 20000)),
               max_live_parameters=int(rng.integers(1, 40000)),
               max_reuse_distance=int(rng.integers(0, 20000)),
               arena_elems=int(largest * rng.uniform(1.0, 4.0)) + int(rng.integers(0, 50)))
    order = list(range(n_modules)) + list(reversed(range(n_modules)))     # forward + backward
    other = list(order)
    if len(other) > 2:
        i, j = rng.choice(len(other), 2, replace=False)
        other[i], other[j] = other[j], other[i]
    passes = [order, order, order, other, order, order, order[:-1], order, order]
    o, c, failed = _run_both(plan_o, plan_c, mods, cfg, passes)
    log = zs.zs_sched_log(c)
    if failed:                     # the failing fetch advanced the position on both sides
        log = log[:len(_oracle_records(o.log))]
    assert log == _oracle_records(o.log)


def test_invariants_on_a_transformer_like_model():
    """Every module's parameters are gathered before its compute, live
    elements stay within max_live_parameters plus one module, prefetch
    happens only with a complete trace, and everything is released at the
    end of a pass."""
    n_layers, N = 6, 4
    numel, mods = [5000], [[0]]
    for L in range(n_layers):
        base = len(numel)
        numel += [4096, 4096, 64, 8192, 8192, 64]
        mods.append([base, base + 1, base + 2])
        mods.append([base + 3, base + 4, base + 5])
    numel.append(5000)
    mods.append([len(numel) - 1, 0])                  # tied output projection
    plan_o = oplan.build_partition(numel, N, threshold=100)
    cfg_c = zs.zs_default_config(N)
    cfg_c.param_persistence_threshold = 100
    plan_c = zs.zs_build_partition(cfg_c, numel)
    cfg = dict(prefetch_bucket_size=20000, max_live_parameters=40000, max_reuse_distance=10000,
               arena_elems=80000)
    fwd = list(range(len(mods)))
    order = fwd + list(reversed(fwd))
    o, c, failed = _run_both(plan_o, plan_c, mods, cfg, [order, order, order])
    assert not failed
    log = zs.zs_sched_log(c)
    assert log == _oracle_records(o.log)
    st = zs.zs_sched_stats(c)
    assert st["passes"] == 3 and st["invalidations"] == 0
    assert st["max_live_elems"] <= 40000 + 2 * 8192 + 64
    assert st["elems_prefetched"] > 0
    # first pass: no prefetch (trace recording), so every gather is a fetch miss
    first_pass_gathers = [e for e in log if e[0] == 1 and e[1] < len(order)]
    assert first_pass_gathers
    # every module's parameters were gathered (or persistent) before its wait
    live = set()
    for e in log:
        if e[0] == 1:
            live.add(e[3])
        elif e[0] == 3 and e[3] >= 0:
            live.discard(e[3])
    assert not live


def _replay_arena(log, size, arena_elems):
    """Replays a log on an element-wise model of the arena: no gather lands
    on space a live parameter holds, and each gather waits for exactly the
    latest release that freed any element of its block (-1: never used)."""
    owner = np.full(arena_elems, -1, dtype=np.int64)      # live parameter per element
    freed = np.full(arena_elems, -1, dtype=np.int64)      # release that last freed it
    where = {}
    blocks = {}
    for kind, pos, op, p, off, aux in log:
        if kind == 1:
            lo, hi = off, off + size(p)
            assert hi <= arena_elems
            assert (owner[lo:hi] == -1).all(), ("gather onto live space", op, p)
            owner[lo:hi] = p
            where[p] = (lo, hi)
            b = blocks.setdefault(op, [aux, -1])
            b[1] = max(b[1], int(freed[lo:hi].max()))
        elif kind == 3 and p >= 0:
            lo, hi = where.pop(p)
            owner[lo:hi] = -1
            freed[lo:hi] = aux
    for op, (waits, need) in blocks.items():
        assert waits == need, (op, waits, need)


@pytest.mark.parametrize("seed", range(6))
def test_gathers_wait_for_exactly_the_releases_they_reuse(seed):
    rng = np.random.default_rng(100 + seed)
    N = int(rng.integers(2, 9))
    numel, mods = _model(rng, 40, 16)
    plan_o = oplan.build_partition(numel, N, threshold=int(rng.integers(0, 500)))
    cfg_c = zs.zs_default_config(N)
    cfg_c.param_persistence_threshold = plan_o.threshold
    plan_c = zs.zs_build_partition(cfg_c, numel)
    largest = max([sum(N * plan_o.params[p].ps for p in set(m)) for m in mods] + [1])
    cfg = dict(prefetch_bucket_size=int(rng.integers(0, 20000)), max_live_parameters=30000,
               max_reuse_distance=int(rng.integers(0, 20000)), arena_elems=3 * largest + 40000)
    fwd = list(range(len(mods)))
    order = fwd + list(reversed(fwd))
    o, c, failed = _run_both(plan_o, plan_c, mods, cfg, [order] * 4)
    assert not failed
    log = zs.zs_sched_log(c)
    assert log == _oracle_records(o.log)
    _replay_arena(log, lambda p: N * plan_o.params[p].ps, cfg["arena_elems"])


def test_gather_cta_cap_is_checked():
    numel = [5000, 7000]
    cfg_c = zs.zs_default_config(2)
    plan_c = zs.zs_build_partition(cfg_c, numel)
    base = dict(prefetch_bucket_size=0, max_live_parameters=100000, max_reuse_distance=0,
                arena_elems=20000)
    for bad in (-1, (1 << 20) + 1):
        with pytest.raises(zs.ZsError) as ei:
            zs.zs_sched_create(plan_c, [[0], [1]], dict(base, gather_ctas=bad))
        assert ei.value.status == zs.ZS_EINVAL
    assert zs.zs_sched_create(plan_c, [[0], [1]], dict(base, gather_ctas=152)).handle


def test_log_keeps_the_most_recent_records():
    numel = [5000, 7000, 3000]
    plan_c = zs.zs_build_partition(zs.zs_default_config(2), numel)
    base = dict(prefetch_bucket_size=8000, max_live_parameters=100000, max_reuse_distance=0,
                arena_elems=40000)
    mods = [[0], [1, 2], [0]]

    def run(limit):
        c = zs.zs_sched_create(plan_c, mods, dict(base, log_limit=limit))
        for _ in range(5):
            for m in range(3):
                zs.zs_sched_fetch(c, m)
                zs.zs_sched_release(c, m)
            zs.zs_sched_end_pass(c)
        return zs.zs_sched_log(c)

    full = run(-1)
    assert run(0) == full                      # the default keeps 2^20 records
    assert len(full) > 20
    assert run(7) == full[-7:]
    with pytest.raises(zs.ZsError) as ei:
        zs.zs_sched_create(plan_c, mods, dict(base, log_limit=-2))
    assert ei.value.status == zs.ZS_EINVAL
