"""The gather scheduler executed on two CUDA streams: at every module's
compute the module's parameters are in the arena with the right bytes,
although the compute stream is slowed down (busy kernels) so that an
ordering mistake — a compute reading before its gather finished, or a
gather overwriting space a later-released module still reads — would show.
The executed log equals the oracle's."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import zero_sharded_optimizer_bucket_gb300 as zs  # noqa: E402
from oracle import sched as osched  # noqa: E402
from oracle import step as ostep  # noqa: E402
from synth import gpu as sgpu  # noqa: E402
from tests import gpu_harness as H  # noqa: E402
from tests.test_sched_host import _oracle_records  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("seed,N,arena_factor,prefetch,ctas,aligned,group,dtype",
                         [(1, 4, 2.0, 30000, 0, False, 0, "bf16"),
                          (2, 8, 1.3, 5000, 1, False, 0, "bf16"),
                          (3, 3, 4.0, 100000, 3, False, 0, "bf16"),
                          (4, 16, 1.1, 0, 0, False, 0, "bf16"),
                          (5, 5, 1.5, 20000, 152, False, 0, "bf16"),
                          (6, 4, 1.5, 30000, 0, True, 0, "bf16"),
                          (7, 2, 1.3, 60000, 2, True, 0, "bf16"),
                          (8, 8, 1.5, 30000, 0, False, 2, "bf16"),
                          (9, 8, 1.5, 30000, 152, True, 4, "fp16")])
def test_scheduled_gathers_are_correct(seed, N, arena_factor, prefetch, ctas, aligned, group,
                                       dtype):
    """ctas caps the gather grid (strided loops cover the rest).  aligned:
    partition sizes are multiples of 8 and >= 1024, so every block of the
    arena starts on a 16-byte boundary and the gathers take the bulk-copy
    path.  group: HSDP shard groups (a gather assembles G shards)."""
    rng = np.random.default_rng(seed)
    G = group or N
    if aligned:
        numel = [8 * G * int(x) for x in rng.integers(128, 2500 // G + 130, size=30)]
    else:
        numel = [int(x) for x in rng.integers(1, 20000, size=30)]
    d = H.DevicePlan(numel, N, threshold=200, seed=seed, group=group, dtype=dtype)
    d.init_weights()
    expect = ostep.gather_model(d.op, d.ost.param_shards)
    mods = [[int(x) for x in rng.integers(0, 30, size=int(rng.integers(1, 5)))] for _ in range(14)]
    largest = max(sum(G * d.op.params[p].ps for p in set(m)) for m in mods)
    # the arena holds the live budget (plus padding) and the largest module,
    # with arena_factor of slack for fragmentation
    cfg = dict(prefetch_bucket_size=prefetch, max_live_parameters=60000,
               max_reuse_distance=20000, arena_elems=int((60000 + 2 * largest) * arena_factor))
    arena = torch.full((cfg["arena_elems"],), -1, dtype=torch.int16, device=d.dev)
    sched = zs.zs_sched_create(d.plan, mods, dict(cfg, gather_ctas=ctas), arena)
    oracle = osched.Scheduler(d.op, mods, osched.SchedConfig(**cfg))
    comp, gath = torch.cuda.Stream(), torch.cuda.Stream()
    sink = torch.zeros(4, device=d.dev)
    order = list(range(len(mods))) + list(reversed(range(len(mods))))
    for _ in range(3):
        for m in order:
            zs.zs_sched_fetch(sched, m, d.bufs["param_shards"].ptr(), comp, gath)
            oracle.fetch(m)
            sgpu.busy(20000, 152, sink, comp, 256)       # slow compute before reading
            views = {}
            for p in set(mods[m]):
                off = zs.zs_sched_param_offset(sched, p)
                q = d.op.params[p]
                if q.persistent:
                    assert off == -1
                    continue
                with torch.cuda.stream(comp):
                    views[p] = arena[off:off + q.numel].clone()
            zs.zs_sched_release(sched, m, comp)
            oracle.release(m)
            comp.synchronize()
            for p, v in views.items():
                q = d.op.params[p]
                got = v.cpu().numpy().view(np.uint16)
                assert np.array_equal(got, expect[q.flat_off:q.flat_off + q.numel]), (m, p)
        zs.zs_sched_end_pass(sched, comp)
        oracle.end_pass()
    torch.cuda.synchronize()
    assert zs.zs_device_wait_timeouts() == 0
    assert zs.zs_sched_log(sched) == _oracle_records(oracle.log)
    st = zs.zs_sched_stats(sched)
    if prefetch:
        assert st["elems_prefetched"] > 0
    d.check_canaries()


def test_shards_rewritten_between_passes_are_gathered():
    """The caller rewrites the parameter shards on the compute stream between
    passes, behind a long kernel; every gather of the next pass must read
    the new shards (the first fetch of a pass waits for the compute
    stream)."""
    rng = np.random.default_rng(21)
    N = 4
    numel = [8 * N * int(x) for x in rng.integers(200, 2000, size=12)]
    d = H.DevicePlan(numel, N, threshold=100, seed=21)
    d.init_weights()
    first = ostep.gather_model(d.op, d.ost.param_shards)
    mods = [[0, 1], [2], [3, 4, 5], [6], [7, 8], [9, 10, 11], [0, 4]]
    largest = max(sum(N * d.op.params[p].ps for p in set(m)) for m in mods)
    cfg = dict(prefetch_bucket_size=200000, max_live_parameters=10**7, max_reuse_distance=0,
               arena_elems=int(sum(N * p.ps for p in d.op.params) + 2 * largest), gather_ctas=152)
    arena = torch.full((cfg["arena_elems"],), -1, dtype=torch.int16, device=d.dev)
    sched = zs.zs_sched_create(d.plan, mods, cfg, arena)
    comp, gath = torch.cuda.Stream(), torch.cuda.Stream()
    sink = torch.zeros(4, device=d.dev)
    # new weights for the second pass, partitioned on the compute stream
    W2 = np.asarray(rng.standard_normal(d.op.input_elems), dtype=np.float32)
    W2d = torch.from_numpy(W2).to(d.dev)
    second = ostep.gather_model(d.op, ostep.partition(d.op, W2).param_shards)
    torch.cuda.synchronize()

    def one_pass(expect):
        for m in range(len(mods)):
            zs.zs_sched_fetch(sched, m, d.bufs["param_shards"].ptr(), comp, gath)
            views = {}
            for p in set(mods[m]):
                off = zs.zs_sched_param_offset(sched, p)
                q = d.op.params[p]
                with torch.cuda.stream(comp):
                    views[p] = arena[off:off + q.numel].clone()
            zs.zs_sched_release(sched, m, comp)
            comp.synchronize()
            for p, v in views.items():
                q = d.op.params[p]
                assert np.array_equal(v.cpu().numpy().view(np.uint16),
                                      expect[q.flat_off:q.flat_off + q.numel]), (m, p)
        zs.zs_sched_end_pass(sched, comp)

    one_pass(first)                     # records the trace
    sgpu.busy(3_000_000, 152, sink, comp, 32)   # a long step on the compute stream ...
    zs.zs_partition(d.plan, W2d, d.state, comp)  # ... that rewrites the shards
    one_pass(second)                    # prefetching pass: must see the new shards
    with pytest.raises(zs.ZsError) as ei:   # the streams are fixed
        zs.zs_sched_fetch(sched, 0, d.bufs["param_shards"].ptr(), gath, comp)
    assert ei.value.status == zs.ZS_EINVAL
    torch.cuda.synchronize()
    assert zs.zs_device_wait_timeouts() == 0
    d.check_canaries()
