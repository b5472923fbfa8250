"""GPU parity: every C-ABI call against the CPU oracle, element by element.

Cases span several tiles and ragged tails: the Tiny workload (two
persistence thresholds), ragged random lists with chunked parameters whose
shards are not 16-byte aligned, numel < N, N = 1, a reduced many-small list
at N = 64, and the empty plan.  Tolerances are listed in gpu_harness.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import zero_sharded_optimizer_bucket_gb300 as zs  # noqa: E402
from oracle import step as ostep  # noqa: E402
from synth import gpu as sgpu  # noqa: E402
from synth import philox, workloads  # noqa: E402
from tests import gpu_harness as H  # noqa: E402

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, adamw=1,
          bias_correction=1)


def _ragged(seed, n=30, N=7):
    rng = np.random.default_rng(seed)
    numel = [int(x) for x in rng.integers(0, 3000, size=n)] + [2501, 1]
    ds = [int(x) for x in rng.permutation(len(numel))]
    return dict(numel=numel, N=N, threshold=50, B=1000, G=5000, U=700, ds_id=ds, seed=seed)


CASES = {
    "tiny_thr0": dict(numel=workloads.tiny().numel, N=4, threshold=0, sigma=1e-3),
    "tiny_thr100": dict(numel=workloads.tiny().numel, N=4, threshold=100, sigma=1e-3),
    "ragged_n7": _ragged(3),
    "ragged_n16_chunks": dict(_ragged(4, n=20, N=16), B=333),
    "numel_lt_n": dict(numel=[1, 2, 3, 5, 0, 9, 17], N=16, threshold=0),
    "n1": dict(numel=[100, 7, 4099, 1], N=1, threshold=5, B=2048),
    "many_small_64": dict(numel=workloads.many_small(60).numel, N=64, threshold=100_000),
    # the largest rank count the library takes (ZS_MAX_RANKS): 256 rank
    # buffers per bucket, most parameters smaller than N
    "n256_max_ranks": dict(_ragged(9, n=14, N=256), B=4000, threshold=20),
    # partition sizes multiples of 8 and >= 1024: gathers into a 16-byte
    # aligned buffer take the bulk-copy path, many 32 KB chunks long; the
    # 70001-element parameter sends any request holding it to the other path
    "aligned_bulk": dict(numel=[65536, 131136, 8192, 192000, 500, 1048576, 70001], N=8,
                         threshold=1000, B=300_000),
}


def make(case, **over):
    kw = dict(CASES[case])
    kw.update(over)
    return H.DevicePlan(**kw)


@pytest.fixture(params=list(CASES))
def case(request):
    return request.param


# -------------------------------------------------------------------------
def test_generator_gpu_matches_cpu():
    n = 300_001
    t = torch.empty(n, dtype=torch.int16, device="cuda")
    sgpu.fill_grad_bf16(t, 12345, 77, 1e-3, outlier_frac=0.01)
    ref = philox.grad_bf16(77, 0, np.arange(12345, 12345 + n, dtype=np.uint64), 1e-3, 0.01)
    assert np.array_equal(t.cpu().numpy().view(np.uint16), ref)
    w = torch.empty(n, dtype=torch.float32, device="cuda")
    sgpu.fill_weight_f32(w, 2**33, 5, 0.02)
    ref = philox.weight_f32(5, np.arange(2**33, 2**33 + n, dtype=np.uint64), 0.02)
    assert np.array_equal(w.cpu().numpy().view(np.uint32), ref.view(np.uint32))


def test_partition(case):
    d = make(case)
    d.init_weights()
    s = d.snapshot()
    o = d.ost
    assert np.array_equal(s["master"], o.master)
    assert np.array_equal(s["param_shards"], o.param_shards)
    assert np.array_equal(s["p_master"], o.p_master)
    assert np.array_equal(s["persist_params"], o.persist_params)
    for k in ("exp_avg", "exp_avg_sq", "p_exp_avg", "p_exp_avg_sq"):
        assert not np.any(s[k])
    d.check_canaries()


def test_reduce_scatter(case):
    d = make(case)
    d.init_weights()
    d.set_grads(99, use_gpu_generator=(case == "many_small_64"))
    d.reduce_scatter_all_buckets()
    for b in range(len(d.op.reduce_buckets)):
        ostep.reduce_scatter(d.op, b, d.grad_bufs[b], d.ost)
    s = d.snapshot()
    assert np.array_equal(s["grad_shards"], d.ost.grad_shards)
    assert np.array_equal(s["persist_grads"], d.ost.persist_grads)
    d.check_canaries()


def test_grad_norm(case):
    d = make(case)
    d.init_weights()
    d.set_grads(7, use_gpu_generator=(case == "many_small_64"))
    d.reduce_scatter_all_buckets(with_scratch=True)
    for b in range(len(d.op.reduce_buckets)):
        ostep.reduce_scatter(d.op, b, d.grad_bufs[b], d.ost)
    for max_norm in (1.0, 0.01, 0.0):
        d.grad_norm(max_norm, recompute=False)
        n1, c1 = float(d.d_norm.np()[0]), float(d.d_coef.np()[0])
        d.grad_norm(max_norm, recompute=True)
        n2, c2 = float(d.d_norm.np()[0]), float(d.d_coef.np()[0])
        # partials from the reduce-scatter and recomputed ones: same bits
        assert (n1, c1) == (n2, c2)
        norm, coef, skip = ostep.grad_norm(d.op, d.ost, max_norm)
        assert abs(n1 - float(norm)) <= 1e-5 * float(norm)
        assert abs(c1 - float(coef)) <= 1e-5 * float(coef)
        assert int(d.d_flags.np()[0]) == 0 and not skip
    d.check_canaries()


def test_reduce_scatter_ranges(case):
    """zs_reduce_scatter_range over random runs of consecutive buckets: the
    reduced gradients bit for bit as the oracle's, the partial sums the
    same bits as the recomputed ones; ranges outside the plan are argument
    errors."""
    d = make(case)
    d.init_weights()
    d.set_grads(123, use_gpu_generator=(case == "many_small_64"))
    nb = len(d.op.reduce_buckets)
    rng = np.random.default_rng(nb)
    cuts = sorted({0, nb, *[int(x) for x in rng.integers(0, nb + 1, size=min(nb, 5))]})
    N = d.N
    for a, b in zip(cuts[:-1], cuts[1:]):
        zs.zs_reduce_scatter_range(d.plan, a, b - a, d.ptr_table[a * N:],
                                   d.bufs["grad_shards"].ptr(), d.bufs["persist_grads"].ptr(),
                                   d.scratch.ptr())
    zs.zs_reduce_scatter_range(d.plan, nb, 0, None, d.bufs["grad_shards"].ptr(),
                               d.bufs["persist_grads"].ptr(), None)          # empty: nothing
    for b in range(nb):
        ostep.reduce_scatter(d.op, b, d.grad_bufs[b], d.ost)
    s = d.snapshot()
    assert np.array_equal(s["grad_shards"], d.ost.grad_shards)
    assert np.array_equal(s["persist_grads"], d.ost.persist_grads)
    d.grad_norm(1.0, recompute=False)
    n1 = float(d.d_norm.np()[0])
    d.grad_norm(1.0, recompute=True)
    assert H.same_bits(n1, d.d_norm.np()[0])
    for first, n in [(-1, 1), (0, nb + 1), (nb, 1)]:
        with pytest.raises(zs.ZsError):
            zs.zs_reduce_scatter_range(d.plan, first, n, d.ptr_table,
                                       d.bufs["grad_shards"].ptr(),
                                       d.bufs["persist_grads"].ptr(), None)
    d.check_canaries()


@pytest.mark.parametrize("kind", ["huge", "tiny_tensor", "all_tiny"])
def test_grad_norm_out_of_range_values(kind):
    """Values whose squares leave float32's exact range send their tiles to
    the float64 sum: a few gradients of 2^70 (squares overflow float32), one
    whole tensor of 2^-100 (squares underflow), every gradient 2^-100.  The
    norm from the reduce-scatter's partials and the recomputed one keep the
    same bits, and both match the oracle's exactly rounded norm."""
    d = make("ragged_n16_chunks")
    d.init_weights()
    d.set_grads(55)
    big, tiny = 0x6280, 0x0D80              # bf16 bits of 2^70 and 2^-100
    host = d.pool.cpu().numpy().view(np.uint16)
    if kind == "huge":
        for b, k, i in [(0, 0, 3), (1, 5, 0), (len(d.grad_bufs) - 1, 15, 7)]:
            host[d.ptrs[b][k] // 2 - d.pool.data_ptr() // 2 + i] = big
    elif kind == "tiny_tensor":
        ent = d.op.reduce_buckets[2][0]
        for k in range(d.N):
            o = d.ptrs[2][k] // 2 - d.pool.data_ptr() // 2 + ent.buf_off
            host[o:o + ent.e_hi - ent.e_lo] = tiny
    else:
        host[:] = tiny
    d.pool.copy_(torch.from_numpy(host.view(np.int16).copy()))
    for b in range(len(d.grad_bufs)):
        for k in range(d.N):
            o = d.ptrs[b][k] // 2 - d.pool.data_ptr() // 2
            d.grad_bufs[b][k] = host[o:o + len(d.grad_bufs[b][k])].copy()
    d.reduce_scatter_all_buckets(with_scratch=True)
    for b in range(len(d.op.reduce_buckets)):
        ostep.reduce_scatter(d.op, b, d.grad_bufs[b], d.ost)
    assert np.array_equal(d.snapshot()["grad_shards"], d.ost.grad_shards)
    d.grad_norm(1.0, recompute=False)
    n1, c1 = float(d.d_norm.np()[0]), float(d.d_coef.np()[0])
    d.grad_norm(1.0, recompute=True)
    n2, c2 = float(d.d_norm.np()[0]), float(d.d_coef.np()[0])
    assert H.same_bits(n1, n2) and H.same_bits(c1, c2)
    norm, coef, skip = ostep.grad_norm(d.op, d.ost, 1.0)
    assert not skip and int(d.d_flags.np()[0]) == 0
    print(f"{kind}: norm {n1!r} (oracle {float(norm)!r})")
    assert abs(n1 - float(norm)) <= 1e-5 * float(norm)
    assert abs(c1 - float(coef)) <= 1e-5 * float(coef)
    assert zs.zs_device_wait_timeouts() == 0
    d.check_canaries()


def test_adam_isolated_bit_exact(case):
    """Adam on the device with the oracle's clip coefficient: the same fp32
    operations in the same order, so the same bits."""
    d = make(case)
    d.init_weights()
    for t in (1, 2, 3):
        d.set_grads(1000 + t, use_gpu_generator=(case == "many_small_64"))
        d.reduce_scatter_all_buckets(with_scratch=False)
        for b in range(len(d.op.reduce_buckets)):
            ostep.reduce_scatter(d.op, b, d.grad_bufs[b], d.ost)
        coef = np.float32(0.37) if t == 2 else np.float32(1.0)
        d.d_coef.t.fill_(float(coef))
        d.d_flags.t.zero_()
        for sg in range(len(d.op.sub_groups)):
            d.adam(HP, t, sub_group=sg)
        ostep.adam_step(d.op, -1, HP, t, coef, False, d.ost)
        s = d.snapshot()
        for k, ref in [("master", d.ost.master), ("exp_avg", d.ost.exp_avg),
                       ("exp_avg_sq", d.ost.exp_avg_sq), ("p_master", d.ost.p_master),
                       ("p_exp_avg", d.ost.p_exp_avg), ("p_exp_avg_sq", d.ost.p_exp_avg_sq)]:
            assert np.array_equal(s[k].view(np.uint32), ref.view(np.uint32)), k
        assert np.array_equal(s["param_shards"], d.ost.param_shards)
        assert np.array_equal(s["persist_params"], d.ost.persist_params)
    d.check_canaries()


def test_adam_l2_and_no_bias_correction():
    d = make("ragged_n7")
    d.init_weights()
    d.set_grads(5)
    d.reduce_scatter_all_buckets(with_scratch=False)
    for b in range(len(d.op.reduce_buckets)):
        ostep.reduce_scatter(d.op, b, d.grad_bufs[b], d.ost)
    hp = dict(HP, adamw=0, bias_correction=0, weight_decay=0.1)
    d.d_coef.t.fill_(1.0)
    d.d_flags.t.zero_()
    d.adam(hp, 4)
    ostep.adam_step(d.op, -1, hp, 4, np.float32(1.0), False, d.ost)
    s = d.snapshot()
    assert np.array_equal(s["master"].view(np.uint32), d.ost.master.view(np.uint32))
    assert np.array_equal(s["p_master"].view(np.uint32), d.ost.p_master.view(np.uint32))


def test_all_gather_coalesced(case):
    d = make(case)
    d.init_weights()
    rng = np.random.default_rng(17)
    n = len(d.numel)
    for trial in range(4):
        req = [int(x) for x in rng.permutation(n)[:max(1, int(rng.integers(1, n + 1)))]]
        flat_ref, views_ref = ostep.all_gather_coalesced(d.op, req, d.ost.param_shards)
        for lead in (0, 1, 3):       # output start 0, 2 or 6 bytes past a 16-byte boundary
            out = H.Guarded(len(flat_ref) + lead, torch.int16, d.dev)
            views = zs.zs_all_gather_coalesced(d.plan, req, d.bufs["param_shards"].ptr(),
                                               out.ptr() + 2 * lead, len(flat_ref))
            torch.cuda.synchronize()
            assert views == views_ref
            got = out.u16()[lead:]
            assert np.array_equal(got, flat_ref)
            assert not np.any(out.u16()[:lead])
            assert out.guards_ok()
    # too small a buffer and duplicates are argument errors
    if d.op.flat_elems > 0:
        with pytest.raises(zs.ZsError):
            part = [p.index for p in d.op.params if not p.persistent and p.ps > 0]
            zs.zs_all_gather_coalesced(d.plan, part, d.bufs["param_shards"].ptr(), d.flat.ptr(), 0)
    with pytest.raises(zs.ZsError):
        zs.zs_all_gather_coalesced(d.plan, [0, 0], d.bufs["param_shards"].ptr(), d.flat.ptr(),
                                   d.op.flat_elems)
    assert zs.zs_device_wait_timeouts() == 0


def test_fused_equals_unfused(case):
    """zs_shard_step and the per-call chain give the same bits."""
    a, b = make(case), make(case)
    for d in (a, b):
        d.init_weights()
    for t in (1, 2):
        for d in (a, b):
            d.set_grads(500 + t, use_gpu_generator=(case == "many_small_64"))
        a.shard_step(HP, t, 1.0)
        b.reduce_scatter_all_buckets(with_scratch=True)
        b.grad_norm(1.0, recompute=False)
        b.adam(HP, t)
        b.gather_model_unfused(b.flat)
        sa, sb = a.snapshot(), b.snapshot()
        for k in sa:
            assert np.array_equal(sa[k].view(np.uint8), sb[k].view(np.uint8)), k
        assert np.array_equal(a.flat.u16(), b.flat.u16())
        assert float(a.d_norm.np()[0]) == float(b.d_norm.np()[0])
    a.check_canaries()
    b.check_canaries()


def test_multistep_vs_oracle(case):
    """Whole steps (fused), state carried over, against the oracle's steps:
    the norm within 1e-5; the state, the parameters and the gathered replica
    bit for bit when the clip coefficients agree in bits, else within the
    per-element bound.  The many-small list runs its 5 steps."""
    d = make(case)
    d.init_weights()
    steps = 3 if case.startswith("tiny") else 5 if case == "many_small_64" else 2
    for t in range(1, steps + 1):
        d.set_grads(2000 + t, use_gpu_generator=(case == "many_small_64"))
        d.shard_step(HP, t, 1.0)
        prev = H.oracle_state(d.ost)
        norm, coef, skip, flat = ostep.shard_step(d.op, d.ost, d.grad_bufs, HP, t, 1.0)
        s = d.snapshot()
        assert np.array_equal(s["grad_shards"], d.ost.grad_shards)
        assert abs(float(d.d_norm.np()[0]) - float(norm)) <= 1e-5 * float(norm)
        exact = H.same_bits(d.d_coef.np()[0], coef)
        print(f"{case} step {t}: norm {float(d.d_norm.np()[0])!r} (oracle {float(norm)!r}), "
              f"coefficient bits {'equal' if exact else 'differ'}")
        H.assert_state(s, d.ost, prev, f"{case} step {t}", exact)
        H.assert_16bit(s["param_shards"], d.ost.param_shards, "param_shards", "bf16", exact)
        H.assert_16bit(s["persist_params"], d.ost.persist_params, "persist_params", "bf16", exact)
        H.assert_16bit(d.flat.u16(), flat, "gathered", "bf16", exact)
        # the gathered buffer is exactly the device's own shards, repacked
        part = ostep.gather_model(d.op, s["param_shards"])
        assert np.array_equal(d.flat.u16(), part)
    d.check_canaries()


def test_nonfinite_gradient_skips_update():
    d = make("ragged_n7")
    d.init_weights()
    d.set_grads(3)
    # an Inf in one rank's gradient of the first entry of bucket 0
    host = d.pool.cpu()
    host[0] = 0x7F80
    d.pool.copy_(host)
    before = d.snapshot()
    d.shard_step(HP, 1, 1.0)
    after = d.snapshot()
    assert int(d.d_flags.np()[0]) == zs.ZS_SKIP_NONFINITE
    assert not np.isfinite(float(d.d_norm.np()[0]))
    for k in ("master", "exp_avg", "exp_avg_sq", "param_shards", "p_master", "persist_params"):
        assert np.array_equal(before[k].view(np.uint8), after[k].view(np.uint8)), k


def test_bad_pointer_in_device_table_skips_update():
    """A misaligned rank pointer in the fused step's device table is never
    dereferenced: the kernel poisons the norm and the update is skipped."""
    d = make("tiny_thr0")
    d.init_weights()
    d.set_grads(3)
    tbl = d.ptr_table.cpu()
    tbl[1] += 2
    d.ptr_table.copy_(tbl)
    before = d.snapshot()
    d.shard_step(HP, 1, 1.0)
    after = d.snapshot()
    assert int(d.d_flags.np()[0]) == zs.ZS_SKIP_NONFINITE
    assert np.array_equal(before["master"], after["master"])


def test_empty_and_all_persistent_plans():
    d = H.DevicePlan([], 8)
    d.init_weights()
    d.set_grads(1)
    d.shard_step(HP, 1, 1.0)
    assert float(d.d_norm.np()[0]) == 0.0 and float(d.d_coef.np()[0]) == 1.0
    d = H.DevicePlan([10, 300, 5], 4, threshold=1_000)
    d.init_weights()
    d.set_grads(2)
    d.shard_step(HP, 1, 1.0)
    norm, coef, skip, flat = ostep.shard_step(d.op, d.ost, d.grad_bufs, HP, 1, 1.0)
    s = d.snapshot()
    assert np.array_equal(s["persist_grads"], d.ost.persist_grads)
    H.assert_f32_close(s["p_master"], d.ost.p_master, "p_master")
    d.check_canaries()


def test_argument_errors_enqueue_nothing():
    d = make("tiny_thr0")
    d.init_weights()
    d.set_grads(1)
    before = d.snapshot()
    bad = [d.ptrs[0][0] + 2] + d.ptrs[0][1:]
    with pytest.raises(zs.ZsError) as ei:
        zs.zs_reduce_scatter(d.plan, 0, bad, d.bufs["grad_shards"].ptr(),
                             d.bufs["persist_grads"].ptr(), None)
    assert ei.value.status == zs.ZS_EINVAL
    with pytest.raises(zs.ZsError):
        zs.zs_reduce_scatter(d.plan, 0, d.ptrs[0], d.bufs["grad_shards"].ptr() + 2,
                             d.bufs["persist_grads"].ptr(), None)
    with pytest.raises(zs.ZsError):
        zs.zs_adam_step(d.plan, 0, HP, 0, d.d_coef.ptr(), d.d_flags.ptr(), d.state)
    after = d.snapshot()
    for k in before:
        assert np.array_equal(before[k].view(np.uint8), after[k].view(np.uint8))


@pytest.mark.parametrize("case", ["ragged_n16_chunks", "many_small_64", "n256_max_ranks"])
def test_same_steps_twice_same_bits(case):
    """Determinism: the fused step run twice from the same start on the same
    gradients gives the same bits everywhere (the rank sum and the norm tree
    are fixed; no atomics decide an order)."""
    runs = []
    for _ in range(2):
        d = make(case)
        d.init_weights()
        for t in (1, 2):
            d.set_grads(900 + t, use_gpu_generator=(case == "many_small_64"))
            d.shard_step(HP, t, 1.0)
        runs.append((d.snapshot(), d.flat.u16().copy(), float(d.d_norm.np()[0])))
        d.check_canaries()
    (sa, fa, na), (sb, fb, nb) = runs
    for k in sa:
        assert np.array_equal(sa[k].view(np.uint8), sb[k].view(np.uint8)), k
    assert np.array_equal(fa, fb) and na == nb
