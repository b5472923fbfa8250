"""GPU parity of HSDP (shard within groups of G ranks, replicate across the
N/G groups): the grouped rank sum bit-exact against the oracle, whole steps,
fused == per-call chain, and G = N bit-identical to plain ZeRO-3."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

from oracle import step as ostep  # noqa: E402
from synth import workloads  # noqa: E402
from tests import gpu_harness as H  # noqa: E402

pytestmark = pytest.mark.gpu
HP = dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8, weight_decay=0.01, adamw=1,
          bias_correction=1)


def _ragged(seed, n=24):
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(0, 3000, size=n)] + [2501, 1]


CASES = {
    "tiny_n8_g2": dict(numel=workloads.tiny().numel, N=8, threshold=100, group=2),
    "ragged_n12_g3": dict(numel=_ragged(5), N=12, threshold=50, B=1000, G=5000, U=700, group=3),
    "ragged_n16_g4_fp16": dict(numel=_ragged(6), N=16, threshold=50, B=900, group=4,
                               dtype="fp16", log2_scale=-3),
    "many_small_n64_g8": dict(numel=workloads.many_small(30).numel, N=64, threshold=100_000,
                              group=8),
}


@pytest.fixture(params=list(CASES))
def case(request):
    return request.param


def test_hsdp_steps_vs_oracle(case):
    d = H.DevicePlan(**CASES[case])
    d.init_weights()
    assert d.info["shard_group_size"] == d.op.group
    for t in (1, 2):
        d.set_grads(300 + t, use_gpu_generator=case.startswith("many"))
        d.shard_step(HP, t, 1.0)
        prev = H.oracle_state(d.ost)
        norm, coef, skip, flat = ostep.shard_step(d.op, d.ost, d.grad_bufs, HP, t, 1.0)
        s = d.snapshot()
        assert np.array_equal(s["grad_shards"], d.ost.grad_shards)
        assert np.array_equal(s["persist_grads"], d.ost.persist_grads)
        assert abs(float(d.d_norm.np()[0]) - float(norm)) <= 1e-5 * float(norm)
        exact = H.same_bits(d.d_coef.np()[0], coef)
        H.assert_state(s, d.ost, prev, f"{case} step {t}", exact)
        H.assert_16bit(d.flat.u16(), flat, "gathered", d.dtype, exact)
    d.check_canaries()


def test_hsdp_fused_equals_unfused(case):
    a, b = H.DevicePlan(**CASES[case]), H.DevicePlan(**CASES[case])
    for d in (a, b):
        d.init_weights()
        d.set_grads(400, use_gpu_generator=case.startswith("many"))
    a.shard_step(HP, 1, 1.0)
    b.reduce_scatter_all_buckets(with_scratch=True)
    b.grad_norm(1.0, recompute=False)
    b.adam(HP, 1)
    b.gather_model_unfused(b.flat)
    xa, xb = a.snapshot(), b.snapshot()
    for k in xa:
        assert np.array_equal(xa[k].view(np.uint8), xb[k].view(np.uint8)), k
    assert np.array_equal(a.flat.u16(), b.flat.u16())


def test_group_equal_to_n_is_zero3():
    kw = dict(numel=_ragged(9), N=8, threshold=50, B=1200)
    a, b = H.DevicePlan(**kw), H.DevicePlan(**kw, group=8)
    for d in (a, b):
        d.init_weights()
        d.set_grads(11)
        d.shard_step(HP, 1, 1.0)
    xa, xb = a.snapshot(), b.snapshot()
    for k in xa:
        assert np.array_equal(xa[k].view(np.uint8), xb[k].view(np.uint8)), k
    assert np.array_equal(a.flat.u16(), b.flat.u16())


def test_hsdp_ranges_equal_per_bucket(case):
    """zs_reduce_scatter_range over random runs of buckets gives the
    per-bucket calls' bits (grouped sums, fp16 included), and the same norm
    partials."""
    import zero_sharded_optimizer_bucket_gb300 as zs
    a, b = H.DevicePlan(**CASES[case]), H.DevicePlan(**CASES[case])
    for d in (a, b):
        d.init_weights()
        d.set_grads(500, use_gpu_generator=case.startswith("many"))
    a.reduce_scatter_all_buckets(with_scratch=True)
    nb = len(b.op.reduce_buckets)
    rng = np.random.default_rng(nb + 1)
    cuts = sorted({0, nb, *[int(x) for x in rng.integers(0, nb + 1, size=min(nb, 4))]})
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        zs.zs_reduce_scatter_range(b.plan, lo, hi - lo, b.ptr_table[lo * b.N:],
                                   b.bufs["grad_shards"].ptr(), b.bufs["persist_grads"].ptr(),
                                   b.scratch.ptr())
    xa, xb = a.snapshot(), b.snapshot()
    for k in ("grad_shards", "persist_grads"):
        assert np.array_equal(xa[k], xb[k]), k
    for d in (a, b):
        d.grad_norm(1.0, recompute=False)
    assert H.same_bits(a.d_norm.np()[0], b.d_norm.np()[0])
    b.check_canaries()
