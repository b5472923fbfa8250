"""zs_grad_norm_noalloc: the gradient norm for callers that cannot allocate
device memory (a plugin handed only its inputs and outputs by a host
framework that owns every allocation, or a step loop that must keep
cudaMalloc and its device-wide synchronisation out).  It must give what
zs_grad_norm with a caller scratch buffer gives, call after call, although
every call reuses the one scratch array built into the library.

This file is collected last so that a run stopping at the first failure
has run every other test before it."""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import zero_sharded_optimizer_bucket_gb300 as zs  # noqa: E402
from oracle import step as ostep  # noqa: E402
from synth import workloads  # noqa: E402
from tests import gpu_harness as H  # noqa: E402

pytestmark = pytest.mark.gpu


def _run_both(d, max_norm):
    """(norm, coef, flags) from zs_grad_norm with caller scratch, and from the
    no-allocation entry point into separate device scalars."""
    d.grad_norm(max_norm, recompute=True)
    ref = (float(d.d_norm.np()[0]), float(d.d_coef.np()[0]), int(d.d_flags.np()[0]))
    out_norm = H.Guarded(1, torch.float32, d.dev)
    out_coef = H.Guarded(1, torch.float32, d.dev)
    out_flags = H.Guarded(1, torch.int32, d.dev)
    zs.zs_grad_norm_noalloc(d.plan, d.bufs["grad_shards"].ptr(), d.bufs["persist_grads"].ptr(),
                            max_norm, out_norm.ptr(), out_coef.ptr(), out_flags.ptr())
    torch.cuda.synchronize()
    got = (float(out_norm.np()[0]), float(out_coef.np()[0]), int(out_flags.np()[0]))
    assert out_norm.guards_ok() and out_coef.guards_ok() and out_flags.guards_ok()
    return ref, got


@pytest.mark.parametrize("case", ["many_small", "ragged"])
def test_noalloc_norm_matches_scratch_version_two_calls(case):
    if case == "many_small":
        d = H.DevicePlan(workloads.many_small(40).numel, 64, threshold=100_000)
    else:
        rng = np.random.default_rng(8)
        numel = [int(x) for x in rng.integers(0, 30_000, size=40)]
        d = H.DevicePlan(numel, 7, threshold=50, B=3000)
    d.init_weights()
    # two calls in a row on different gradients: the second call must not
    # see anything the first one left in the shared array
    for call, (seed, max_norm) in enumerate([(41, 1.0), (42, 0.05)]):
        d.set_grads(seed, use_gpu_generator=True)
        d.reduce_scatter_all_buckets(with_scratch=False)
        ref, got = _run_both(d, max_norm)
        # the same kernels on the same reduced gradients: the same bits
        assert ref[2] == got[2] == 0, f"call {call}"
        assert _bits(got[0]) == _bits(ref[0]), f"call {call}: norm {got[0]!r} vs {ref[0]!r}"
        assert _bits(got[1]) == _bits(ref[1]), f"call {call}: coef {got[1]!r} vs {ref[1]!r}"
        # and the oracle's norm of its own reduce-scatter of the same rank
        # gradients, within the norm tolerance
        for b in range(len(d.op.reduce_buckets)):
            ostep.reduce_scatter(d.op, b, d.grad_bufs[b], d.ost)
        onorm, ocoef, oskip = ostep.grad_norm(d.op, d.ost, max_norm)
        assert not oskip
        assert abs(got[0] - float(onorm)) <= 1e-5 * float(onorm), f"call {call}: vs oracle"
        assert abs(got[1] - float(ocoef)) <= 1e-5 * float(ocoef), f"call {call}: coef vs oracle"
        assert float(ocoef) < 1.0              # clipping is active
    d.check_canaries()


def _bits(x):
    return int(np.float32(x).view(np.uint32))


def test_noalloc_rejects_plans_beyond_the_array():
    # 256 ranks x 4200 one-element shards: one tile per shard, more tiles
    # than the built-in array has room for partial sums
    cfg = zs.zs_default_config(256)
    cfg.param_persistence_threshold = 0
    plan = zs.zs_build_partition(cfg, [256] * 4200)
    info = zs.zs_plan_info(plan)
    assert info["norm_scratch_elems"] > zs.ZS_NOALLOC_NORM_MAX_SCRATCH
    scal = torch.zeros(4, dtype=torch.float32, device="cuda")
    flags = torch.zeros(4, dtype=torch.int32, device="cuda")
    with pytest.raises(zs.ZsError) as ei:
        zs.zs_grad_norm_noalloc(plan, scal, scal, 1.0, scal, scal[1:], flags)
    assert ei.value.status == zs.ZS_EINVAL and "built-in array" in str(ei.value)
