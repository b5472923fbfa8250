"""The benchmark's end-to-end leg (gradients streamed from pinned host
memory through a device ring, a reduce-scatter per bucket as its copy
lands, the norm, the update, each step's result read back without a host
wait) leaves exactly the state of the fused step run on the same
gradients: master, moments, shards, gathered parameters, bit for bit."""
from __future__ import annotations

import gc

import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bench  # noqa: E402
from synth import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def test_e2e_leg_equals_fused_steps():
    w = workloads.llama_layer()
    a = bench.DeviceWorkload(w, "cuda:0")
    b = bench.DeviceWorkload(w, "cuda:0")
    try:
        total = sum(a.N * workloads.pool_align(L) for L in a.buf_elems)
        assert a.pool_elems >= total     # no wrap: the host buffer holds the same gradients
        r = bench.run_e2e(a, steps=2, warmup=1)
        for _ in range(3):
            b.step()
        torch.cuda.synchronize()
        assert a.t == b.t == 3 and r["skip_flags"] == [0, 0, 0]
        for name in ("gs", "ps", "master", "m", "v", "gP", "pP", "pm", "pmm", "pmv", "flat"):
            x, y = getattr(a, name), getattr(b, name)
            assert torch.equal(x.view(torch.int16) if x.dtype == torch.int16 else x.view(torch.int32),
                               y.view(torch.int16) if y.dtype == torch.int16 else y.view(torch.int32)), name
        assert torch.equal(a.d_norm[:1], b.d_norm[:1])
    finally:
        del a, b
        gc.collect()
        torch.cuda.empty_cache()
