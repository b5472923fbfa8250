"""The per-call API under CUDA-graph capture: the per-call chain of one
step (zs_reduce_scatter per bucket, zs_grad_norm, zs_adam_step per
sub-group, zs_all_gather_coalesced per gather bucket), captured once and
replayed, gives the same bits as the same step run eagerly (no call
synchronises the host or allocates, so capture records every launch)."""
from __future__ import annotations

import gc

import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bench  # noqa: E402
from synth import workloads  # noqa: E402

pytestmark = pytest.mark.gpu


def test_captured_per_call_step_equals_eager():
    w = workloads.llama_layer()
    a = bench.DeviceWorkload(w, "cuda:0")
    b = bench.DeviceWorkload(w, "cuda:0")
    try:
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            a.unfused_step()                 # step 1, eager (also warms the launchers)
            b.unfused_step()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            a.unfused_step()                 # step 2, captured (t = 2 by value)
        with torch.cuda.stream(s):
            g.replay()
            b.unfused_step()                 # step 2, eager
        torch.cuda.synchronize()
        assert a.t == b.t == 2
        for name in ("gs", "ps", "master", "m", "v", "gP", "pP", "pm", "pmm", "pmv", "flat"):
            x, y = getattr(a, name), getattr(b, name)
            view = torch.int16 if x.dtype == torch.int16 else torch.int32
            assert torch.equal(x.view(view), y.view(view)), name
        assert torch.equal(a.d_norm[:1], b.d_norm[:1])
    finally:
        del a, b
        gc.collect()
        torch.cuda.empty_cache()
