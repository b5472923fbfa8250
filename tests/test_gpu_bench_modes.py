"""The benchmark's gather-schedule mode runs end to end on a small workload
with both stand-in computes and prints one consistent JSON line."""
from __future__ import annotations

import json

import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bench  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("compute", ["busy", "gemm"])
def test_gather_schedule_mode(compute, capsys):
    bench.main(["--gather-schedule", "--workload", "llama_layer", "--gather-compute", compute])
    line = [x for x in capsys.readouterr().out.splitlines() if x.startswith("{")][-1]
    d = json.loads(line)
    assert d["mode"] == "gather_schedule" and d["workload"] == "llama_layer"
    for k in ("compute_only_ms", "gathers_only_ms", "prefetch_overlapped_ms", "no_prefetch_ms"):
        assert d[k] > 0
    # overlapped can not beat the slower of the two parts by much, nor lose
    # more than the sum of both
    assert d["prefetch_overlapped_ms"] >= 0.9 * max(d["compute_only_ms"], d["gathers_only_ms"])
    assert d["prefetch_overlapped_ms"] <= 1.2 * (d["compute_only_ms"] + d["gathers_only_ms"])
    st = d["sched_stats"]
    assert st["passes"] == 3 and st["invalidations"] == 0 and st["gathers"] > 0
    assert (d["compute_tflops"] is not None) == (compute == "gemm")
