"""The bulk gather's bounded device wait, made to run out on purpose: a
wait on an mbarrier that nothing arrives on gives up after its limit, the
timeout is counted and reported as ZS_ETIMEOUT, and the CUDA context keeps
working (a gather right after is exact).  Nothing faults, traps or hangs."""
from __future__ import annotations

import time

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import zero_sharded_optimizer_bucket_gb300 as zs  # noqa: E402
from oracle import step as ostep  # noqa: E402
from tests import gpu_harness as H  # noqa: E402

pytestmark = pytest.mark.gpu


def test_wait_runs_out_and_is_reported():
    zs.zs_device_wait_timeouts(reset=True)
    assert zs.zs_device_wait_timeouts() == 0
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    zs.zs_test_wait_timeout(20_000_000)            # 20 ms
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert 0.015 <= waited < 5.0
    assert zs.zs_device_wait_timeouts(reset=True) == 1
    assert zs.zs_device_wait_timeouts() == 0
    # the context still works: an aligned gather (bulk path) is exact
    numel = [65536, 131136, 8192, 192000]
    d = H.DevicePlan(numel, 8, threshold=1000, seed=5)
    d.init_weights()
    req = [0, 1, 2, 3]
    flat_ref, views_ref = ostep.all_gather_coalesced(d.op, req, d.ost.param_shards)
    out = H.Guarded(len(flat_ref), torch.int16, d.dev)
    assert zs.zs_all_gather_coalesced(d.plan, req, d.bufs["param_shards"].ptr(), out.ptr(),
                                      len(flat_ref)) == views_ref
    torch.cuda.synchronize()
    assert np.array_equal(out.u16(), flat_ref) and out.guards_ok()
    assert zs.zs_device_wait_timeouts() == 0
