"""GPU parity of the fp16 mode with a dynamic loss scale, against the oracle:
reduce-scatter and gathers bit-exact, unscale-and-clip, the device-resident
loss-scale schedule across an overflow and a growth window, Adam with the
oracle's coefficient bit-exact, fused == per-call chain."""
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


def _ragged(seed, n=24, N=7):
    rng = np.random.default_rng(seed)
    numel = [int(x) for x in rng.integers(0, 3000, size=n)] + [2501, 1]
    return dict(numel=numel, N=N, threshold=50, B=1000, G=5000, U=700, seed=seed)


CASES = {
    "tiny_fp16": dict(numel=workloads.tiny().numel, N=4, threshold=0),
    "ragged_fp16": _ragged(6),
    "many_small_fp16": dict(numel=workloads.many_small(30).numel, N=64, threshold=100_000),
}


def make(case, **kw):
    a = dict(CASES[case], dtype="fp16", log2_scale=-2)
    a.update(kw)
    return H.DevicePlan(**a)


@pytest.fixture(params=list(CASES))
def case(request):
    return request.param


class DevScaler:
    def __init__(self, dev, scale, window, factor=2.0, min_scale=1.0):
        self.s = torch.tensor([scale, 0, 0, 0], dtype=torch.float32, device=dev)
        self.g = torch.zeros(4, dtype=torch.int32, device=dev)
        self.c = zs.make_loss_scaler(self.s, self.g, factor, min_scale, window)

    def read(self):
        return float(self.s[0]), int(self.g[0])


def test_generator_fp16_gpu_matches_cpu():
    n = 200_003
    t = torch.empty(n, dtype=torch.int16, device="cuda")
    sgpu.fill_grad_fp16(t, 777, 9, -3, outlier_frac=0.02, outlier_log2=18)
    ref = philox.grad_fp16(9, 0, np.arange(777, 777 + n, dtype=np.uint64), -3, 0.02, 18)
    assert np.array_equal(t.cpu().numpy().view(np.uint16), ref)


def test_fp16_partition_and_reduce_scatter(case):
    d = make(case)
    d.init_weights()
    s = d.snapshot()
    assert np.array_equal(s["param_shards"], d.ost.param_shards)
    assert np.array_equal(s["persist_params"], d.ost.persist_params)
    d.set_grads(31, use_gpu_generator=case.startswith("many"))
    d.reduce_scatter_all_buckets()
    for b in range(len(d.op.reduce_buckets)):
        ostep.reduce_scatter(d.op, b, d.grad_bufs[b], d.ost)
    s = d.snapshot()
    assert np.array_equal(s["grad_shards"], d.ost.grad_shards)
    assert np.array_equal(s["persist_grads"], d.ost.persist_grads)
    d.check_canaries()


def test_unscale_and_clip(case):
    d = make(case)
    d.init_weights()
    d.set_grads(32, use_gpu_generator=case.startswith("many"))
    d.reduce_scatter_all_buckets(with_scratch=True)
    for b in range(len(d.op.reduce_buckets)):
        ostep.reduce_scatter(d.op, b, d.grad_bufs[b], d.ost)
    for S, max_norm in [(1024.0, 1.0), (32.0, 1e-3), (1.0, 0.0)]:
        sc = DevScaler(d.dev, S, 0)                     # static scale
        zs.zs_unscale_and_clip(d.plan, d.bufs["grad_shards"].ptr(), d.bufs["persist_grads"].ptr(),
                               d.scratch.ptr(), False, max_norm, sc.c, d.d_norm.ptr(),
                               d.d_coef.ptr(), d.d_flags.ptr())
        norm, coef, skip = ostep.unscale_and_clip(d.op, d.ost, max_norm, S)
        assert abs(float(d.d_norm.np()[0]) - float(norm)) <= 1e-5 * float(norm)
        assert abs(float(d.d_coef.np()[0]) - float(coef)) <= 1e-5 * float(coef)
        assert sc.read() == (S, 0) and int(d.d_flags.np()[0]) == 0
    # a static scale of 1 is zs_grad_norm, bit for bit
    sc = DevScaler(d.dev, 1.0, 0)
    zs.zs_unscale_and_clip(d.plan, d.bufs["grad_shards"].ptr(), d.bufs["persist_grads"].ptr(),
                           d.scratch.ptr(), True, 1.0, sc.c, d.d_norm.ptr(), d.d_coef.ptr(),
                           d.d_flags.ptr())
    a = (float(d.d_norm.np()[0]), float(d.d_coef.np()[0]))
    d.grad_norm(1.0, recompute=True)
    assert a == (float(d.d_norm.np()[0]), float(d.d_coef.np()[0]))
    d.check_canaries()


def test_fp16_adam_bit_exact_with_oracle_coefficient(case):
    d = make(case)
    d.init_weights()
    for t in (1, 2):
        d.set_grads(40 + t, use_gpu_generator=case.startswith("many"))
        d.reduce_scatter_all_buckets(with_scratch=False)
        for b in range(len(d.op.reduce_buckets)):
            ostep.reduce_scatter(d.op, b, d.grad_bufs[b], d.ost)
        coef = np.float32(1.0) / np.float32(256.0)
        d.d_coef.t.fill_(float(coef))
        d.d_flags.t.zero_()
        d.adam(HP, t)
        ostep.adam_step(d.op, -1, HP, t, coef, False, d.ost)
        s = d.snapshot()
        for k, ref in [("master", d.ost.master), ("exp_avg", d.ost.exp_avg),
                       ("exp_avg_sq", d.ost.exp_avg_sq), ("p_master", d.ost.p_master)]:
            assert np.array_equal(s[k].view(np.uint32), ref.view(np.uint32)), k
        assert np.array_equal(s["param_shards"], d.ost.param_shards)
        assert np.array_equal(s["persist_params"], d.ost.persist_params)


def test_fp16_scaled_steps_with_overflow_and_growth(case):
    """Fused scaled steps against the oracle's: step 2 overflows (an inf in
    one rank's gradient), the update is skipped and the scale halves; with
    a window of 2 the scale doubles again after two good steps."""
    d = make(case)
    d.init_weights()
    sc = DevScaler(d.dev, 1024.0, 2)
    osc = ostep.LossScaler(scale=1024.0, window=2)
    for t in range(1, 5):
        d.set_grads(60 + t, use_gpu_generator=case.startswith("many"))
        if t == 2:
            host = d.pool.cpu()
            host[0] = 0x7C00
            d.pool.copy_(host)
            d.grad_bufs[0][0][0] = 0x7C00
        zs.zs_shard_step_scaled(d.plan, d.ptr_table, d.state, d.scratch.ptr(), HP, t, 1.0, sc.c,
                                d.d_norm.ptr(), d.d_coef.ptr(), d.d_flags.ptr(), d.flat.ptr())
        prev = H.oracle_state(d.ost)
        norm, coef, skip, flat = ostep.shard_step(d.op, d.ost, d.grad_bufs, HP, t, 1.0, osc)
        torch.cuda.synchronize()
        assert sc.read() == (osc.scale, osc.good), f"step {t}"
        assert int(d.d_flags.np()[0]) == int(skip)
        s = d.snapshot()
        assert np.array_equal(s["grad_shards"], d.ost.grad_shards)
        # a skipped step leaves the state alone on both sides: bits
        exact = skip or H.same_bits(d.d_coef.np()[0], coef)
        H.assert_state(s, d.ost, prev, f"{case} step {t}", exact)
        H.assert_16bit(s["param_shards"], d.ost.param_shards, "param_shards", "fp16", exact)
        H.assert_16bit(d.flat.u16(), flat, "gathered", "fp16", exact)
    assert [osc.scale] == [1024.0]     # 1024 -> 512 (overflow) -> 1024 after two good steps
    d.check_canaries()


def test_fp16_fused_equals_unfused(case):
    a, b = make(case), make(case)
    for d in (a, b):
        d.init_weights()
    sa, sb = DevScaler(a.dev, 512.0, 3), DevScaler(b.dev, 512.0, 3)
    for t in (1, 2):
        for d in (a, b):
            d.set_grads(80 + t, use_gpu_generator=case.startswith("many"))
        zs.zs_shard_step_scaled(a.plan, a.ptr_table, a.state, a.scratch.ptr(), HP, t, 1.0, sa.c,
                                a.d_norm.ptr(), a.d_coef.ptr(), a.d_flags.ptr(), a.flat.ptr())
        b.reduce_scatter_all_buckets(with_scratch=True)
        zs.zs_unscale_and_clip(b.plan, b.bufs["grad_shards"].ptr(), b.bufs["persist_grads"].ptr(),
                               b.scratch.ptr(), False, 1.0, sb.c, b.d_norm.ptr(), b.d_coef.ptr(),
                               b.d_flags.ptr())
        b.adam(HP, t)
        b.gather_model_unfused(b.flat)
        xa, xb = a.snapshot(), b.snapshot()
        for k in xa:
            assert np.array_equal(xa[k].view(np.uint8), xb[k].view(np.uint8)), k
        assert np.array_equal(a.flat.u16(), b.flat.u16())
        assert sa.read() == sb.read()


def test_scaler_argument_errors():
    d = make("tiny_fp16")
    d.init_weights()
    bad = zs.make_loss_scaler(None)
    with pytest.raises(zs.ZsError):
        zs.zs_unscale_and_clip(d.plan, d.bufs["grad_shards"].ptr(), d.bufs["persist_grads"].ptr(),
                               d.scratch.ptr(), True, 1.0, bad, d.d_norm.ptr(), d.d_coef.ptr(),
                               d.d_flags.ptr())
    s = torch.ones(4, device="cuda")
    bad = zs.make_loss_scaler(s, None, 2.0, 1.0, 10)       # window needs the counter
    with pytest.raises(zs.ZsError):
        zs.zs_unscale_and_clip(d.plan, d.bufs["grad_shards"].ptr(), d.bufs["persist_grads"].ptr(),
                               d.scratch.ptr(), True, 1.0, bad, d.d_norm.ptr(), d.d_coef.ptr(),
                               d.d_flags.ptr())
