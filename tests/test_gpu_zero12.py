"""ZeRO-1/2 residency on the same kernels ([Core flow] §4 table: stage 1
shards the optimizer state, stage 2 also the gradients, both keep the full
parameters on every rank).

Stage 2: the fused step without a shard buffer writes the new parameters
only into the full replica (model flat space).  Its replica and optimizer
state are checked against the oracle's own steps (the replica against the
oracle's gather of its updated shards), and against the ZeRO-3 step's
gathered output and state bit for bit.
Stage 1: the gradient all-reduce is the reduce-scatter followed by the
all-gather of the reduced gradients; it must equal the oracle's all-reduce
mean of the full gradients."""
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
from tests import test_gpu_parity as P  # noqa: E402

pytestmark = pytest.mark.gpu
HP = P.HP


@pytest.mark.parametrize("case", ["tiny_thr100", "ragged_n16_chunks", "many_small_64",
                                  "ragged_n16_chunks_hsdp4"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_zero2_step_equals_zero3_replica(case, dtype):
    """The last case is HSDP (groups of 4 of the 16 ranks): stage-2
    residency within each replica group."""
    if case.endswith("_hsdp4"):
        kw = dict(P.CASES[case[:-len("_hsdp4")]], dtype=dtype, log2_scale=-2, group=4)
    else:
        kw = dict(P.CASES[case], dtype=dtype, log2_scale=-2)
    a, b = H.DevicePlan(**kw), H.DevicePlan(**kw)
    for d in (a, b):
        d.init_weights()
    shards_before = b.bufs["param_shards"].u16().copy()
    st2 = zs.make_state(**{k: (None if k == "param_shards" else v.ptr()) for k, v in b.bufs.items()})
    sa = torch.tensor([256.0, 0, 0, 0], device=a.dev)
    sb = sa.clone()
    ga, gb = torch.zeros(4, dtype=torch.int32, device=a.dev), torch.zeros(4, dtype=torch.int32, device=a.dev)
    osc = ostep.LossScaler(scale=256.0, window=2) if dtype == "fp16" else None
    for t in (1, 2, 3):
        for d in (a, b):
            d.set_grads(700 + t, use_gpu_generator=case.startswith("many"))
        if dtype == "fp16":
            zs.zs_shard_step_scaled(a.plan, a.ptr_table, a.state, a.scratch.ptr(), HP, t, 1.0,
                                    zs.make_loss_scaler(sa, ga, 2.0, 1.0, 2), a.d_norm.ptr(),
                                    a.d_coef.ptr(), a.d_flags.ptr(), a.flat.ptr())
            zs.zs_shard_step_scaled(b.plan, b.ptr_table, st2, b.scratch.ptr(), HP, t, 1.0,
                                    zs.make_loss_scaler(sb, gb, 2.0, 1.0, 2), b.d_norm.ptr(),
                                    b.d_coef.ptr(), b.d_flags.ptr(), b.flat.ptr())
        else:
            a.shard_step(HP, t, 1.0)
            zs.zs_shard_step(b.plan, b.ptr_table, st2, b.scratch.ptr(), HP, t, 1.0, b.d_norm.ptr(),
                             b.d_coef.ptr(), b.d_flags.ptr(), b.flat.ptr())
        xa, xb = a.snapshot(), b.snapshot()
        # the stage-2 run against the oracle's own step: state, and the
        # replica against the oracle's gather of its updated shards
        prev = H.oracle_state(b.ost)
        norm, coef, skip, flat = ostep.shard_step(b.op, b.ost, b.grad_bufs, HP, t, 1.0, osc)
        assert int(b.d_flags.np()[0]) == int(skip)
        assert np.array_equal(xb["grad_shards"], b.ost.grad_shards)
        exact = skip or H.same_bits(b.d_coef.np()[0], coef)
        H.assert_state(xb, b.ost, prev, f"{case} {dtype} stage 2 step {t}", exact)
        H.assert_16bit(b.flat.u16(), flat, "stage-2 replica", dtype, exact)
        H.assert_16bit(xb["persist_params"], b.ost.persist_params, "persist_params", dtype, exact)
        # and against the ZeRO-3 run, bit for bit
        for k in ("master", "exp_avg", "exp_avg_sq", "p_master", "persist_params", "grad_shards"):
            assert np.array_equal(xa[k].view(np.uint8), xb[k].view(np.uint8)), k
        assert np.array_equal(a.flat.u16(), b.flat.u16())
    # the replica holds the parameters: every shard is a slice of it
    assert np.array_equal(ostep.gather_model(a.op, a.snapshot()["param_shards"]), b.flat.u16())
    assert np.array_equal(b.bufs["param_shards"].u16(), shards_before)
    b.check_canaries()


@pytest.mark.parametrize("case", ["tiny_thr100", "ragged_n7", "numel_lt_n"])
def test_zero1_gradient_allreduce(case):
    d = P.make(case)
    d.init_weights()
    d.set_grads(91)
    d.reduce_scatter_all_buckets(with_scratch=False)
    out = H.Guarded(d.op.flat_elems, torch.int16, d.dev)
    for g in d.op.gather_buckets:
        zs.zs_all_gather_coalesced(d.plan, g.params, d.bufs["grad_shards"].ptr(),
                                   out.ptr() + 2 * g.flat_off, g.flat_elems)
    torch.cuda.synchronize()
    got = out.u16()
    N = d.N
    # oracle: all-reduce mean of each rank's full gradient, parameter by parameter
    full = {}
    for b_, ents in enumerate(d.op.reduce_buckets):
        for e in ents:
            vals = np.stack([d.grad_bufs[b_][k][e.buf_off:e.buf_off + e.e_hi - e.e_lo]
                             for k in range(N)])
            full.setdefault(e.param, []).append((e.e_lo, ostep.reduce_mean(vals, d.dtype)))
    for p in d.op.params:
        if p.persistent or p.numel == 0:
            continue
        ref = np.concatenate([v for _, v in sorted(full[p.index], key=lambda x: x[0])])
        assert np.array_equal(got[p.flat_off:p.flat_off + p.numel], ref), p.index
    assert out.guards_ok()
