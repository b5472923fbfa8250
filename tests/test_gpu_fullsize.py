"""Full-size parity on sampled outputs, in the launch configuration bench.py
times (bench.DeviceWorkload + zs_shard_step).

The oracle computes each sampled element on its own: the N rank gradients
of that element (drawn by synth at the element's pool position), the rank
mean, one AdamW step from the partitioned initial weight.  max_norm = 0
makes the clip coefficient exactly 1 on both sides, so no value computed by
the device is ever an input of the oracle.  The gradient norm at full size
is checked through a property that holds at any size: it equals the norm
of the device's reduced-gradient buffers (float64 sum).
"""
from __future__ import annotations

import gc

import numpy as np
import pytest

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("needs a CUDA GPU", allow_module_level=True)

import bench  # noqa: E402
import zero_sharded_optimizer_bucket_gb300 as zs  # noqa: E402
from oracle import plan as oplan  # noqa: E402
from oracle import step as ostep  # noqa: E402
from synth import philox, workloads  # noqa: E402
from tests import gpu_harness as H  # noqa: E402

pytestmark = pytest.mark.gpu


def _oracle_plan(w):
    return oplan.build_partition(w.numel, w.n_ranks, threshold=w.persistence_threshold,
                                 reduce_bucket_size=w.reduce_bucket_size,
                                 prefetch_bucket_size=w.prefetch_bucket_size,
                                 sub_group_size=w.sub_group_size, ds_id=w.ds_id, dtype=w.dtype,
                                 shard_group_size=w.shard_group_size or None)


def _grads(w, idx):
    if w.dtype == "fp16":
        return philox.grad_fp16(w.seed, 0, idx, w.fp16_log2_scale)
    return philox.grad_bf16(w.seed, 0, idx, w.grad_sigma, w.outlier_frac, w.outlier_scale)


def _samples(op, rng, n_random=3000):
    """(rank, column) of random shard elements plus the first, last,
    padding and alignment columns of 40 random partitioned parameters."""
    N, S = op.group, op.S            # shard rows: a group's owners
    rs = list(rng.integers(0, N, size=n_random))
    cs = list(rng.integers(0, S, size=n_random))
    part = [p for p in op.params if not p.persistent and p.ps > 0]
    for p in rng.permutation(len(part))[:40]:
        p = part[p]
        for r in (0, N // 2, N - 1):
            for j in (0, p.ps - 1, p.ps // 2, min(p.ps + 3, (p.ps + 7) // 8 * 8 - 1)):
                if 0 <= j < (p.ps + 7) // 8 * 8:
                    rs.append(r)
                    cs.append(p.shard_off + j)
    return np.array(rs, dtype=np.int64), np.array(cs, dtype=np.int64)


def _locate(op, w, dw, cols, ranks):
    """For each sampled element: kind (0 data, 1 padding/alignment), its
    parameter element index e, input index and the N pool indices of its
    rank gradients."""
    part = sorted([p for p in op.params if not p.persistent and p.ps > 0], key=lambda p: p.shard_off)
    starts = np.array([p.shard_off for p in part], dtype=np.int64)
    pi = np.searchsorted(starts, cols, side="right") - 1
    N = op.n_ranks
    kind = np.ones(len(cols), dtype=np.int64)
    win = np.zeros(len(cols), dtype=np.int64)
    pool_idx = np.zeros((N, len(cols)), dtype=np.uint64)
    for s, (c, r, k) in enumerate(zip(cols, ranks, pi)):
        p = part[k]
        j = int(c) - p.shard_off
        if j >= p.ps:
            continue
        e = int(r) * p.ps + j
        if e >= p.numel:
            continue
        for b in p.reduce_buckets:
            ent = [x for x in op.reduce_buckets[b] if x.param == p.index][0]
            if ent.e_lo <= e < ent.e_hi:
                pos = ent.buf_off + e - ent.e_lo
                pool_idx[:, s] = [dw.offs[b][q] + pos for q in range(N)]
                break
        kind[s] = 0
        win[s] = p.input_off + e
    return kind, win, pool_idx


@pytest.mark.parametrize("name", ["llama_layer", "many_small", "llama3_16_layers", "llama3_8b",
                                  "llama3_8b_fp16", "llama3_8b_hsdp", "giant_param"])
def test_fullsize_sampled(name):
    w = workloads.WORKLOADS[name]()
    op = _oracle_plan(w)
    dw = bench.DeviceWorkload(w, "cuda:0", max_norm=0.0)
    try:
        assert dw.info["shard_elems"] == op.S and dw.info["flat_elems"] == op.flat_elems
        dw.step()
        torch.cuda.synchronize()
        # max_norm = 0: no clipping, the coefficient is 1 / loss scale (1 for bf16)
        S = np.float32(w.loss_scale if w.dtype == "fp16" else 1.0)
        coef = np.float32(1.0) / S
        assert int(dw.d_flags[0]) == 0 and float(dw.d_coef[0]) == float(coef)
        rng = np.random.default_rng(11)
        ranks, cols = _samples(op, rng)
        idx = torch.from_numpy(ranks * op.S + cols).to(dw.dev)
        got = {k: getattr(dw, a).index_select(0, idx).cpu().numpy()
               for k, a in [("gs", "gs"), ("ps", "ps"), ("p", "master"), ("m", "m"), ("v", "v")]}
        kind, win, pidx = _locate(op, w, dw, cols, ranks)
        data = kind == 0
        vals = _grads(w, pidx[:, data].ravel()).reshape(op.n_ranks, -1)
        gs_ref = ostep.reduce_mean_groups(vals, op.group, w.dtype)
        W = philox.weight_f32(w.seed, win[data].astype(np.uint64), w.weight_sigma)
        z = np.zeros_like(W)
        p1, m1, v1, pb = ostep.adam_update(W, z, z, gs_ref, coef,
                                           ostep.adam_consts(w.hparams(), 1), w.dtype)
        assert np.array_equal(got["gs"].view(np.uint16)[data], gs_ref)
        H.assert_f32_close(got["p"][data], p1, "master")
        H.assert_f32_close(got["m"][data], m1, "exp_avg")
        H.assert_f32_close(got["v"][data], v1, "exp_avg_sq")
        if w.dtype == "fp16":
            H.assert_fp16_within_ulp(got["ps"].view(np.uint16)[data], pb, "param_shards")
        else:
            H.assert_bf16_within_ulp(got["ps"].view(np.uint16)[data], pb, "param_shards")
        # padding and alignment columns stay exactly zero
        for k in ("gs", "ps", "p", "m", "v"):
            assert not np.any(got[k].view(np.uint8).reshape(len(cols), -1)[~data])
        # gathered parameters: the bf16 shard values at their flat positions
        part = sorted([p for p in op.params if not p.persistent and p.ps > 0],
                      key=lambda p: p.shard_off)
        starts = np.array([p.shard_off for p in part])
        fpos, fsrc = [], []
        for s in np.nonzero(data)[0]:
            p = part[np.searchsorted(starts, cols[s], side="right") - 1]
            fpos.append(p.flat_off + int(ranks[s]) * p.ps + int(cols[s]) - p.shard_off)
            fsrc.append(s)
        fl = dw.flat.index_select(0, torch.tensor(fpos, device=dw.dev)).cpu().numpy()
        assert np.array_equal(fl.view(np.uint16), got["ps"].view(np.uint16)[fsrc])
        # the same positions after zs_all_gather_coalesced of every gather
        # bucket into a cleared flat buffer (the Llama plans take the
        # bulk-copy path: all partition sizes are multiples of 8)
        dw.flat.zero_()
        for g in op.gather_buckets:
            zs.zs_all_gather_coalesced(dw.plan, g.params, dw.ps, dw.flat[g.flat_off:],
                                       g.flat_elems)
        torch.cuda.synchronize()
        fl = dw.flat.index_select(0, torch.tensor(fpos, device=dw.dev)).cpu().numpy()
        assert np.array_equal(fl.view(np.uint16), got["ps"].view(np.uint16)[fsrc])
        assert zs.zs_device_wait_timeouts() == 0
        # persistent parameters: sampled elements
        pers = [p for p in op.params if p.persistent and p.numel > 0]
        if pers:
            P = pers[:: max(1, len(pers) // 30)]
            ents = []
            for p in P:
                for e in sorted(set([0, p.numel - 1, p.numel // 3])):
                    b = p.reduce_buckets[0]
                    ent = [x for x in op.reduce_buckets[b] if x.param == p.index][0]
                    ents.append((p.persist_off + e, p.input_off + e,
                                 [dw.offs[b][q] + ent.buf_off + e for q in range(op.n_ranks)]))
            pidx2 = torch.tensor([x[0] for x in ents], device=dw.dev)
            pv = _grads(w, np.array([x[2] for x in ents], dtype=np.uint64).T.ravel()
                        ).reshape(op.n_ranks, -1)
            gP_ref = ostep.reduce_mean_groups(pv, op.group, w.dtype)
            assert np.array_equal(dw.gP.index_select(0, pidx2).cpu().numpy().view(np.uint16), gP_ref)
            Wp = philox.weight_f32(w.seed, np.array([x[1] for x in ents], dtype=np.uint64),
                                   w.weight_sigma)
            zp = np.zeros_like(Wp)
            pp1 = ostep.adam_update(Wp, zp, zp, gP_ref, coef,
                                    ostep.adam_consts(w.hparams(), 1), w.dtype)[0]
            H.assert_f32_close(dw.pm.index_select(0, pidx2).cpu().numpy(), pp1, "p_master")
        # the norm is the norm of the reduced-gradient buffers
        tot = 0.0
        for buf, n in ((dw.gs, op.group * op.S), (dw.gP, op.Pn_alloc)):
            for ch in buf[:n].split(1 << 27):
                x = ch.view(torch.float16 if w.dtype == "fp16" else torch.bfloat16).double()
                tot += float((x * x).sum())
        ref = float(np.sqrt(tot)) / float(S)
        assert abs(float(dw.d_norm[0]) - ref) <= 1e-5 * ref
    finally:
        del dw
        gc.collect()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["llama3_8b", "many_small", "llama3_8b_fp16", "llama3_8b_hsdp"])
def test_fullsize_whole_buckets(name):
    """Every element of whole reduce buckets at full size (the first two,
    the middle one, the last one and every 64th): reduced gradient bit for
    bit, fp32 master / moments within tolerance, the cast parameter within
    one ulp, and its place in the gathered replica.  The rank gradients are
    read back from the device pool the shared generator filled (its GPU fill
    is pinned bit for bit to the CPU one), not regenerated on the host."""
    w = workloads.WORKLOADS[name]()
    op = _oracle_plan(w)
    dw = bench.DeviceWorkload(w, "cuda:0", max_norm=0.0)
    try:
        dw.step()
        torch.cuda.synchronize()
        N, S = op.n_ranks, op.S
        # max_norm = 0: no clipping; the coefficient is 1 / loss scale
        coef = np.float32(1.0) / np.float32(w.loss_scale if w.dtype == "fp16" else 1.0)
        within_ulp = H.assert_fp16_within_ulp if w.dtype == "fp16" else H.assert_bf16_within_ulp
        c = ostep.adam_consts(w.hparams(), 1)
        nb = len(op.reduce_buckets)
        picks = sorted({0, min(1, nb - 1), nb // 2, nb - 1, *range(0, nb, 64)})
        checked = 0
        for b in picks:
            for ent in op.reduce_buckets[b]:
                p = op.params[ent.param]
                L = ent.e_hi - ent.e_lo
                e = np.arange(ent.e_lo, ent.e_hi, dtype=np.int64)
                rows = [dw.pool[dw.offs[b][k] + ent.buf_off:dw.offs[b][k] + ent.buf_off + L]
                        for k in range(N)]
                vals = torch.stack(rows).cpu().numpy().view(np.uint16)
                gs_ref = ostep.reduce_mean_groups(vals, op.group, w.dtype)
                if p.persistent:
                    idx = torch.from_numpy(p.persist_off + e).to(dw.dev)
                    got_g = dw.gP.index_select(0, idx)
                    got_p, got_ps = dw.pm.index_select(0, idx), dw.pP.index_select(0, idx)
                    got_m, got_v = dw.pmm.index_select(0, idx), dw.pmv.index_select(0, idx)
                else:
                    r, j = e // p.ps, e % p.ps
                    idx = torch.from_numpy(r * S + p.shard_off + j).to(dw.dev)
                    got_g = dw.gs.index_select(0, idx)
                    got_p, got_ps = dw.master.index_select(0, idx), dw.ps.index_select(0, idx)
                    got_m, got_v = dw.m.index_select(0, idx), dw.v.index_select(0, idx)
                assert np.array_equal(got_g.cpu().numpy().view(np.uint16), gs_ref), (b, p.index)
                W = philox.weight_f32(w.seed, (p.input_off + e).astype(np.uint64), w.weight_sigma)
                z = np.zeros_like(W)
                p1, m1, v1, pb = ostep.adam_update(W, z, z, gs_ref, coef, c, w.dtype)
                H.assert_f32_close(got_p.cpu().numpy(), p1, "master")
                H.assert_f32_close(got_m.cpu().numpy(), m1, "exp_avg")
                H.assert_f32_close(got_v.cpu().numpy(), v1, "exp_avg_sq")
                pbits = got_ps.cpu().numpy().view(np.uint16)
                within_ulp(pbits, pb, "params")
                if not p.persistent:
                    fl = dw.flat.index_select(0, torch.from_numpy(p.flat_off + e).to(dw.dev))
                    assert np.array_equal(fl.cpu().numpy().view(np.uint16), pbits)
                checked += L
        assert checked > 0
    finally:
        del dw
        gc.collect()
        torch.cuda.empty_cache()
