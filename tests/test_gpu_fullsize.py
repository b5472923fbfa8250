"""Full-size parity, in the launch configuration bench.py times
(bench.DeviceWorkload + zs_shard_step).

test_fullsize_sampled: max_norm = 0 makes the clip coefficient exactly
1 / loss scale on both sides, so the device's state must equal the oracle's
bit for bit.  The oracle computes each sampled element on its own: the N
rank gradients of that element (drawn by synth at the element's pool
position), the rank mean, one AdamW step from the partitioned initial
weight.

test_fullsize_whole_buckets: the workloads' own settings, clipping on
(max_norm 1.0) and their step counts (5 AdamW steps for the many-small
list).  The oracle's global norm is streamed over every reduce bucket
(oracle.step.bucket_sq_counts on the N rank buffers of each bucket, read
back from the device pool the shared generator filled); its clip
coefficient drives the oracle's Adam on whole buckets.  No value the
device computes is an input of the oracle.
"""
from __future__ import annotations

import gc
import os
from concurrent.futures import ThreadPoolExecutor

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
        # the same coefficient bits on both sides: the same float32 operations
        H.assert_state({"master": got["p"][data], "exp_avg": got["m"][data],
                        "exp_avg_sq": got["v"][data]},
                       {"master": p1, "exp_avg": m1, "exp_avg_sq": v1}, None,
                       f"{name} sampled", True, keys=("master", "exp_avg", "exp_avg_sq"))
        H.assert_16bit(got["ps"].view(np.uint16)[data], pb, "param_shards", w.dtype, True)
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
            got_pm = dw.pm.index_select(0, pidx2).cpu().numpy()
            assert np.array_equal(got_pm.view(np.uint32), pp1.view(np.uint32)), "p_master"
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


def _bucket_rows(dw, op, b):
    """The N rank gradient buffers of bucket b, read back from the device
    pool (input data: the shared generator filled it)."""
    L = op.bucket_buf_elems[b]
    rows = torch.stack([dw.pool[dw.offs[b][k]:dw.offs[b][k] + L] for k in range(op.n_ranks)])
    return list(rows.cpu().numpy().view(np.uint16))


def oracle_norm_streamed(dw, op, max_norm, scale):
    """The oracle's (norm, coef, skip) over every reduce bucket: the rank
    buffers are read back one bucket at a time and handed to the oracle's
    per-bucket counts, several buckets at once on host threads (numpy
    releases the interpreter lock in its array loops); counts add up in any
    order."""
    nb = len(op.reduce_buckets)
    workers = max(1, min(16, os.cpu_count() or 1))
    counts = np.zeros(1 << 15, dtype=np.int64)
    with ThreadPoolExecutor(workers) as ex:
        pending = []
        for b in range(nb):
            pending.append(ex.submit(ostep.bucket_sq_counts, op, b, _bucket_rows(dw, op, b)))
            if len(pending) >= 2 * workers:
                counts += pending.pop(0).result()
        for f in pending:
            counts += f.result()
    return ostep.clip_from_sumsq(ostep.sumsq_from_counts(counts, op.dtype), max_norm, scale)


@pytest.mark.parametrize("name", ["llama_layer", "many_small", "llama3_16_layers", "llama3_8b",
                                  "llama3_8b_fp16", "llama3_8b_hsdp"])
def test_fullsize_whole_buckets(name):
    """Every element of whole reduce buckets at full size (the first two,
    the middle one, the last one and every 64th), with the workload's
    clipping and step count: the norm against the oracle's streamed norm,
    the reduced gradient bit for bit, the fp32 master / moments and the cast
    parameter against the oracle's Adam with the oracle's coefficient (bit
    for bit when the device's coefficient has the same bits, as the device
    norm is accumulated without rounding error), and the parameter's place
    in the gathered replica."""
    w = workloads.WORKLOADS[name]()
    op = _oracle_plan(w)
    dw = bench.DeviceWorkload(w, "cuda:0", max_norm=w.max_norm)
    try:
        assert w.max_norm > 0
        N, S = op.n_ranks, op.S
        scale = float(w.loss_scale) if w.dtype == "fp16" else 1.0
        onorm, ocoef, oskip = oracle_norm_streamed(dw, op, w.max_norm, scale)
        assert not oskip and float(ocoef) * scale < 1.0          # clipping is active
        nb = len(op.reduce_buckets)
        picks = sorted({0, min(1, nb - 1), nb // 2, nb - 1, *range(0, nb, 64)})
        # the oracle's side of every picked entry: reduced gradient, initial state
        ref = []
        for b in picks:
            rows = _bucket_rows(dw, op, b)
            for ent in op.reduce_buckets[b]:
                p = op.params[ent.param]
                L = ent.e_hi - ent.e_lo
                e = np.arange(ent.e_lo, ent.e_hi, dtype=np.int64)
                vals = np.stack([r[ent.buf_off:ent.buf_off + L] for r in rows])
                gs_ref = ostep.reduce_mean_groups(vals, op.group, w.dtype)
                W = philox.weight_f32(w.seed, (p.input_off + e).astype(np.uint64), w.weight_sigma)
                if p.persistent:
                    idx = p.persist_off + e
                else:
                    idx = (e // p.ps) * S + p.shard_off + e % p.ps
                z = np.zeros_like(W)
                ref.append(dict(b=b, p=p, e=e, idx=torch.from_numpy(idx).to(dw.dev), gs=gs_ref,
                                st={"master": W, "exp_avg": z, "exp_avg_sq": z.copy()}))
        steps = w.steps
        checked = 0
        for t in range(1, steps + 1):
            dw.step()
            torch.cuda.synchronize()
            assert int(dw.d_flags[0]) == 0
            dnorm, dcoef = float(dw.d_norm[0]), float(dw.d_coef[0])
            assert abs(dnorm - float(onorm)) <= 1e-5 * float(onorm), (dnorm, float(onorm))
            exact = H.same_bits(dcoef, ocoef)
            print(f"{name} step {t}: norm {dnorm!r} (oracle {float(onorm)!r}), coefficient "
                  f"{dcoef!r} (oracle {float(ocoef)!r}): bits {'equal' if exact else 'differ'}")
            c = ostep.adam_consts(w.hparams(), t)
            for r in ref:
                p, e = r["p"], r["e"]
                prev = r["st"]
                p1, m1, v1, pb = ostep.adam_update(prev["master"], prev["exp_avg"],
                                                   prev["exp_avg_sq"], r["gs"], ocoef, c, w.dtype)
                r["st"] = {"master": p1, "exp_avg": m1, "exp_avg_sq": v1}
                if t < steps and t != 1:
                    continue             # compared after the first and the last step
                idx = r["idx"]
                if p.persistent:
                    bufs = (dw.gP, dw.pm, dw.pmm, dw.pmv, dw.pP)
                else:
                    bufs = (dw.gs, dw.master, dw.m, dw.v, dw.ps)
                got_g, got_p, got_m, got_v, got_ps = (x.index_select(0, idx).cpu().numpy()
                                                      for x in bufs)
                assert np.array_equal(got_g.view(np.uint16), r["gs"]), (r["b"], p.index)
                H.assert_state({"master": got_p, "exp_avg": got_m, "exp_avg_sq": got_v},
                               r["st"], prev, f"{name} step {t} bucket {r['b']} param {p.index}",
                               exact, keys=("master", "exp_avg", "exp_avg_sq"))
                pbits = got_ps.view(np.uint16)
                H.assert_16bit(pbits, pb, "params", w.dtype, exact)
                if not p.persistent:
                    fl = dw.flat.index_select(0, torch.from_numpy(p.flat_off + e).to(dw.dev))
                    assert np.array_equal(fl.cpu().numpy().view(np.uint16), pbits)
                checked += len(e)
        assert checked > 0
    finally:
        del dw
        gc.collect()
        torch.cuda.empty_cache()


@pytest.mark.parametrize("name", ["many_small", "llama3_8b", "llama3_8b_hsdp"])
def test_fullsize_per_bucket_calls_equal_fused(name):
    """zs_reduce_scatter bucket by bucket, at full size, gives the fused
    launch's results bit for bit: every reduced gradient and every tile's
    norm partial.  The per-bucket launches take each bucket's tiles largest
    first; where a bucket's CTAs fit in one wave (the 8B lists) they also
    prefetch their first pass into L2 while they wait on the previous
    launch; many_small's buckets take several waves.  The fused launch is
    the one test_fullsize_whole_buckets checks against the oracle."""
    w = workloads.WORKLOADS[name]()
    dw = bench.DeviceWorkload(w, "cuda:0", max_norm=w.max_norm)
    try:
        nt = dw.info["n_tiles"]
        zs.zs_reduce_scatter_all(dw.plan, dw.ptr_table, dw.gs, dw.gP, dw.scratch)
        torch.cuda.synchronize()
        gs, gP = dw.gs.clone(), dw.gP.clone()
        part = dw.scratch[:nt].clone()
        # every element must be written again
        dw.gs.fill_(-1)
        dw.gP.fill_(-1)
        dw.scratch.fill_(float("nan"))
        for b in range(len(dw.buf_elems)):
            zs.zs_reduce_scatter(dw.plan, b, dw.bucket_ptrs(b), dw.gs, dw.gP, dw.scratch)
        torch.cuda.synchronize()
        assert torch.equal(dw.gs, gs)
        assert torch.equal(dw.gP, gP)
        assert torch.equal(dw.scratch[:nt].view(torch.int64), part.view(torch.int64))
    finally:
        del dw
        gc.collect()
        torch.cuda.empty_cache()
