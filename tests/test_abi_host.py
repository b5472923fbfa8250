"""Host-side checks of libzs (no GPU needed): every symbol include/zs.h
declares is exported, the C++ plan equals the oracle's plan, the work table
partitions shard and persistent space exactly, and argument errors are
reported before any device work."""
from __future__ import annotations

import ctypes
import os
import re

import numpy as np
import pytest

from oracle import plan as oplan
from synth import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
zs = pytest.importorskip("zero_sharded_optimizer_bucket_gb300")


def _declared_functions():
    text = open(os.path.join(ROOT, "include", "zs.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s*(zs_[a-z0-9_]+)\s*\(",
                       text, flags=re.M)
    return sorted(set(names))


def test_library_exports_every_declared_symbol():
    names = _declared_functions()
    assert len(names) >= 20
    lib = ctypes.CDLL(zs.LIB_PATH)
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing


def _cpp_plan(numel, N, ds_id=None, **kw):
    cfg = zs.zs_default_config(N)
    for k, v in kw.items():
        setattr(cfg, k, v)
    return zs.zs_build_partition(cfg, numel, ds_id)


def _compare(numel, N, ds_id=None, threshold=100_000, B=5_000_000, G=50_000_000, U=10**9,
             group=0):
    op = oplan.build_partition(numel, N, threshold=threshold, reduce_bucket_size=B,
                               prefetch_bucket_size=G, sub_group_size=U, ds_id=ds_id,
                               shard_group_size=group or None)
    cp = _cpp_plan(numel, N, ds_id, param_persistence_threshold=threshold,
                   reduce_bucket_size=B, prefetch_bucket_size=G, sub_group_size=U,
                   shard_group_size=group)
    info = zs.zs_plan_info(cp)
    assert info["n_params"] == len(numel)
    assert info["n_ranks"] == N and info["shard_group_size"] == op.group
    assert info["shard_elems"] == op.S and info["shard_elems_logical"] == op.S_logical
    assert info["persist_elems"] == op.Pn_alloc and info["persist_elems_logical"] == op.Pn
    assert info["flat_elems"] == op.flat_elems and info["psi"] == op.psi
    assert info["padding_elems"] == op.padding_elems
    assert info["bytes_per_rank"] == op.bytes_per_rank()
    assert info["n_reduce_buckets"] == len(op.reduce_buckets)
    assert info["n_gather_buckets"] == len(op.gather_buckets)
    assert info["n_sub_groups"] == len(op.sub_groups)
    for k, i in enumerate(op.order):
        assert zs.zs_param_at(cp, k) == i
    for p in op.params:
        q = zs.zs_param_info(cp, p.index)
        assert (q["numel"], q["ds_id"], q["persistent"]) == (p.numel, p.ds_id, int(p.persistent))
        assert q["partition_size"] == p.ps and q["padding"] == p.pad
        assert q["shard_offset"] == p.shard_off and q["persist_offset"] == p.persist_off
        assert q["flat_offset"] == p.flat_off and q["input_offset"] == p.input_off
        assert q["sub_group"] == p.sub_group and q["gather_bucket"] == p.gather_bucket
        assert q["n_reduce_buckets"] == len(p.reduce_buckets)
        if p.reduce_buckets:
            assert q["first_reduce_bucket"] == p.reduce_buckets[0]
    for b, ents in enumerate(op.reduce_buckets):
        bi = zs.zs_bucket_info(cp, b)
        assert bi["n_entries"] == len(ents) and bi["buf_elems"] == op.bucket_buf_elems[b]
        for q, e in enumerate(ents):
            assert zs.zs_bucket_entry(cp, b, q) == (e.param, e.e_lo, e.e_hi, e.buf_off)
    for g, gb in enumerate(op.gather_buckets):
        gi = zs.zs_gather_bucket_info(cp, g)
        assert gi["n_params"] == len(gb.params) and gi["flat_offset"] == gb.flat_off
        assert gi["flat_elems"] == gb.flat_elems
        assert [zs.zs_gather_bucket_param(cp, g, i) for i in range(len(gb.params))] == gb.params
    for s, sg in enumerate(op.sub_groups):
        si = zs.zs_sub_group_info(cp, s)
        assert (si["n_params"], si["shard_lo"], si["shard_hi"], si["persist_lo"], si["persist_hi"]) \
            == (len(sg.params), sg.s_lo, sg.s_hi, sg.p_lo, sg.p_hi)
    return op, cp


@pytest.mark.parametrize("seed", range(20))
def test_cpp_plan_equals_oracle_random(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(0, 60))
    numel = [int(x) for x in rng.integers(0, 5000, size=n)]
    N = int(rng.choice([1, 2, 3, 4, 5, 8, 16, 64, 256]))
    ds = [int(x) for x in rng.permutation(n) * 7 - 3] if seed % 2 else None
    op, cp = _compare(numel, N, ds, threshold=int(rng.integers(0, 300)),
                      B=int(rng.integers(1, 6000)), G=int(rng.integers(1, 30000)),
                      U=int(rng.integers(1, 4000)))
    _check_tiles(op, cp)


@pytest.mark.parametrize("name", ["tiny", "llama_layer", "llama3_16_layers", "llama3_8b"])
def test_cpp_plan_equals_oracle_workloads(name):
    w = workloads.WORKLOADS[name]()
    _compare(w.numel, w.n_ranks, threshold=w.persistence_threshold)


@pytest.mark.parametrize("N,group", [(8, 2), (16, 4), (12, 3), (64, 8), (6, 1)])
def test_cpp_plan_equals_oracle_hsdp(N, group):
    rng = np.random.default_rng(N * 7 + group)
    numel = [int(x) for x in rng.integers(0, 4000, size=40)]
    op, cp = _compare(numel, N, threshold=30, B=1500, G=6000, U=900, group=group)
    _check_tiles(op, cp)


def test_hsdp_group_must_divide_n():
    with pytest.raises(zs.ZsError):
        _cpp_plan([10], 8, shard_group_size=3)


def test_cpp_plan_equals_oracle_many_small():
    w = workloads.many_small(2000)
    op, cp = _compare(w.numel, w.n_ranks, threshold=w.persistence_threshold)
    _check_tiles(op, cp)


def test_llama3_8b_plan_shape():
    w = workloads.llama3_8b()
    info = zs.zs_plan_info(_cpp_plan(w.numel, w.n_ranks))
    assert info["n_sub_groups"] == 1
    # per layer: q 4 chunks, k 1, v 1, o 4, gate/up/down 12 each, both norms 1
    # = 47; embed and lm_head ceil(525336576 / 5e6) = 106 chunks each; the
    # final norm joins the last layer's norm bucket
    assert info["n_reduce_buckets"] == 106 + 32 * 47 + 106
    # gather buckets per layer: [q, k, v, o] (41.9M <= 5e7), then gate, up and
    # down (58.7M each) alone; embed and lm_head alone; the norms persist
    assert info["n_gather_buckets"] == 32 * 4 + 2
    assert info["psi"] == 8_030_261_248


def _check_launch_order(cp, t):
    """The reduce-scatter's launch order: within each bucket a permutation
    of the bucket's tiles, most valid elements first, then longest, then
    table order."""
    order = zs.zs_plan_launch_order(cp)
    assert order.size == len(t)
    for b in range(zs.zs_plan_info(cp)["n_reduce_buckets"]):
        bi = zs.zs_bucket_info(cp, b)
        f, n = bi["first_tile"], bi["n_tiles"]
        o = order[f:f + n].astype(np.int64)
        assert sorted(o.tolist()) == list(range(f, f + n)), b
        key = [(-int(t[i]["valid"]), -int(t[i]["len"]), int(i)) for i in o]
        assert key == sorted(key), b


def _check_tiles(op, cp):
    """Tiles cover every shard-space and persistent-space element exactly
    once, and each valid element maps to the bucket position and input
    position the oracle's definitions give."""
    t = zs.zs_plan_table(cp)
    _check_launch_order(cp, t)
    N, S = op.group, op.S
    cover = np.zeros(N * S, dtype=np.int32)
    pcover = np.zeros(op.Pn_alloc, dtype=np.int32)
    # expected source of each valid shard element: (bucket, src index, input index)
    for x in t:
        L, V = int(x["len"]), int(x["valid"])
        assert 0 <= V <= L
        d = int(x["dst"])
        if x["flat"] < 0:
            pcover[d:d + L] += 1
        else:
            cover[d:d + L] += 1
            assert x["flat_len"] <= L
    assert np.all(cover == 1) and np.all(pcover == 1)
    # spot-check the element mappings against the oracle's bucket entries
    pos = {}
    for b, ents in enumerate(op.reduce_buckets):
        for e in ents:
            pos[(e.param, b)] = e
    rng = np.random.default_rng(0)
    for x in t[rng.permutation(len(t))[:200]] if len(t) else []:
        b = int(x["bucket"])
        V, d = int(x["valid"]), int(x["dst"])
        for li in sorted(set([0, max(V - 1, 0), V // 2])):
            if li >= V:
                continue
            src = int(x["src"]) + li
            ents = [e for e in op.reduce_buckets[b] if e.buf_off <= src < e.buf_off + e.e_hi - e.e_lo]
            assert len(ents) == 1
            e = ents[0]
            p = op.params[e.param]
            el = e.e_lo + (src - e.buf_off)          # element of the parameter
            assert int(x["win"]) + li == p.input_off + el
            if p.persistent:
                assert d + li == p.persist_off + el
            else:
                r, col = oplan.owner(op, p.index, el)
                assert d + li == r * S + col
                assert int(x["flat"]) + li == p.flat_off + el


# ---------------------------------------------------------- errors -------
def test_build_partition_errors():
    with pytest.raises(zs.ZsError) as ei:
        _cpp_plan([10, -1], 4)
    assert ei.value.status == zs.ZS_EINVAL
    with pytest.raises(zs.ZsError):
        _cpp_plan([10, 20], 4, ds_id=[3, 3])
    with pytest.raises(zs.ZsError):
        _cpp_plan([10], 0)
    with pytest.raises(zs.ZsError):
        _cpp_plan([10], 4, reduce_bucket_size=0)
    empty = _cpp_plan([], 8)
    info = zs.zs_plan_info(empty)
    assert info["n_params"] == 0 and info["n_tiles"] == 0 and info["n_reduce_buckets"] == 0


def test_query_errors():
    plan = _cpp_plan([100, 2000], 4, param_persistence_threshold=0)
    for f, args in [(zs.zs_param_info, (2,)), (zs.zs_param_info, (-1,)),
                    (zs.zs_bucket_info, (5,)), (zs.zs_bucket_entry, (0, 9)),
                    (zs.zs_gather_bucket_info, (3,)), (zs.zs_sub_group_info, (1,)),
                    (zs.zs_param_at, (2,))]:
        with pytest.raises(zs.ZsError) as ei:
            f(plan, *args)
        assert ei.value.status == zs.ZS_EINVAL


def test_device_calls_reject_bad_arguments_before_any_launch():
    plan = _cpp_plan([100, 2000, 7], 4, param_persistence_threshold=50)
    # not uploaded
    with pytest.raises(zs.ZsError) as ei:
        zs.zs_reduce_scatter(plan, 0, [16] * 4, 16, 16)
    assert ei.value.status == zs.ZS_ESTATE
    zs.zs_plan_upload(plan, 4096, 1 << 20) if False else None
    # upload argument checks (no copy is made when they fail)
    with pytest.raises(zs.ZsError):
        zs.zs_plan_upload(plan, None, 1 << 20)
    with pytest.raises(zs.ZsError):
        zs.zs_plan_upload(plan, 8, 1 << 20)           # misaligned
    with pytest.raises(zs.ZsError):
        zs.zs_plan_upload(plan, 4096, 16)             # too small
    # pretend an upload happened at a fake aligned address: only host checks run below
    plan2 = _cpp_plan([], 4)
    zs.zs_plan_upload(plan2, None, 0)                 # empty plan needs no table
    with pytest.raises(zs.ZsError):
        zs.zs_reduce_scatter(plan2, 0, [16] * 4, 16, 16)   # no bucket 0
    with pytest.raises(zs.ZsError):
        zs.zs_adam_step(plan2, 3, dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                       weight_decay=0.0), 1, 16, 16, zs.make_state())
    with pytest.raises(zs.ZsError):
        zs.zs_adam_step(plan2, -1, dict(lr=1e-3, beta1=0.9, beta2=0.999, eps=1e-8,
                                        weight_decay=0.0), 0, 16, 16, zs.make_state())
    with pytest.raises(zs.ZsError):
        zs.zs_adam_step(plan2, -1, dict(lr=1e-3, beta1=1.0, beta2=0.999, eps=1e-8,
                                        weight_decay=0.0), 1, 16, 16, zs.make_state())
    with pytest.raises(zs.ZsError):
        zs.zs_all_gather_coalesced(plan2, [0], 16, 16, 100)
    with pytest.raises(zs.ZsError):
        zs.zs_grad_norm(plan2, None, None, None, False, 1.0, 16, 16, 16)


def test_wait_timeout_hook_checks_its_limit():
    for bad in (0, -1, 2_000_000_001):
        with pytest.raises(zs.ZsError) as ei:
            zs.zs_test_wait_timeout(bad)
        assert ei.value.status == zs.ZS_EINVAL


def test_parameter_larger_than_2_to_32_elements():
    """Offsets, chunk buckets and tiles of a parameter of 2^33 + 5 elements
    (beyond any 32-bit index), next to small ones: the plan equals the
    oracle's and its tiles cover every destination element once."""
    numel = [3000, 2 ** 33 + 5, 77, 2 ** 20 + 1]
    op, cp = _compare(numel, 16, threshold=100, B=50_000_000, G=60_000_000, U=2 ** 31)
    info = zs.zs_plan_info(cp)
    big = zs.zs_param_info(cp, 1)
    ps = -(-(2 ** 33 + 5) // 16)
    assert big["partition_size"] == ps and big["padding"] == 16 * ps - (2 ** 33 + 5)
    assert big["n_reduce_buckets"] == -(-(2 ** 33 + 5) // 50_000_000)
    assert info["flat_elems"] == sum(16 * -(-n // 16) for n in numel if n >= 100)
    tiles = zs.zs_plan_table(cp)
    part = tiles[tiles["flat"] >= 0]
    # every shard row of every partitioned parameter is tiled exactly once
    assert int(part["len"].astype(np.int64).sum()) == 16 * info["shard_elems"]
    assert int(tiles["valid"].astype(np.int64).sum()) == info["psi"]
