"""A1 partition plan of the oracle (integer logic only).

Definitions (each a reading of the pages; the design notes list them):

* Order.  Parameters are handled in ds_id order; the default ds_id is the
  parameter's index.  all_gather_coalesced sorts by ds_id so that every rank
  packs the same order ([ZeRO-3 chapter] §5.2 and §7, third bullet).
* Persistence.  A parameter with numel < param_persistence_threshold stays
  whole and is never partitioned ([ZeRO-3 chapter] §5.3, last paragraph).
* Partition.  Rank r owns flat elements [r*ps, (r+1)*ps) of a partitioned
  parameter ([ZeRO-3 chapter] §3.1, item 1) with ps = ceil(numel / N); the
  elements numel .. N*ps-1 are zero padding (the pages state the range but
  not ps; ceil is the smallest equal split that covers the tensor).
* Shard space.  All partition shards of one rank lie in one row of a [N][S]
  buffer (the flat gradient-partition buffer of [ZeRO-3 chapter] §6.1; the
  fp32 partitions of §6.1 use the same layout).  Parameter p occupies columns
  [S_p, S_p + ps_p); S_p is the running sum of ps rounded up to 8 elements
  (16 bytes), so that every shard starts 16-byte aligned.  The up-to-7
  alignment columns after a shard hold zero and are never used.
* Persistent space.  Persistent parameters lie whole, once, in a [Pn] buffer
  at offsets P_p = running sum of numel rounded up to 8.
* Model flat space.  The gathered parameters of the whole model, partitioned
  parameters only, in ds_id order: parameter p at F_p = running sum of N*ps
  (no alignment: a gathered parameter is the N shards back to back, and the
  view of the parameter is its first numel elements; [ZeRO-3 chapter] §5.2).
* Input space.  The full parameters of the model, all of them, in ds_id
  order at W_p = running sum of numel: the layout of the weights given to
  the partition step.
* Reduce buckets.  Gradients enter buckets in ds_id order ([ZeRO-3 chapter]
  §6.2, IPG bucket, reduce_bucket_size 5e6 from the [Core flow] config).  A
  bucket is closed when adding the next parameter would exceed
  reduce_bucket_size elements.  A parameter larger than reduce_bucket_size
  closes the open bucket and is split into element-range chunks
  [c*B, (c+1)*B), one bucket each.  Inside a bucket's gradient buffer each
  entry starts at a multiple of 8 elements.
* Gather buckets.  Partitioned parameters in ds_id order, closed when the
  next parameter's N*ps would exceed prefetch_bucket_size (5e7,
  [ZeRO-3 chapter] §5.2 item 3); a larger parameter is gathered alone.
* Sub-groups.  All parameters in ds_id order, weighted by their per-rank
  footprint (ps for a partitioned, numel for a persistent parameter), closed
  when the next would exceed sub_group_size (1e9, [ZeRO-3 chapter] §6.1).
* HSDP.  With shard_group_size G (a divisor of N; default N) the N ranks
  form N/G replica groups of G consecutive ranks: parameters are
  partitioned over the G ranks of a group, the groups hold identical
  replicas ([Core flow] §4: FSDP inside a group, DDP across groups).  Every
  layout above then uses G in place of N; the gradient mean still runs over
  all N ranks (see step.reduce_scatter).
"""
from __future__ import annotations

from dataclasses import dataclass, field


def _ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def _align8(x: int) -> int:
    return (x + 7) // 8 * 8


@dataclass
class Param:
    index: int
    ds_id: int
    numel: int
    persistent: bool
    ps: int = 0            # partition size (partitioned), 0 for persistent
    pad: int = 0           # N*ps - numel (partitioned)
    shard_off: int = -1    # S_p
    persist_off: int = -1  # P_p
    flat_off: int = -1     # F_p
    input_off: int = 0     # W_p
    sub_group: int = -1
    gather_bucket: int = -1
    reduce_buckets: list = field(default_factory=list)


@dataclass
class BucketEntry:
    param: int     # caller index
    e_lo: int      # first flat element of the parameter in this bucket
    e_hi: int      # one past the last
    buf_off: int   # offset of element e_lo in the bucket's gradient buffer


@dataclass
class SubGroup:
    params: list
    s_lo: int
    s_hi: int
    p_lo: int
    p_hi: int


@dataclass
class GatherBucket:
    params: list
    flat_off: int
    flat_elems: int


@dataclass
class Plan:
    n_ranks: int            # N: ranks that contribute gradients
    group: int              # G: ranks a parameter is partitioned over (N unless HSDP)
    dtype: str              # 16-bit storage of gradients and parameters: "bf16" | "fp16"
    threshold: int
    reduce_bucket_size: int
    prefetch_bucket_size: int
    sub_group_size: int
    params: list            # by caller index
    order: list             # caller indices in ds_id order
    S: int                  # shard row length (aligned)
    S_logical: int          # sum of ps
    Pn_alloc: int
    Pn: int                 # sum of persistent numel
    psi: int
    flat_elems: int
    input_elems: int
    reduce_buckets: list    # list of list of BucketEntry
    bucket_buf_elems: list
    gather_buckets: list
    sub_groups: list

    @property
    def padding_elems(self) -> int:
        return sum(p.pad for p in self.params if not p.persistent)

    def bytes_per_rank(self) -> int:
        """16 bytes per element a rank holds ([ZeRO-3 chapter] intro: 16Ψ/N;
        [Core flow] §1: 2 (param) + 2 (grad) + 12 (fp32 master, m, v))."""
        return 16 * self.S_logical + 16 * self.Pn


def build_partition(numel, n_ranks: int, threshold: int = 100_000,
                    reduce_bucket_size: int = 5_000_000,
                    prefetch_bucket_size: int = 50_000_000,
                    sub_group_size: int = 1_000_000_000, ds_id=None,
                    dtype: str = "bf16", shard_group_size: int = None) -> Plan:
    numel = [int(x) for x in numel]
    n = len(numel)
    if n_ranks < 1:
        raise ValueError("n_ranks must be >= 1")
    if reduce_bucket_size < 1 or prefetch_bucket_size < 1 or sub_group_size < 1:
        raise ValueError("bucket and sub-group sizes must be >= 1")
    if any(x < 0 for x in numel):
        raise ValueError("numel must be >= 0")
    if dtype not in ("bf16", "fp16"):
        raise ValueError("dtype must be bf16 or fp16")
    if ds_id is None:
        ds_id = list(range(n))
    ds_id = [int(x) for x in ds_id]
    if len(set(ds_id)) != n:
        raise ValueError("ds_id must be unique")
    order = sorted(range(n), key=lambda i: ds_id[i])
    group = n_ranks if not shard_group_size else int(shard_group_size)
    if group < 1 or n_ranks % group:
        raise ValueError("shard_group_size must divide n_ranks")
    N = group      # every layout below is over the shard owners of a group
    params = [Param(index=i, ds_id=ds_id[i], numel=numel[i],
                    persistent=numel[i] < threshold) for i in range(n)]

    s_run = p_run = f_run = w_run = 0
    S_logical = Pn = 0
    for i in order:
        p = params[i]
        p.input_off = w_run
        w_run += p.numel
        if p.persistent:
            p.persist_off = p_run
            p_run += _align8(p.numel)
            Pn += p.numel
        else:
            p.ps = _ceil_div(p.numel, N)
            p.pad = N * p.ps - p.numel
            p.shard_off = s_run
            s_run += _align8(p.ps)
            S_logical += p.ps
            p.flat_off = f_run
            f_run += N * p.ps

    # reduce buckets
    B = reduce_bucket_size
    buckets, cur, cur_n = [], [], 0

    def close():
        nonlocal cur, cur_n
        if cur:
            buckets.append(cur)
        cur, cur_n = [], 0

    for i in order:
        m = params[i].numel
        if m > B:
            close()
            for c in range(_ceil_div(m, B)):
                buckets.append([(i, c * B, min((c + 1) * B, m))])
            continue
        if cur and cur_n + m > B:
            close()
        cur.append((i, 0, m))
        cur_n += m
    close()
    reduce_buckets, buf_elems = [], []
    for b, ents in enumerate(buckets):
        off = 0
        row = []
        for (i, lo, hi) in ents:
            row.append(BucketEntry(i, lo, hi, off))
            params[i].reduce_buckets.append(b)
            off += _align8(hi - lo)
        reduce_buckets.append(row)
        buf_elems.append(off)

    # gather buckets
    G = prefetch_bucket_size
    gathers, cur, cur_n = [], [], 0
    for i in order:
        p = params[i]
        if p.persistent:
            continue
        size = N * p.ps
        if cur and cur_n + size > G:
            gathers.append(cur)
            cur, cur_n = [], 0
        cur.append(i)
        cur_n += size
    if cur:
        gathers.append(cur)
    gather_buckets = []
    for g, ids in enumerate(gathers):
        for i in ids:
            params[i].gather_bucket = g
        gather_buckets.append(GatherBucket(ids, params[ids[0]].flat_off,
                                           sum(N * params[i].ps for i in ids)))

    # sub-groups
    U = sub_group_size
    groups, cur, cur_n = [], [], 0
    for i in order:
        p = params[i]
        w = p.numel if p.persistent else p.ps
        if cur and cur_n + w > U:
            groups.append(cur)
            cur, cur_n = [], 0
        cur.append(i)
        cur_n += w
    if cur:
        groups.append(cur)
    sub_groups = []
    s_cur = p_cur = 0
    for g, ids in enumerate(groups):
        s_lo, p_lo = s_cur, p_cur
        for i in ids:
            p = params[i]
            p.sub_group = g
            if p.persistent:
                p_cur = p.persist_off + _align8(p.numel)
            else:
                s_cur = p.shard_off + _align8(p.ps)
        sub_groups.append(SubGroup(ids, s_lo, s_cur, p_lo, p_cur))

    return Plan(n_ranks=n_ranks, group=group, dtype=dtype, threshold=threshold, reduce_bucket_size=B,
                prefetch_bucket_size=G, sub_group_size=U, params=params,
                order=order, S=s_run, S_logical=S_logical, Pn_alloc=p_run, Pn=Pn,
                psi=sum(numel), flat_elems=f_run, input_elems=w_run,
                reduce_buckets=reduce_buckets, bucket_buf_elems=buf_elems,
                gather_buckets=gather_buckets, sub_groups=sub_groups)


def owner(plan: Plan, param: int, e: int):
    """(rank, column in the rank's shard row) of flat element e of a
    partitioned parameter: rank e // ps, offset e % ps ([ZeRO-3 chapter] §3.1)."""
    p = plan.params[param]
    r, j = divmod(e, p.ps)
    return r, p.shard_off + j
