// A1 — the partition plan, built on the host with integer arithmetic only.
//
// Definitions ([ZeRO-3 chapter] = "03 · ZeRO-3：参数分片与 all-gather 调度"):
//   ps = ceil(numel / N); rank r owns [r*ps, (r+1)*ps)            (§3.1 item 1)
//   persistent iff numel < param_persistence_threshold            (§5.3)
//   reduce buckets: ds_id order, closed when the next parameter would
//     exceed reduce_bucket_size; a larger parameter is cut into chunks of
//     reduce_bucket_size elements, one bucket each                 (§6.2)
//   gather buckets: partitioned parameters, N*ps elements each, closed at
//     prefetch_bucket_size; a larger parameter is gathered alone  (§5.2)
//   sub-groups: ds_id order, per-rank footprint (ps, or numel when
//     persistent), closed at sub_group_size                       (§6.1)
// plus the tile table the kernels walk.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>

#include "zs_internal.h"

namespace {

thread_local std::string g_last_error;

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t align8(int64_t x) { return (x + 7) / 8 * 8; }

void emit_partitioned_tiles(zs_plan &P, const ZsParam &p, const ZsEntry &e, int32_t bucket) {
    const int64_t N = P.G, ps = p.ps;   // shard owners
    if (ps == 0) return;
    // the bucket holding the last element also owns the padding numel..N*ps-1
    const int64_t hi = (e.e_hi == p.numel) ? N * ps : e.e_hi;
    for (int64_t r = e.e_lo / ps; r < N && r * ps < hi; ++r) {
        const int64_t lo_v = std::max(e.e_lo, r * ps), hi_v = std::min(hi, (r + 1) * ps);
        if (lo_v >= hi_v) continue;
        int64_t j = lo_v - r * ps;
        const int64_t jend = hi_v - r * ps;
        while (j < jend) {
            const int64_t jb = std::min(jend, (j / ZS_TILE_ELEMS + 1) * ZS_TILE_ELEMS);
            const int64_t ev = r * ps + j;
            ZsTile t;
            t.dst = r * P.S + p.shard_off + j;
            t.len = (int32_t)(jb - j + (jb == ps ? align8(ps) - ps : 0));
            t.valid = (int32_t)std::max<int64_t>(0, std::min(p.numel - ev, jb - j));
            t.src = e.buf_off + (ev - e.e_lo);
            t.flat = p.flat_off + ev;
            t.flat_len = (int32_t)(jb - j);
            t.win = p.input_off + ev;
            t.bucket = bucket;
            P.tiles.push_back(t);
            j = jb;
        }
    }
}

void emit_persistent_tiles(zs_plan &P, const ZsParam &p, const ZsEntry &e, int32_t bucket) {
    int64_t a = e.e_lo;
    while (a < e.e_hi) {
        const int64_t b = std::min(e.e_hi, (a / ZS_TILE_ELEMS + 1) * ZS_TILE_ELEMS);
        ZsTile t;
        t.dst = p.persist_off + a;
        t.len = (int32_t)(b - a + (b == p.numel ? align8(p.numel) - p.numel : 0));
        t.valid = (int32_t)(b - a);
        t.src = e.buf_off + (a - e.e_lo);
        t.flat = -1;
        t.flat_len = 0;
        t.win = p.input_off + a;
        t.bucket = bucket;
        P.tiles.push_back(t);
        a = b;
    }
}

zs_status build(zs_plan &P, int32_t n, const int64_t *numel, const int64_t *ds_id) {
    const zs_config &c = P.cfg;
    // every layout is over the G shard owners of a replica group
    P.G = c.shard_group_size > 0 ? c.shard_group_size : c.n_ranks;
    const int64_t N = P.G;
    P.params.resize(n);
    for (int32_t i = 0; i < n; ++i) {
        ZsParam &p = P.params[i];
        std::memset(&p, 0, sizeof(p));
        p.numel = numel[i];
        p.ds_id = ds_id ? ds_id[i] : i;
        p.persistent = numel[i] < c.param_persistence_threshold ? 1 : 0;
        p.shard_off = p.persist_off = p.flat_off = -1;
        p.sub_group = p.gather_bucket = p.first_rb = -1;
    }
    P.order.resize(n);
    for (int32_t i = 0; i < n; ++i) P.order[i] = i;
    std::stable_sort(P.order.begin(), P.order.end(),
                     [&](int32_t a, int32_t b) { return P.params[a].ds_id < P.params[b].ds_id; });
    for (int32_t k = 1; k < n; ++k)
        if (P.params[P.order[k]].ds_id == P.params[P.order[k - 1]].ds_id)
            return zs_fail(ZS_EINVAL, "zs_build_partition: duplicate ds_id %lld",
                           (long long)P.params[P.order[k]].ds_id);

    // layouts
    int64_t s_run = 0, p_run = 0, f_run = 0, w_run = 0;
    for (int32_t k = 0; k < n; ++k) {
        ZsParam &p = P.params[P.order[k]];
        p.position = k;
        p.input_off = w_run;
        w_run += p.numel;
        if (p.persistent) {
            p.persist_off = p_run;
            p_run += align8(p.numel);
            P.Pn += p.numel;
        } else {
            p.ps = ceil_div(p.numel, N);
            p.pad = N * p.ps - p.numel;
            p.shard_off = s_run;
            s_run += align8(p.ps);
            P.S_logical += p.ps;
            p.flat_off = f_run;
            f_run += N * p.ps;
            P.padding += p.pad;
        }
    }
    P.S = s_run;
    P.Pn_alloc = p_run;
    P.flat_elems = f_run;
    P.psi = w_run;

    // reduce buckets (entries first, tiles after the layout is known)
    const int64_t B = c.reduce_bucket_size;
    std::vector<ZsEntry> cur;
    int64_t cur_n = 0;
    auto close = [&]() {
        if (cur.empty()) return;
        ZsBucket b{};
        b.first_entry = (int32_t)P.entries.size();
        b.n_entries = (int32_t)cur.size();
        int64_t off = 0;
        for (ZsEntry &e : cur) {
            e.buf_off = off;
            off += align8(e.e_hi - e.e_lo);
            b.grad_elems += e.e_hi - e.e_lo;
            P.entries.push_back(e);
        }
        b.buf_elems = off;
        P.buckets.push_back(b);
        cur.clear();
        cur_n = 0;
    };
    for (int32_t k = 0; k < n; ++k) {
        const int32_t i = P.order[k];
        const int64_t m = P.params[i].numel;
        if (m > B) {
            close();
            for (int64_t ch = 0; ch < ceil_div(m, B); ++ch) {
                cur.push_back(ZsEntry{i, ch * B, std::min((ch + 1) * B, m), 0});
                close();
            }
            continue;
        }
        if (!cur.empty() && cur_n + m > B) close();
        cur.push_back(ZsEntry{i, 0, m, 0});
        cur_n += m;
    }
    close();
    for (int32_t b = 0; b < (int32_t)P.buckets.size(); ++b) {
        ZsBucket &bk = P.buckets[b];
        bk.first_tile = (int64_t)P.tiles.size();
        for (int32_t q = 0; q < bk.n_entries; ++q) {
            const ZsEntry &e = P.entries[bk.first_entry + q];
            ZsParam &p = P.params[e.param];
            if (p.first_rb < 0) p.first_rb = b;
            p.n_rb += 1;
            if (p.persistent)
                emit_persistent_tiles(P, p, e, b);
            else
                emit_partitioned_tiles(P, p, e, b);
        }
        bk.n_tiles = (int64_t)P.tiles.size() - bk.first_tile;
        P.max_buf = std::max(P.max_buf, bk.buf_elems);
    }
    if (P.tiles.size() > (size_t)INT32_MAX)
        return zs_fail(ZS_EINVAL, "zs_build_partition: %zu work tiles exceed the int32 launch order",
                       P.tiles.size());
    // the reduce-scatter's launch order: per bucket, most valid elements
    // first (then longest, then table order)
    P.rs_order.resize(P.tiles.size());
    for (const ZsBucket &bk : P.buckets) {
        int32_t *o = P.rs_order.data() + bk.first_tile;
        for (int64_t i = 0; i < bk.n_tiles; ++i) o[i] = (int32_t)(bk.first_tile + i);
        std::stable_sort(o, o + bk.n_tiles, [&P](int32_t a, int32_t b) {
            const ZsTile &x = P.tiles[a], &y = P.tiles[b];
            return x.valid != y.valid ? x.valid > y.valid : x.len > y.len;
        });
    }

    // gather buckets
    const int64_t G = c.prefetch_bucket_size;
    int64_t g_n = 0;
    for (int32_t k = 0; k < n; ++k) {
        const int32_t i = P.order[k];
        ZsParam &p = P.params[i];
        if (p.persistent) continue;
        const int64_t size = N * p.ps;
        if (P.gathers.empty() || (P.gathers.back().n > 0 && g_n + size > G)) {
            ZsGather g{};
            g.first = (int32_t)P.gather_params.size();
            g.flat_off = p.flat_off;
            P.gathers.push_back(g);
            g_n = 0;
        }
        ZsGather &g = P.gathers.back();
        P.gather_params.push_back(i);
        g.n += 1;
        g.flat_elems += size;
        g_n += size;
        p.gather_bucket = (int32_t)P.gathers.size() - 1;
    }
    for (const ZsGather &g : P.gathers) P.max_gather = std::max(P.max_gather, g.flat_elems);

    // sub-groups
    const int64_t U = c.sub_group_size;
    int64_t u_n = 0, s_cur = 0, p_cur = 0;
    for (int32_t k = 0; k < n; ++k) {
        const int32_t i = P.order[k];
        ZsParam &p = P.params[i];
        const int64_t w = p.persistent ? p.numel : p.ps;
        if (P.sub_groups.empty() || (P.sub_groups.back().n > 0 && u_n + w > U)) {
            ZsSubGroup s{};
            s.first = k;
            s.s_lo = s.s_hi = s_cur;
            s.p_lo = s.p_hi = p_cur;
            P.sub_groups.push_back(s);
            u_n = 0;
        }
        ZsSubGroup &s = P.sub_groups.back();
        s.n += 1;
        u_n += w;
        if (p.persistent)
            p_cur = p.persist_off + align8(p.numel);
        else
            s_cur = p.shard_off + align8(p.ps);
        s.s_hi = s_cur;
        s.p_hi = p_cur;
        p.sub_group = (int32_t)P.sub_groups.size() - 1;
    }
    P.n_level1 = std::max<int64_t>(1, ceil_div((int64_t)P.tiles.size(), ZS_LEVEL1_CHUNK));
    return ZS_OK;
}

}  // namespace

zs_status zs_fail(zs_status status, const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return status;
}

void zs_clear_error() { g_last_error.clear(); }

extern "C" {

const char *zs_last_error(void) { return g_last_error.c_str(); }

const char *zs_version(void) { return "libzs 0.1 (sm_103a)"; }

void zs_default_config(zs_config *cfg, int32_t n_ranks) {
    if (!cfg) return;
    cfg->n_ranks = n_ranks;
    cfg->dtype = ZS_DTYPE_BF16;
    cfg->shard_group_size = 0;
    cfg->reserved = 0;
    cfg->param_persistence_threshold = 100000;
    cfg->reduce_bucket_size = 5000000;
    cfg->prefetch_bucket_size = 50000000;
    cfg->sub_group_size = 1000000000;
}

zs_status zs_build_partition(const zs_config *cfg, int32_t n_params, const int64_t *numel,
                             const int64_t *ds_id, zs_plan **out) {
    if (!cfg || !out) return zs_fail(ZS_EINVAL, "zs_build_partition: NULL config or output");
    *out = nullptr;
    if (cfg->n_ranks < 1) return zs_fail(ZS_EINVAL, "zs_build_partition: n_ranks must be >= 1");
    if (cfg->reserved != 0) return zs_fail(ZS_EINVAL, "zs_build_partition: reserved field must be 0");
    if (cfg->shard_group_size < 0 ||
        (cfg->shard_group_size > 0 && cfg->n_ranks % cfg->shard_group_size != 0))
        return zs_fail(ZS_EINVAL, "zs_build_partition: shard_group_size %d must divide n_ranks %d",
                       cfg->shard_group_size, cfg->n_ranks);
    if (cfg->dtype != ZS_DTYPE_BF16 && cfg->dtype != ZS_DTYPE_FP16)
        return zs_fail(ZS_EINVAL, "zs_build_partition: dtype must be ZS_DTYPE_BF16 or ZS_DTYPE_FP16");
    if (cfg->reduce_bucket_size < 1 || cfg->prefetch_bucket_size < 1 || cfg->sub_group_size < 1)
        return zs_fail(ZS_EINVAL, "zs_build_partition: bucket and sub-group sizes must be >= 1");
    if (n_params < 0 || (n_params > 0 && !numel))
        return zs_fail(ZS_EINVAL, "zs_build_partition: bad parameter list");
    for (int32_t i = 0; i < n_params; ++i)
        if (numel[i] < 0) return zs_fail(ZS_EINVAL, "zs_build_partition: numel[%d] < 0", i);
    zs_plan *P = new (std::nothrow) zs_plan();
    if (!P) return zs_fail(ZS_ENOMEM, "zs_build_partition: out of host memory");
    P->cfg = *cfg;
    zs_status st;
    try {
        st = build(*P, n_params, numel, ds_id);
    } catch (const std::bad_alloc &) {
        st = zs_fail(ZS_ENOMEM, "zs_build_partition: out of host memory");
    }
    if (st != ZS_OK) {
        delete P;
        return st;
    }
    *out = P;
    zs_clear_error();
    return ZS_OK;
}

void zs_free_plan(zs_plan *plan) { delete plan; }

zs_status zs_plan_info(const zs_plan *P, zs_plan_info_t *o) {
    if (!P || !o) return zs_fail(ZS_EINVAL, "zs_plan_info: NULL argument");
    std::memset(o, 0, sizeof(*o));
    o->n_ranks = P->cfg.n_ranks;
    o->n_params = (int32_t)P->params.size();
    o->n_reduce_buckets = (int32_t)P->buckets.size();
    o->n_gather_buckets = (int32_t)P->gathers.size();
    o->n_sub_groups = (int32_t)P->sub_groups.size();
    o->dtype = P->cfg.dtype;
    o->shard_group_size = P->G;
    o->psi = P->psi;
    o->shard_elems = P->S;
    o->shard_elems_logical = P->S_logical;
    o->persist_elems = P->Pn_alloc;
    o->persist_elems_logical = P->Pn;
    o->flat_elems = P->flat_elems;
    o->padding_elems = P->padding;
    o->max_bucket_buf_elems = P->max_buf;
    o->max_gather_elems = P->max_gather;
    o->bytes_per_rank = 16 * (P->S_logical + P->Pn);
    o->n_tiles = (int64_t)P->tiles.size();
    o->device_table_bytes = zs_table_bytes((int64_t)P->tiles.size());
    o->norm_scratch_elems = (int64_t)P->tiles.size() + P->n_level1;
    return ZS_OK;
}

zs_status zs_param_info(const zs_plan *P, int32_t i, zs_param_info_t *o) {
    if (!P || !o) return zs_fail(ZS_EINVAL, "zs_param_info: NULL argument");
    if (i < 0 || i >= (int32_t)P->params.size())
        return zs_fail(ZS_EINVAL, "zs_param_info: parameter %d out of range", i);
    const ZsParam &p = P->params[i];
    std::memset(o, 0, sizeof(*o));
    o->numel = p.numel;
    o->ds_id = p.ds_id;
    o->partition_size = p.ps;
    o->padding = p.pad;
    o->shard_offset = p.shard_off;
    o->persist_offset = p.persist_off;
    o->flat_offset = p.flat_off;
    o->input_offset = p.input_off;
    o->persistent = p.persistent;
    o->position = p.position;
    o->sub_group = p.sub_group;
    o->gather_bucket = p.gather_bucket;
    o->first_reduce_bucket = p.first_rb;
    o->n_reduce_buckets = p.n_rb;
    return ZS_OK;
}

zs_status zs_param_at(const zs_plan *P, int32_t pos, int32_t *param) {
    if (!P || !param) return zs_fail(ZS_EINVAL, "zs_param_at: NULL argument");
    if (pos < 0 || pos >= (int32_t)P->order.size())
        return zs_fail(ZS_EINVAL, "zs_param_at: position %d out of range", pos);
    *param = P->order[pos];
    return ZS_OK;
}

zs_status zs_bucket_info(const zs_plan *P, int32_t b, zs_bucket_info_t *o) {
    if (!P || !o) return zs_fail(ZS_EINVAL, "zs_bucket_info: NULL argument");
    if (b < 0 || b >= (int32_t)P->buckets.size())
        return zs_fail(ZS_EINVAL, "zs_bucket_info: bucket %d out of range", b);
    const ZsBucket &k = P->buckets[b];
    std::memset(o, 0, sizeof(*o));
    o->n_entries = k.n_entries;
    o->buf_elems = k.buf_elems;
    o->grad_elems = k.grad_elems;
    o->first_tile = k.first_tile;
    o->n_tiles = k.n_tiles;
    return ZS_OK;
}

zs_status zs_bucket_entry(const zs_plan *P, int32_t b, int32_t q, int32_t *param, int64_t *lo,
                          int64_t *hi, int64_t *off) {
    if (!P || !param || !lo || !hi || !off) return zs_fail(ZS_EINVAL, "zs_bucket_entry: NULL argument");
    if (b < 0 || b >= (int32_t)P->buckets.size() || q < 0 || q >= P->buckets[b].n_entries)
        return zs_fail(ZS_EINVAL, "zs_bucket_entry: (%d, %d) out of range", b, q);
    const ZsEntry &e = P->entries[P->buckets[b].first_entry + q];
    *param = e.param;
    *lo = e.e_lo;
    *hi = e.e_hi;
    *off = e.buf_off;
    return ZS_OK;
}

zs_status zs_gather_bucket_info(const zs_plan *P, int32_t g, zs_gather_bucket_info_t *o) {
    if (!P || !o) return zs_fail(ZS_EINVAL, "zs_gather_bucket_info: NULL argument");
    if (g < 0 || g >= (int32_t)P->gathers.size())
        return zs_fail(ZS_EINVAL, "zs_gather_bucket_info: gather bucket %d out of range", g);
    std::memset(o, 0, sizeof(*o));
    o->n_params = P->gathers[g].n;
    o->flat_offset = P->gathers[g].flat_off;
    o->flat_elems = P->gathers[g].flat_elems;
    return ZS_OK;
}

zs_status zs_gather_bucket_param(const zs_plan *P, int32_t g, int32_t i, int32_t *param) {
    if (!P || !param) return zs_fail(ZS_EINVAL, "zs_gather_bucket_param: NULL argument");
    if (g < 0 || g >= (int32_t)P->gathers.size() || i < 0 || i >= P->gathers[g].n)
        return zs_fail(ZS_EINVAL, "zs_gather_bucket_param: (%d, %d) out of range", g, i);
    *param = P->gather_params[P->gathers[g].first + i];
    return ZS_OK;
}

zs_status zs_sub_group_info(const zs_plan *P, int32_t s, zs_sub_group_info_t *o) {
    if (!P || !o) return zs_fail(ZS_EINVAL, "zs_sub_group_info: NULL argument");
    if (s < 0 || s >= (int32_t)P->sub_groups.size())
        return zs_fail(ZS_EINVAL, "zs_sub_group_info: sub-group %d out of range", s);
    const ZsSubGroup &g = P->sub_groups[s];
    std::memset(o, 0, sizeof(*o));
    o->n_params = g.n;
    o->shard_lo = g.s_lo;
    o->shard_hi = g.s_hi;
    o->persist_lo = g.p_lo;
    o->persist_hi = g.p_hi;
    return ZS_OK;
}

zs_status zs_plan_table(const zs_plan *P, void *host_out, int64_t bytes) {
    if (!P || (!host_out && bytes > 0)) return zs_fail(ZS_EINVAL, "zs_plan_table: NULL argument");
    const int64_t n = (int64_t)P->tiles.size();
    const int64_t need = zs_table_tile_bytes(n);
    if (bytes < need) return zs_fail(ZS_EINVAL, "zs_plan_table: %lld bytes < %lld", (long long)bytes,
                                     (long long)need);
    if (need) std::memcpy(host_out, P->tiles.data(), (size_t)need);
    if (n && bytes >= zs_table_bytes(n))
        std::memcpy(static_cast<char *>(host_out) + need, P->rs_order.data(), (size_t)n * 4);
    return ZS_OK;
}

}  // extern "C"
