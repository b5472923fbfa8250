// Gather scheduler: trace, fetch with prefetch, release by reuse distance
// ([ZeRO-3 chapter] §5.1-5.3, the PartitionedParameterCoordinator), run on
// two CUDA streams.  Host code only; the gathers are zs_all_gather_coalesced
// calls on the gather stream, ordered against the compute stream with
// events (a gather's output is waited for by the module that uses it; a
// gather that reuses released arena space waits for that release).
#include <algorithm>
#include <deque>
#include <new>
#include <utility>
#include <vector>

#include "zs_launch.h"

namespace {

struct Seg {
    int64_t off, size, rel;  // rel: latest release that freed part of it (-1 none)
};

}  // namespace

struct zs_sched {
    const zs_plan *P = nullptr;
    std::vector<std::vector<int32_t>> modules;
    std::vector<int64_t> module_numel;     // elements of each module's parameter uses
    zs_sched_config cfg{};
    uint16_t *arena = nullptr;             // NULL: plan only
    std::vector<int32_t> trace, recording;
    bool complete = false, invalid = false;
    int64_t pos = 0, queue_pos = 0;
    std::vector<int32_t> queue;            // parameter uses of the trace, in order
    std::vector<int64_t> queue_start;      // first queue entry of each trace position
    std::vector<char> live_flag;
    std::vector<int64_t> offset;
    std::vector<int32_t> producer;
    std::vector<Seg> free_;
    int64_t live = 0, ops = 0, releases = 0, arena_used = 0;
    std::deque<zs_sched_event> log;     // the most recent records (log_limit)
    int64_t log_cap = 0;                  // < 0: unlimited
    // CUDA events, pooled per pass: op_ev[op - pass_first_op] and
    // rel_ev[rel - pass_first_rel].  The first fetch of a pass makes the
    // gather stream wait for the compute stream (pass_ev), which covers
    // every release recorded before it, so older events are never needed.
    std::vector<cudaEvent_t> op_ev, rel_ev;
    cudaEvent_t pass_ev = nullptr;
    int64_t pass_first_op = 0, pass_first_rel = 0;
    void *cstream = nullptr, *gstream = nullptr;   // fixed at the first device call
    bool streams_set = false;
    zs_sched_stats_t st{};
};

namespace {

int64_t psize(const zs_sched *s, int32_t p) { return (int64_t)s->P->G * s->P->params[p].ps; }
bool gatherable(const zs_sched *s, int32_t p) {
    return !s->P->params[p].persistent && s->P->params[p].ps > 0;
}
int64_t numel(const zs_sched *s, int32_t p) { return s->P->params[p].numel; }

std::vector<int32_t> dedup(const std::vector<int32_t> &v) {
    std::vector<int32_t> out;
    for (int32_t p : v)
        if (std::find(out.begin(), out.end(), p) == out.end()) out.push_back(p);
    return out;
}

void sort_ds(const zs_sched *s, std::vector<int32_t> &v) {
    std::sort(v.begin(), v.end(), [&](int32_t a, int32_t b) {
        return s->P->params[a].position < s->P->params[b].position;
    });
}

// One block for the parameters (ds_id order).  Free space is a sorted list
// of segments tagged with the release that freed them; a block may span
// adjacent segments and waits for the latest of their releases.  The
// placement with the oldest such release (never used first), then the
// lowest offset, is taken.  On success the free list is updated and the
// offsets / the release to wait for are returned.
bool alloc(zs_sched *s, std::vector<int32_t> params, std::vector<int64_t> &offs, int64_t &waits) {
    sort_ds(s, params);
    int64_t total = 0;
    for (int32_t p : params) total += psize(s, p);
    const int64_t n = (int64_t)s->free_.size();
    int64_t bi = -1, bj = -1, bwait = 0, boff = 0, bacc = 0;
    for (int64_t i = 0; i < n; ++i) {
        int64_t acc = 0, wait = -1;
        for (int64_t j = i; j < n; ++j) {
            const Seg &g = s->free_[j];
            if (j > i && s->free_[j - 1].off + s->free_[j - 1].size != g.off) break;
            acc += g.size;
            wait = std::max(wait, g.rel);
            if (acc >= total) {
                const int64_t off = s->free_[i].off;
                if (bi < 0 || wait < bwait || (wait == bwait && off < boff)) {
                    bi = i, bj = j, bwait = wait, boff = off, bacc = acc;
                }
                break;
            }
        }
    }
    if (bi < 0) return false;
    const int64_t rest = bacc - total, rel_j = s->free_[bj].rel;
    s->free_.erase(s->free_.begin() + bi, s->free_.begin() + bj + 1);
    if (rest > 0) s->free_.insert(s->free_.begin() + bi, Seg{boff + total, rest, rel_j});
    waits = bwait;
    offs.clear();
    int64_t run = boff;
    for (int32_t p : params) {
        offs.push_back(run);
        run += psize(s, p);
    }
    return true;
}

void free_seg(zs_sched *s, int32_t p, int64_t rel) {
    s->free_.push_back(Seg{s->offset[p], psize(s, p), rel});
    std::sort(s->free_.begin(), s->free_.end(), [](const Seg &a, const Seg &b) { return a.off < b.off; });
    std::vector<Seg> merged;
    for (const Seg &g : s->free_) {  // merge neighbours freed by the same release
        if (!merged.empty() && merged.back().off + merged.back().size == g.off &&
            merged.back().rel == g.rel) {
            merged.back().size += g.size;
        } else {
            merged.push_back(g);
        }
    }
    s->free_.swap(merged);
    s->offset[p] = -1;
}

// Appends a log record, dropping the oldest beyond the log limit.
void log_event(zs_sched *s, const zs_sched_event &e) {
    s->log.push_back(e);
    if (s->log_cap >= 0 && (int64_t)s->log.size() > s->log_cap) s->log.pop_front();
}

zs_status cuda_err(cudaError_t e, const char *what) {
    return zs_fail(ZS_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

zs_status ensure_event(std::vector<cudaEvent_t> &v, int64_t idx) {
    while ((int64_t)v.size() <= idx) {
        cudaEvent_t e;
        const cudaError_t r = cudaEventCreateWithFlags(&e, cudaEventDisableTiming);
        if (r != cudaSuccess) return cuda_err(r, "zs_sched: cudaEventCreate");
        v.push_back(e);
    }
    return ZS_OK;
}

// One coalesced gather of `params` (nonempty) for module position pos.
// Returns ZS_OK, or ZS_ENOMEM when the block does not fit (nothing changed).
zs_status gather(zs_sched *s, std::vector<int32_t> params, int64_t pos, const void *shards,
                 void *gstream, bool prefetch) {
    sort_ds(s, params);
    std::vector<int64_t> offs;
    int64_t waits = -1;
    if (!alloc(s, params, offs, waits)) return ZS_ENOMEM;
    const int64_t op = s->ops++;
    int64_t elems = 0, block = 0;
    for (size_t i = 0; i < params.size(); ++i) {
        const int32_t p = params[i];
        s->live_flag[p] = 1;
        s->offset[p] = offs[i];
        s->producer[p] = (int32_t)op;
        s->live += numel(s, p);
        elems += numel(s, p);
        block += psize(s, p);
        log_event(s, zs_sched_event{1, (int32_t)pos, (int32_t)op, p, offs[i], waits});
    }
    s->arena_used += block;
    s->st.gathers += 1;
    s->st.params_gathered += (int64_t)params.size();
    s->st.elems_gathered += elems;
    if (prefetch) s->st.elems_prefetched += elems;
    s->st.max_live_elems = std::max(s->st.max_live_elems, s->live);
    s->st.max_arena_elems = std::max(s->st.max_arena_elems, s->arena_used);
    if (!s->arena) return ZS_OK;
    const cudaStream_t gs = (cudaStream_t)gstream;
    zs_status r;
    if (waits >= s->pass_first_rel) {      // older releases precede the pass-start wait
        const cudaError_t e = cudaStreamWaitEvent(gs, s->rel_ev[waits - s->pass_first_rel], 0);
        if (e != cudaSuccess) return cuda_err(e, "zs_sched: cudaStreamWaitEvent");
    }
    std::vector<int64_t> views(params.size());
    r = zs_gather_impl(s->P, (int32_t)params.size(), params.data(), shards, s->arena + offs[0],
                       block, views.data(), gstream, (int)s->cfg.gather_ctas, false,
                       "zs_sched_fetch");
    if (r) return r;
    for (size_t i = 0; i < params.size(); ++i)
        if (views[i] != offs[i] - offs[0])
            return zs_fail(ZS_ESTATE, "zs_sched: gather layout mismatch (internal)");
    if ((r = ensure_event(s->op_ev, op - s->pass_first_op))) return r;
    const cudaError_t e = cudaEventRecord(s->op_ev[op - s->pass_first_op], gs);
    if (e != cudaSuccess) return cuda_err(e, "zs_sched: cudaEventRecord");
    return ZS_OK;
}

bool probe(zs_sched *s, const std::vector<int32_t> &params) {
    const std::vector<Seg> saved = s->free_;
    std::vector<int64_t> offs;
    int64_t w;
    const bool ok = alloc(s, params, offs, w);
    s->free_ = saved;
    return ok;
}

// Walk the trace's parameter uses after the current module within the
// budget; one coalesced gather per module reached, so that a compute waits
// only for the gather of its own parameters.
zs_status prefetch(zs_sched *s, int64_t pos, const void *shards, void *gstream) {
    s->queue_pos = std::max(s->queue_pos, s->queue_start[pos + 1]);
    const int64_t cap = std::min(s->cfg.prefetch_bucket_size, s->cfg.max_live_parameters - s->live);
    std::vector<int32_t> group;
    int64_t gpos = -1, added = 0;
    zs_status r;
    // trace position of queue entry i
    auto position_of = [&](int64_t i) {
        return (int64_t)(std::upper_bound(s->queue_start.begin(), s->queue_start.end() - 1, i) -
                         s->queue_start.begin()) - 1;
    };
    while (s->queue_pos < (int64_t)s->queue.size() && added < cap) {
        const int32_t p = s->queue[s->queue_pos];
        if (!gatherable(s, p) || s->live_flag[p] ||
            std::find(group.begin(), group.end(), p) != group.end()) {
            ++s->queue_pos;
            continue;
        }
        const int64_t k = position_of(s->queue_pos);
        if (!group.empty() && k != gpos) {
            if ((r = gather(s, group, pos, shards, gstream, true))) return r;
            group.clear();
        }
        group.push_back(p);
        if (!probe(s, group)) {
            group.pop_back();
            break;
        }
        gpos = k;
        added += numel(s, p);
        ++s->queue_pos;
    }
    if (group.empty()) return ZS_OK;
    return gather(s, group, pos, shards, gstream, true);
}

bool reused_soon(const zs_sched *s, int32_t p, int64_t pos) {
    int64_t dist = 0;
    for (int64_t k = pos + 1; k < (int64_t)s->trace.size(); ++k) {
        const std::vector<int32_t> &m = s->modules[s->trace[k]];
        if (std::find(m.begin(), m.end(), p) != m.end()) return dist <= s->cfg.max_reuse_distance;
        dist += s->module_numel[s->trace[k]];
    }
    return false;
}

void drop(zs_sched *s, int32_t p, int64_t rel) {
    s->live_flag[p] = 0;
    s->producer[p] = -1;
    s->live -= numel(s, p);
    s->arena_used -= psize(s, p);
    free_seg(s, p, rel);
}

zs_status record_release(zs_sched *s, int64_t rel, void *cstream) {
    if (!s->arena) return ZS_OK;
    zs_status r = ensure_event(s->rel_ev, rel - s->pass_first_rel);
    if (r) return r;
    const cudaError_t e = cudaEventRecord(s->rel_ev[rel - s->pass_first_rel], (cudaStream_t)cstream);
    return e == cudaSuccess ? ZS_OK : cuda_err(e, "zs_sched: cudaEventRecord");
}

// The scheduler's streams are fixed by its first device call; every later
// call must pass the same ones (gstream NULL: not checked, the call has none).
zs_status check_streams(zs_sched *s, void *cstream, void *gstream, bool has_gather,
                        const char *fn) {
    if (!s->arena) return ZS_OK;
    if (!s->streams_set) {
        if (!has_gather) return ZS_OK;      // fixed by the first fetch
        s->cstream = cstream;
        s->gstream = gstream;
        s->streams_set = true;
        return ZS_OK;
    }
    if (cstream != s->cstream || (has_gather && gstream != s->gstream))
        return zs_fail(ZS_EINVAL,
                       "%s: the compute and gather streams must be the same in every call", fn);
    return ZS_OK;
}

void build_queue(zs_sched *s) {
    s->queue.clear();
    s->queue_start.assign(s->trace.size() + 1, 0);
    for (size_t k = 0; k < s->trace.size(); ++k) {
        s->queue_start[k] = (int64_t)s->queue.size();
        for (int32_t p : s->modules[s->trace[k]]) s->queue.push_back(p);
    }
    s->queue_start[s->trace.size()] = (int64_t)s->queue.size();
}

}  // namespace

extern "C" {

zs_status zs_sched_create(const zs_plan *P, int32_t n_modules, const int32_t *module_offsets,
                          const int32_t *module_params, const zs_sched_config *cfg,
                          void *d_arena, zs_sched **out) {
    const char *fn = "zs_sched_create";
    if (!P || !cfg || !out || n_modules < 0 || (n_modules > 0 && (!module_offsets || !module_params)))
        return zs_fail(ZS_EINVAL, "%s: bad arguments", fn);
    *out = nullptr;
    if (cfg->prefetch_bucket_size < 0 || cfg->max_live_parameters < 0 || cfg->max_reuse_distance < 0 ||
        cfg->arena_elems < 0 || cfg->gather_ctas < 0 || cfg->gather_ctas > (1 << 20) ||
        cfg->log_limit < -1)
        return zs_fail(ZS_EINVAL, "%s: negative size in the configuration", fn);
    if (d_arena && (reinterpret_cast<uintptr_t>(d_arena) & 15))
        return zs_fail(ZS_EINVAL, "%s: arena not 16-byte aligned", fn);
    const int32_t np = (int32_t)P->params.size();
    zs_sched *s = new (std::nothrow) zs_sched();
    if (!s) return zs_fail(ZS_ENOMEM, "%s: out of host memory", fn);
    try {
        s->P = P;
        s->cfg = *cfg;
        s->log_cap = cfg->log_limit == 0 ? (int64_t)1 << 20 : cfg->log_limit;
        s->arena = static_cast<uint16_t *>(d_arena);
        s->modules.resize(n_modules);
        s->module_numel.assign(n_modules, 0);
        for (int32_t m = 0; m < n_modules; ++m) {
            const int32_t a = module_offsets[m], b = module_offsets[m + 1];
            if (a < 0 || b < a) {
                delete s;
                return zs_fail(ZS_EINVAL, "%s: module offsets not increasing at %d", fn, m);
            }
            int64_t need = 0;
            for (int32_t i = a; i < b; ++i) {
                const int32_t p = module_params[i];
                if (p < 0 || p >= np) {
                    delete s;
                    return zs_fail(ZS_EINVAL, "%s: module %d uses parameter %d out of range", fn, m, p);
                }
                s->modules[m].push_back(p);
                s->module_numel[m] += P->params[p].numel;
            }
            for (int32_t p : dedup(s->modules[m]))
                if (gatherable(s, p)) need += psize(s, p);
            if (need > cfg->arena_elems) {
                delete s;
                return zs_fail(ZS_EINVAL, "%s: module %d needs %lld arena elements, the arena has %lld",
                               fn, m, (long long)need, (long long)cfg->arena_elems);
            }
        }
        s->live_flag.assign(np, 0);
        s->offset.assign(np, -1);
        s->producer.assign(np, -1);
        if (cfg->arena_elems > 0) s->free_.push_back(Seg{0, cfg->arena_elems, -1});
    } catch (const std::bad_alloc &) {
        delete s;
        return zs_fail(ZS_ENOMEM, "%s: out of host memory", fn);
    }
    *out = s;
    zs_clear_error();
    return ZS_OK;
}

void zs_sched_destroy(zs_sched *s) {
    if (!s) return;
    for (cudaEvent_t e : s->op_ev) cudaEventDestroy(e);
    for (cudaEvent_t e : s->rel_ev) cudaEventDestroy(e);
    if (s->pass_ev) cudaEventDestroy(s->pass_ev);
    delete s;
}

zs_status zs_sched_fetch(zs_sched *s, int32_t m, const void *shards, void *cstream, void *gstream) {
    const char *fn = "zs_sched_fetch";
    if (!s) return zs_fail(ZS_EINVAL, "%s: NULL scheduler", fn);
    if (m < 0 || m >= (int32_t)s->modules.size())
        return zs_fail(ZS_EINVAL, "%s: module %d out of range", fn, m);
    if (s->arena && s->P->S > 0 && (!shards || (reinterpret_cast<uintptr_t>(shards) & 15)))
        return zs_fail(ZS_EINVAL, "%s: param_shards NULL or not 16-byte aligned", fn);
    zs_status r = check_streams(s, cstream, gstream, true, fn);
    if (r) return r;
    if (s->pos == 0) {
        // a new pass: its gathers read shards that the caller may have
        // rewritten (the optimizer step) on the compute stream since the
        // last pass, so the gather stream waits for the compute stream here
        s->pass_first_op = s->ops;
        s->pass_first_rel = s->releases;
        if (s->arena) {
            cudaError_t e = cudaSuccess;
            if (!s->pass_ev) e = cudaEventCreateWithFlags(&s->pass_ev, cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventRecord(s->pass_ev, (cudaStream_t)cstream);
            if (e == cudaSuccess) e = cudaStreamWaitEvent((cudaStream_t)gstream, s->pass_ev, 0);
            if (e != cudaSuccess) return cuda_err(e, "zs_sched_fetch: pass-start wait");
        }
    }
    const int64_t pos = s->pos++;
    if (s->complete && !s->invalid && (pos >= (int64_t)s->trace.size() || s->trace[pos] != m)) {
        s->invalid = true;
        s->st.invalidations += 1;
    }
    if (!s->complete && !s->invalid) s->recording.push_back(m);
    std::vector<int32_t> need;
    for (int32_t p : dedup(s->modules[m]))
        if (gatherable(s, p) && !s->live_flag[p]) need.push_back(p);
    if (!need.empty()) {
        r = gather(s, need, pos, shards, gstream, false);
        if (r == ZS_ENOMEM)
            return zs_fail(ZS_ENOMEM, "%s: module %d does not fit the free arena", fn, m);
        if (r) return r;
        s->st.fetch_misses += (int64_t)need.size();
    }
    std::vector<int32_t> ops;
    for (int32_t p : s->modules[m])
        if (s->live_flag[p] && std::find(ops.begin(), ops.end(), s->producer[p]) == ops.end())
            ops.push_back(s->producer[p]);
    std::sort(ops.begin(), ops.end());
    if (ops.empty()) log_event(s, zs_sched_event{2, (int32_t)pos, -1, -1, 0, 0});
    for (int32_t op : ops) {
        log_event(s, zs_sched_event{2, (int32_t)pos, op, -1, 0, 0});
        if (s->arena) {
            const cudaError_t e =
                cudaStreamWaitEvent((cudaStream_t)cstream, s->op_ev[op - s->pass_first_op], 0);
            if (e != cudaSuccess) return cuda_err(e, "zs_sched_fetch: cudaStreamWaitEvent");
        }
    }
    if (s->complete && !s->invalid) {
        if ((r = prefetch(s, pos, shards, gstream))) return r;
    }
    zs_clear_error();
    return ZS_OK;
}

zs_status zs_sched_release(zs_sched *s, int32_t m, void *cstream) {
    const char *fn = "zs_sched_release";
    if (!s) return zs_fail(ZS_EINVAL, "%s: NULL scheduler", fn);
    if (m < 0 || m >= (int32_t)s->modules.size())
        return zs_fail(ZS_EINVAL, "%s: module %d out of range", fn, m);
    zs_status r = check_streams(s, cstream, nullptr, false, fn);
    if (r) return r;
    const int64_t pos = s->pos - 1;
    const int64_t rel = s->releases++;
    r = record_release(s, rel, cstream);
    if (r) return r;
    bool any = false;
    for (int32_t p : dedup(s->modules[m])) {
        if (!s->live_flag[p]) continue;
        if (s->complete && !s->invalid && reused_soon(s, p, pos)) continue;
        drop(s, p, rel);
        log_event(s, zs_sched_event{3, (int32_t)pos, -1, p, 0, rel});
        any = true;
    }
    if (!any) log_event(s, zs_sched_event{3, (int32_t)pos, -1, -1, 0, rel});
    zs_clear_error();
    return ZS_OK;
}

zs_status zs_sched_end_pass(zs_sched *s, void *cstream) {
    if (!s) return zs_fail(ZS_EINVAL, "zs_sched_end_pass: NULL scheduler");
    zs_status r = check_streams(s, cstream, nullptr, false, "zs_sched_end_pass");
    if (r) return r;
    const int64_t rel = s->releases++;
    r = record_release(s, rel, cstream);
    if (r) return r;
    std::vector<int32_t> out;
    for (int32_t p = 0; p < (int32_t)s->live_flag.size(); ++p)
        if (s->live_flag[p]) out.push_back(p);
    sort_ds(s, out);
    for (int32_t p : out) {
        drop(s, p, rel);
        log_event(s, zs_sched_event{3, (int32_t)s->pos, -1, p, 0, rel});
    }
    if (out.empty()) log_event(s, zs_sched_event{3, (int32_t)s->pos, -1, -1, 0, rel});
    if (s->complete && !s->invalid && s->pos != (int64_t)s->trace.size()) {
        s->invalid = true;
        s->st.invalidations += 1;
    }
    if (!s->complete && !s->invalid) {
        s->trace = s->recording;
        s->complete = true;
        build_queue(s);
    } else if (s->invalid) {
        s->trace.clear();
        s->complete = false;
        s->invalid = false;
        s->queue.clear();
        s->queue_start.clear();
    }
    s->recording.clear();
    s->pos = 0;
    s->queue_pos = 0;
    s->st.passes += 1;
    zs_clear_error();
    return ZS_OK;
}

zs_status zs_sched_param_offset(const zs_sched *s, int32_t p, int64_t *offset) {
    if (!s || !offset) return zs_fail(ZS_EINVAL, "zs_sched_param_offset: NULL argument");
    if (p < 0 || p >= (int32_t)s->live_flag.size())
        return zs_fail(ZS_EINVAL, "zs_sched_param_offset: parameter %d out of range", p);
    if (s->P->params[p].persistent) {
        *offset = -1;
        return ZS_OK;
    }
    if (!s->live_flag[p])
        return zs_fail(ZS_ESTATE, "zs_sched_param_offset: parameter %d is not gathered", p);
    *offset = s->offset[p];
    return ZS_OK;
}

zs_status zs_sched_stats(const zs_sched *s, zs_sched_stats_t *out) {
    if (!s || !out) return zs_fail(ZS_EINVAL, "zs_sched_stats: NULL argument");
    *out = s->st;
    return ZS_OK;
}

zs_status zs_sched_log(const zs_sched *s, zs_sched_event *out, int64_t cap, int64_t *n) {
    if (!s || !n || (cap > 0 && !out)) return zs_fail(ZS_EINVAL, "zs_sched_log: NULL argument");
    *n = (int64_t)s->log.size();
    const int64_t k = std::min<int64_t>(cap, *n);
    for (int64_t i = 0; i < k; ++i) out[i] = s->log[i];
    return ZS_OK;
}

}  // extern "C"
