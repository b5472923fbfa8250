// C ABI entry points that enqueue device work: argument checks on the host,
// then the launchers.  Nothing here allocates device memory or waits on it.
#include <algorithm>
#include <cmath>
#include <vector>

#include "zs_launch.h"

namespace {

bool al(const void *p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

zs_status cuda_status(cudaError_t e, const char *what) {
    if (e != cudaSuccess)
        return zs_fail(ZS_ECUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
    zs_clear_error();
    return ZS_OK;
}

zs_status need_table(const zs_plan *P, const char *fn) {
    if (!P) return zs_fail(ZS_EINVAL, "%s: NULL plan", fn);
    if (!P->tiles.empty() && !P->d_tiles)
        return zs_fail(ZS_ESTATE, "%s: plan not uploaded (call zs_plan_upload first)", fn);
    return ZS_OK;
}

// Pointers of the spaces a call touches: shard arrays when N*S > 0,
// persistent arrays when Pn > 0.
zs_status check_state(const zs_plan *P, const zs_shard_state *st, bool grads, bool update,
                      const char *fn, bool shards_optional = false) {
    if (!st) return zs_fail(ZS_EINVAL, "%s: NULL state", fn);
    const bool shard = P->S > 0, pers = P->Pn_alloc > 0;
    struct Item { const void *p; bool used; const char *name; };
    const Item items[] = {
        {st->grad_shards, shard && grads, "grad_shards"},
        {st->param_shards, shard && update && !(shards_optional && !st->param_shards),
         "param_shards"},
        {st->master, shard && update, "master"},
        {st->exp_avg, shard && update, "exp_avg"},
        {st->exp_avg_sq, shard && update, "exp_avg_sq"},
        {st->persist_grads, pers && grads, "persist_grads"},
        {st->persist_params, pers && update, "persist_params"},
        {st->p_master, pers && update, "p_master"},
        {st->p_exp_avg, pers && update, "p_exp_avg"},
        {st->p_exp_avg_sq, pers && update, "p_exp_avg_sq"},
    };
    for (const Item &it : items)
        if (it.used && !al(it.p, 16))
            return zs_fail(ZS_EINVAL, "%s: %s is NULL or not 16-byte aligned", fn, it.name);
    return ZS_OK;
}

zs_status adam_scalars(const zs_adam_hparams *hp, int64_t step, ZsAdamScalars *c, const char *fn) {
    if (!hp) return zs_fail(ZS_EINVAL, "%s: NULL hyper-parameters", fn);
    if (step < 1) return zs_fail(ZS_EINVAL, "%s: step %lld < 1", fn, (long long)step);
    if (!(hp->lr >= 0.0f) || !(hp->eps >= 0.0f) || !(hp->weight_decay >= 0.0f) ||
        !(hp->beta1 >= 0.0f && hp->beta1 < 1.0f) || !(hp->beta2 >= 0.0f && hp->beta2 < 1.0f))
        return zs_fail(ZS_EINVAL, "%s: hyper-parameters out of range", fn);
    c->lr = hp->lr;
    c->b1 = hp->beta1;
    c->b2 = hp->beta2;
    c->eps = hp->eps;
    c->wd = hp->weight_decay;
    // 1 - beta, lr * wd and 1 - beta^t in double, rounded once to float
    c->omb1 = (float)(1.0 - (double)hp->beta1);
    c->omb2 = (float)(1.0 - (double)hp->beta2);
    c->lr_wd = (float)((double)hp->lr * (double)hp->weight_decay);
    if (hp->bias_correction) {
        c->bc1 = (float)(1.0 - std::pow((double)hp->beta1, (double)step));
        c->bc2 = (float)(1.0 - std::pow((double)hp->beta2, (double)step));
    } else {
        c->bc1 = c->bc2 = 1.0f;
    }
    c->adamw = hp->adamw ? 1 : 0;
    return ZS_OK;
}

zs_status check_scalars(const float *a, const float *b, const int32_t *f, const char *fn) {
    if (!al(a, 4) || !al(b, 4) || !al(f, 4))
        return zs_fail(ZS_EINVAL, "%s: device scalar pointers must be non-NULL and 4-byte aligned", fn);
    return ZS_OK;
}

zs_status check_scratch(const zs_plan *P, const double *s, const char *fn) {
    if (!al(s, 8)) return zs_fail(ZS_EINVAL, "%s: norm_scratch NULL or not 8-byte aligned", fn);
    (void)P;
    return ZS_OK;
}

}  // namespace

extern "C" {

zs_status zs_plan_upload(zs_plan *P, void *d_table, int64_t bytes, void *stream) {
    if (!P) return zs_fail(ZS_EINVAL, "zs_plan_upload: NULL plan");
    const int64_t ntiles = (int64_t)P->tiles.size();
    const int64_t need = zs_table_bytes(ntiles), tile_bytes = zs_table_tile_bytes(ntiles);
    if (ntiles == 0) {
        P->d_tiles = static_cast<const ZsTile *>(d_table);
        P->d_rs_order = nullptr;
        zs_clear_error();
        return ZS_OK;
    }
    if (!al(d_table, 16)) return zs_fail(ZS_EINVAL, "zs_plan_upload: table NULL or not 16-byte aligned");
    if (bytes < need)
        return zs_fail(ZS_EINVAL, "zs_plan_upload: %lld bytes < %lld needed", (long long)bytes,
                       (long long)need);
    char *d = static_cast<char *>(d_table);
    cudaError_t e = cudaMemcpyAsync(d, P->tiles.data(), (size_t)tile_bytes,
                                    cudaMemcpyHostToDevice, (cudaStream_t)stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(d + tile_bytes, P->rs_order.data(), (size_t)ntiles * 4,
                            cudaMemcpyHostToDevice, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_status(e, "zs_plan_upload: cudaMemcpyAsync");
    P->d_tiles = static_cast<const ZsTile *>(d_table);
    P->d_rs_order = reinterpret_cast<const int32_t *>(d + tile_bytes);
    zs_clear_error();
    return ZS_OK;
}

zs_status zs_partition(const zs_plan *P, const float *W, const zs_shard_state *st, void *stream) {
    const char *fn = "zs_partition";
    zs_status r = need_table(P, fn);
    if (r) return r;
    if ((r = check_state(P, st, false, true, fn))) return r;
    if (P->psi > 0 && !al(W, 4)) return zs_fail(ZS_EINVAL, "%s: full_params NULL or misaligned", fn);
    return cuda_status(zsl_partition(P->d_tiles, (int64_t)P->tiles.size(), P->cfg.dtype, W, *st,
                                     (cudaStream_t)stream), fn);
}

zs_status zs_reduce_scatter(const zs_plan *P, int32_t bucket, const void *const *rank_grads,
                            void *grad_shards, void *persist_grads, double *norm_scratch,
                            void *stream) {
    const char *fn = "zs_reduce_scatter";
    zs_status r = need_table(P, fn);
    if (r) return r;
    const int N = P->cfg.n_ranks;
    if (bucket < 0 || bucket >= (int32_t)P->buckets.size())
        return zs_fail(ZS_EINVAL, "%s: bucket %d out of range [0, %d)", fn, bucket,
                       (int)P->buckets.size());
    if (N > ZS_MAX_RANKS) return zs_fail(ZS_EINVAL, "%s: N = %d > ZS_MAX_RANKS", fn, N);
    if (!rank_grads) return zs_fail(ZS_EINVAL, "%s: NULL rank_grads", fn);
    for (int k = 0; k < N; ++k)
        if (!al(rank_grads[k], 16))
            return zs_fail(ZS_EINVAL, "%s: rank_grads[%d] NULL or not 16-byte aligned", fn, k);
    if (P->S > 0 && !al(grad_shards, 16))
        return zs_fail(ZS_EINVAL, "%s: grad_shards NULL or not 16-byte aligned", fn);
    if (P->Pn_alloc > 0 && !al(persist_grads, 16))
        return zs_fail(ZS_EINVAL, "%s: persist_grads NULL or not 16-byte aligned", fn);
    if (norm_scratch && !al(norm_scratch, 8))
        return zs_fail(ZS_EINVAL, "%s: norm_scratch not 8-byte aligned", fn);
    const ZsBucket &b = P->buckets[bucket];
    return cuda_status(zsl_reduce_scatter(P->d_tiles, P->d_rs_order, b.first_tile, b.n_tiles, rank_grads, N, P->G,
                                          P->cfg.dtype,
                                          static_cast<uint16_t *>(grad_shards),
                                          static_cast<uint16_t *>(persist_grads), norm_scratch,
                                          (cudaStream_t)stream), fn);
}

zs_status zs_grad_norm(const zs_plan *P, const void *grad_shards, const void *persist_grads,
                       double *norm_scratch, int32_t recompute, float max_norm, float *d_norm,
                       float *d_clip_coef, int32_t *d_flags, void *stream) {
    const char *fn = "zs_grad_norm";
    zs_status r = need_table(P, fn);
    if (r) return r;
    if ((r = check_scratch(P, norm_scratch, fn))) return r;
    if ((r = check_scalars(d_norm, d_clip_coef, d_flags, fn))) return r;
    if (recompute) {
        if (P->S > 0 && !al(grad_shards, 16))
            return zs_fail(ZS_EINVAL, "%s: grad_shards NULL or not 16-byte aligned", fn);
        if (P->Pn_alloc > 0 && !al(persist_grads, 16))
            return zs_fail(ZS_EINVAL, "%s: persist_grads NULL or not 16-byte aligned", fn);
    }
    return cuda_status(zsl_norm(P->d_tiles, (int64_t)P->tiles.size(), P->n_level1, P->cfg.dtype,
                                static_cast<const uint16_t *>(grad_shards),
                                static_cast<const uint16_t *>(persist_grads), norm_scratch,
                                recompute != 0, max_norm, d_norm, d_clip_coef, d_flags, nullptr,
                                (cudaStream_t)stream), fn);
}

zs_status zs_adam_step(const zs_plan *P, int32_t sub_group, const zs_adam_hparams *hp,
                       int64_t step, const float *d_clip_coef, const int32_t *d_flags,
                       const zs_shard_state *st, void *stream) {
    const char *fn = "zs_adam_step";
    if (!P) return zs_fail(ZS_EINVAL, "%s: NULL plan", fn);
    if (sub_group < -1 || sub_group >= (int32_t)P->sub_groups.size())
        return zs_fail(ZS_EINVAL, "%s: sub_group %d out of range", fn, sub_group);
    ZsAdamScalars c;
    zs_status r = adam_scalars(hp, step, &c, fn);
    if (r) return r;
    if (!al(d_clip_coef, 4) || !al(d_flags, 4))
        return zs_fail(ZS_EINVAL, "%s: d_clip_coef / d_flags NULL or misaligned", fn);
    if ((r = check_state(P, st, true, true, fn))) return r;
    int64_t s_lo = 0, s_hi = P->S, p_lo = 0, p_hi = P->Pn_alloc;
    if (sub_group >= 0) {
        const ZsSubGroup &g = P->sub_groups[sub_group];
        s_lo = g.s_lo; s_hi = g.s_hi; p_lo = g.p_lo; p_hi = g.p_hi;
    }
    return cuda_status(zsl_adam(P->G, P->cfg.dtype, P->S, s_lo, s_hi, p_lo, p_hi, c, d_clip_coef,
                                d_flags, *st, (cudaStream_t)stream), fn);
}

}  // extern "C"

zs_status zs_gather_impl(const zs_plan *P, int32_t n, const int32_t *params,
                         const void *param_shards, void *flat_out, int64_t flat_capacity,
                         int64_t *view_offsets, void *stream, int max_ctas, bool dependent,
                         const char *fn) {
    zs_status r = need_table(P, fn);
    if (r) return r;
    if (n < 0 || (n > 0 && (!params || !view_offsets)))
        return zs_fail(ZS_EINVAL, "%s: bad parameter list", fn);
    const int32_t np = (int32_t)P->params.size();
    std::vector<char> seen((size_t)np, 0);
    std::vector<int32_t> srt;
    srt.reserve((size_t)n);
    for (int32_t i = 0; i < n; ++i) {
        const int32_t k = params[i];
        if (k < 0 || k >= np) return zs_fail(ZS_EINVAL, "%s: parameter %d out of range", fn, k);
        if (seen[k]) return zs_fail(ZS_EINVAL, "%s: parameter %d listed twice", fn, k);
        seen[k] = 1;
        srt.push_back(k);
    }
    // ds_id order: every rank packs the same order ([ZeRO-3 chapter] §5.2, §7)
    std::sort(srt.begin(), srt.end(),
              [&](int32_t a, int32_t b) { return P->params[a].position < P->params[b].position; });
    const int64_t N = P->G;   // a group's shard owners
    std::vector<int64_t> off((size_t)np, -1);
    int64_t total = 0;
    for (int32_t k : srt) {
        const ZsParam &p = P->params[k];
        if (p.persistent) continue;
        off[k] = total;
        total += N * p.ps;
    }
    if (total > 0) {
        if (!al(flat_out, 2)) return zs_fail(ZS_EINVAL, "%s: flat_out NULL or odd address", fn);
        if (!al(param_shards, 16))
            return zs_fail(ZS_EINVAL, "%s: param_shards NULL or not 16-byte aligned", fn);
    }
    if (flat_capacity < total)
        return zs_fail(ZS_EINVAL, "%s: flat_capacity %lld < %lld needed", fn,
                       (long long)flat_capacity, (long long)total);
    ZsGatherArgs a;
    a.n = 0;
    a.N = (int32_t)N;
    a.S = P->S;
    a.out_lo = a.out_hi = 0;
    auto flush = [&]() -> zs_status {
        if (a.n == 0) return ZS_OK;
        const cudaError_t e = zsl_gather(a, static_cast<const uint16_t *>(param_shards),
                                         static_cast<uint16_t *>(flat_out), (cudaStream_t)stream,
                                         max_ctas, dependent);
        a.n = 0;
        return cuda_status(e, fn);
    };
    for (int32_t k : srt) {
        const ZsParam &p = P->params[k];
        if (p.persistent || p.ps == 0) continue;
        if (a.n == 0) a.out_lo = off[k];
        a.e[a.n].out_off = off[k];
        a.e[a.n].shard_off = p.shard_off;
        a.e[a.n].ps = p.ps;
        a.n += 1;
        a.out_hi = off[k] + N * p.ps;
        if (a.n == ZS_GATHER_MAX && (r = flush())) return r;
    }
    if ((r = flush())) return r;
    for (int32_t i = 0; i < n; ++i) view_offsets[i] = off[params[i]];
    zs_clear_error();
    return ZS_OK;
}

extern "C" {

zs_status zs_device_wait_timeouts(int32_t *count, int32_t reset) {
    if (!count) return zs_fail(ZS_EINVAL, "zs_device_wait_timeouts: NULL count");
    int c = 0;
    const cudaError_t e = zsl_bulk_wait_timeouts(&c, reset != 0);
    if (e != cudaSuccess) return cuda_status(e, "zs_device_wait_timeouts");
    *count = c;
    if (c != 0)
        return zs_fail(ZS_ETIMEOUT, "zs_device_wait_timeouts: %d bounded device wait(s) gave up", c);
    zs_clear_error();
    return ZS_OK;
}

zs_status zs_test_wait_timeout(int64_t limit_ns, void *stream) {
    if (limit_ns <= 0 || limit_ns > 2000000000ll)
        return zs_fail(ZS_EINVAL, "zs_test_wait_timeout: limit_ns %lld not in (0, 2e9]",
                       (long long)limit_ns);
    return cuda_status(zsl_wait_timeout_test(limit_ns, (cudaStream_t)stream), "zs_test_wait_timeout");
}

zs_status zs_all_gather_coalesced(const zs_plan *P, int32_t n, const int32_t *params,
                                  const void *param_shards, void *flat_out,
                                  int64_t flat_capacity, int64_t *view_offsets, void *stream) {
    return zs_gather_impl(P, n, params, param_shards, flat_out, flat_capacity, view_offsets,
                          stream, 0, true, "zs_all_gather_coalesced");
}

zs_status zs_unscale_and_clip(const zs_plan *P, const void *grad_shards, const void *persist_grads,
                              double *norm_scratch, int32_t recompute, float max_norm,
                              const zs_loss_scaler *scaler, float *d_norm, float *d_clip_coef,
                              int32_t *d_flags, void *stream) {
    const char *fn = "zs_unscale_and_clip";
    zs_status r = need_table(P, fn);
    if (r) return r;
    if (!scaler || !al(scaler->d_scale, 4))
        return zs_fail(ZS_EINVAL, "%s: scaler or its d_scale NULL / misaligned", fn);
    if (scaler->reserved != 0) return zs_fail(ZS_EINVAL, "%s: scaler reserved field must be 0", fn);
    if (scaler->scale_window > 0) {
        if (!al(scaler->d_good_steps, 4))
            return zs_fail(ZS_EINVAL, "%s: d_good_steps NULL or misaligned", fn);
        if (!(scaler->scale_factor > 1.0f) || !(scaler->min_scale > 0.0f))
            return zs_fail(ZS_EINVAL, "%s: need scale_factor > 1 and min_scale > 0", fn);
    }
    if ((r = check_scratch(P, norm_scratch, fn))) return r;
    if ((r = check_scalars(d_norm, d_clip_coef, d_flags, fn))) return r;
    if (recompute) {
        if (P->S > 0 && !al(grad_shards, 16))
            return zs_fail(ZS_EINVAL, "%s: grad_shards NULL or not 16-byte aligned", fn);
        if (P->Pn_alloc > 0 && !al(persist_grads, 16))
            return zs_fail(ZS_EINVAL, "%s: persist_grads NULL or not 16-byte aligned", fn);
    }
    ZsScaleArgs sc;
    sc.d_scale = scaler->d_scale;
    sc.d_good = scaler->scale_window > 0 ? scaler->d_good_steps : nullptr;
    sc.factor = scaler->scale_factor;
    sc.min_scale = scaler->min_scale;
    sc.window = scaler->scale_window;
    return cuda_status(zsl_norm(P->d_tiles, (int64_t)P->tiles.size(), P->n_level1, P->cfg.dtype,
                                static_cast<const uint16_t *>(grad_shards),
                                static_cast<const uint16_t *>(persist_grads), norm_scratch,
                                recompute != 0, max_norm, d_norm, d_clip_coef, d_flags, &sc,
                                (cudaStream_t)stream), fn);
}

// zs_reduce_scatter_range / zs_reduce_scatter_all; fn names the caller.
static zs_status rs_range(const zs_plan *P, int32_t first_bucket, int32_t n_buckets,
                          const void *const *d_rank_grads, void *grad_shards, void *persist_grads,
                          double *norm_scratch, bool scratch_required, void *stream,
                          const char *fn) {
    zs_status r = need_table(P, fn);
    if (r) return r;
    const int64_t nb = (int64_t)P->buckets.size();
    if (first_bucket < 0 || n_buckets < 0 || (int64_t)first_bucket + n_buckets > nb)
        return zs_fail(ZS_EINVAL, "%s: buckets [%d, %d + %d) not within the plan's %lld", fn,
                       first_bucket, first_bucket, n_buckets, (long long)nb);
    if (P->cfg.n_ranks > ZS_MAX_RANKS)
        return zs_fail(ZS_EINVAL, "%s: N = %d > ZS_MAX_RANKS", fn, P->cfg.n_ranks);
    if (n_buckets > 0 && !al(d_rank_grads, 8))
        return zs_fail(ZS_EINVAL, "%s: d_rank_grads NULL or misaligned", fn);
    if (P->S > 0 && !al(grad_shards, 16))
        return zs_fail(ZS_EINVAL, "%s: grad_shards NULL or not 16-byte aligned", fn);
    if (P->Pn_alloc > 0 && !al(persist_grads, 16))
        return zs_fail(ZS_EINVAL, "%s: persist_grads NULL or not 16-byte aligned", fn);
    if ((scratch_required || norm_scratch) && (r = check_scratch(P, norm_scratch, fn))) return r;
    if (n_buckets == 0) {
        zs_clear_error();
        return ZS_OK;
    }
    // the tiles of consecutive buckets are consecutive in the table
    const ZsBucket &b0 = P->buckets[first_bucket];
    const ZsBucket &b1 = P->buckets[first_bucket + n_buckets - 1];
    const int64_t tile0 = b0.first_tile, ntiles = b1.first_tile + b1.n_tiles - b0.first_tile;
    return cuda_status(zsl_reduce_scatter_all(P->d_tiles, tile0, ntiles, first_bucket,
                                              d_rank_grads, P->cfg.n_ranks, P->G, P->cfg.dtype,
                                              static_cast<uint16_t *>(grad_shards),
                                              static_cast<uint16_t *>(persist_grads),
                                              norm_scratch, (cudaStream_t)stream), fn);
}

zs_status zs_reduce_scatter_range(const zs_plan *P, int32_t first_bucket, int32_t n_buckets,
                                  const void *const *d_rank_grads, void *grad_shards,
                                  void *persist_grads, double *norm_scratch, void *stream) {
    return rs_range(P, first_bucket, n_buckets, d_rank_grads, grad_shards, persist_grads,
                    norm_scratch, false, stream, "zs_reduce_scatter_range");
}

zs_status zs_reduce_scatter_all(const zs_plan *P, const void *const *d_rank_grads,
                                void *grad_shards, void *persist_grads, double *norm_scratch,
                                void *stream) {
    const char *fn = "zs_reduce_scatter_all";
    if (!P) return zs_fail(ZS_EINVAL, "%s: NULL plan", fn);
    return rs_range(P, 0, (int32_t)P->buckets.size(), d_rank_grads, grad_shards, persist_grads,
                    norm_scratch, true, stream, fn);
}

zs_status zs_adam_gather(const zs_plan *P, const zs_adam_hparams *hp, int64_t step,
                         const float *d_clip_coef, const int32_t *d_flags,
                         const zs_shard_state *st, void *flat_out, void *stream) {
    const char *fn = "zs_adam_gather";
    zs_status r = need_table(P, fn);
    if (r) return r;
    ZsAdamScalars c;
    if ((r = adam_scalars(hp, step, &c, fn))) return r;
    if ((r = check_state(P, st, true, true, fn, true))) return r;
    if (!al(d_clip_coef, 4) || !al(d_flags, 4))
        return zs_fail(ZS_EINVAL, "%s: d_clip_coef / d_flags NULL or misaligned", fn);
    if (P->flat_elems > 0 && !al(flat_out, 2))
        return zs_fail(ZS_EINVAL, "%s: flat_out NULL or odd address", fn);
    return cuda_status(zsl_step2(P->d_tiles, (int64_t)P->tiles.size(), P->cfg.dtype, c, d_clip_coef, d_flags,
                                 *st, static_cast<uint16_t *>(flat_out), (cudaStream_t)stream), fn);
}

zs_status zs_shard_step(const zs_plan *P, const void *const *d_rank_grads,
                        const zs_shard_state *st, double *norm_scratch,
                        const zs_adam_hparams *hp, int64_t step, float max_norm, float *d_norm,
                        float *d_clip_coef, int32_t *d_flags, void *flat_out, void *stream) {
    const char *fn = "zs_shard_step";
    zs_status r = need_table(P, fn);
    if (r) return r;
    ZsAdamScalars c;
    if ((r = adam_scalars(hp, step, &c, fn))) return r;
    if ((r = check_state(P, st, true, true, fn, true))) return r;
    if ((r = check_scratch(P, norm_scratch, fn))) return r;
    if ((r = check_scalars(d_norm, d_clip_coef, d_flags, fn))) return r;
    if (P->flat_elems > 0 && !al(flat_out, 2))
        return zs_fail(ZS_EINVAL, "%s: flat_out NULL or odd address", fn);
    if ((r = zs_reduce_scatter_all(P, d_rank_grads, st->grad_shards, st->persist_grads,
                                   norm_scratch, stream)))
        return r;
    if ((r = zs_grad_norm(P, st->grad_shards, st->persist_grads, norm_scratch, 0, max_norm, d_norm,
                          d_clip_coef, d_flags, stream)))
        return r;
    return zs_adam_gather(P, hp, step, d_clip_coef, d_flags, st, flat_out, stream);
}

zs_status zs_shard_step_scaled(const zs_plan *P, const void *const *d_rank_grads,
                               const zs_shard_state *st, double *norm_scratch,
                               const zs_adam_hparams *hp, int64_t step, float max_norm,
                               const zs_loss_scaler *scaler, float *d_norm, float *d_clip_coef,
                               int32_t *d_flags, void *flat_out, void *stream) {
    const char *fn = "zs_shard_step_scaled";
    zs_status r = need_table(P, fn);
    if (r) return r;
    ZsAdamScalars c;
    if ((r = adam_scalars(hp, step, &c, fn))) return r;
    if ((r = check_state(P, st, true, true, fn, true))) return r;
    if ((r = check_scratch(P, norm_scratch, fn))) return r;
    if ((r = check_scalars(d_norm, d_clip_coef, d_flags, fn))) return r;
    if (!scaler || !al(scaler->d_scale, 4) || scaler->reserved != 0 ||
        (scaler->scale_window > 0 && !al(scaler->d_good_steps, 4)))
        return zs_fail(ZS_EINVAL, "%s: bad loss scaler", fn);
    if (P->flat_elems > 0 && !al(flat_out, 2))
        return zs_fail(ZS_EINVAL, "%s: flat_out NULL or odd address", fn);
    if ((r = zs_reduce_scatter_all(P, d_rank_grads, st->grad_shards, st->persist_grads,
                                   norm_scratch, stream)))
        return r;
    if ((r = zs_unscale_and_clip(P, st->grad_shards, st->persist_grads, norm_scratch, 0, max_norm,
                                 scaler, d_norm, d_clip_coef, d_flags, stream)))
        return r;
    return zs_adam_gather(P, hp, step, d_clip_coef, d_flags, st, flat_out, stream);
}

}  // extern "C"
