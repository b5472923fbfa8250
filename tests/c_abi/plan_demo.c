/*
 * A plain C99 client of libzs (include/zs.h only: no C++, no CUDA headers,
 * no Python).  It builds a partition plan, checks its layout against the
 * definitions (ps = ceil(numel / N), shard offsets rounded up to 8,
 * persistence below the threshold), checks that bad arguments come back as
 * ZS_EINVAL with a message, and drives a plan-only gather scheduler through
 * a recording pass and a prefetching pass.  Host calls only: it needs no GPU.
 * Exit status 0 when every check holds.
 */
#include <stdint.h>
#include <stdio.h>
#include <string.h>

#include "zs.h"

static int failures = 0;

#define CHECK(cond)                                                         \
    do {                                                                    \
        if (!(cond)) {                                                      \
            fprintf(stderr, "check failed at line %d: %s\n", __LINE__, #cond); \
            ++failures;                                                     \
        }                                                                   \
    } while (0)

static int64_t align8(int64_t x) { return (x + 7) / 8 * 8; }

int main(void) {
    const int32_t N = 4;
    const int64_t numel[] = {4096, 64, 16384, 1000, 7, 30000};
    const int32_t n = (int32_t)(sizeof(numel) / sizeof(numel[0]));
    zs_config cfg;
    zs_default_config(&cfg, N);
    cfg.param_persistence_threshold = 100;   /* 64 and 7 stay whole */
    cfg.reduce_bucket_size = 20000;
    zs_plan *plan = NULL;
    CHECK(zs_build_partition(&cfg, n, numel, NULL, &plan) == ZS_OK);
    if (!plan) return 1;
    printf("libzs %s\n", zs_version());

    zs_plan_info_t info;
    CHECK(zs_plan_info(plan, &info) == ZS_OK);
    CHECK(info.n_ranks == N && info.n_params == n);
    int64_t S = 0, Pn = 0, psi = 0, flat = 0;
    for (int32_t p = 0; p < n; ++p) {
        zs_param_info_t pi;
        CHECK(zs_param_info(plan, p, &pi) == ZS_OK);
        psi += numel[p];
        if (numel[p] < cfg.param_persistence_threshold) {
            CHECK(pi.persistent == 1 && pi.partition_size == 0 && pi.shard_offset == -1);
            CHECK(pi.persist_offset == Pn);
            Pn += align8(numel[p]);
        } else {
            const int64_t ps = (numel[p] + N - 1) / N;
            CHECK(pi.persistent == 0 && pi.partition_size == ps);
            CHECK(pi.padding == N * ps - numel[p]);
            CHECK(pi.shard_offset == S && pi.flat_offset == flat);
            S += align8(ps);
            flat += N * ps;
        }
    }
    CHECK(info.shard_elems == S && info.persist_elems == Pn);
    CHECK(info.psi == psi && info.flat_elems == flat);

    /* bad arguments: ZS_EINVAL, a message, nothing changed */
    zs_plan *bad = NULL;
    CHECK(zs_build_partition(&cfg, -1, numel, NULL, &bad) == ZS_EINVAL && bad == NULL);
    CHECK(strlen(zs_last_error()) > 0);
    zs_param_info_t pi;
    CHECK(zs_param_info(plan, n, &pi) == ZS_EINVAL);
    zs_config cfg0;
    zs_default_config(&cfg0, 0);
    CHECK(zs_build_partition(&cfg0, n, numel, NULL, &bad) == ZS_EINVAL);

    /* a plan-only scheduler: modules [0], [2, 3], [5], [0, 1] */
    const int32_t offs[] = {0, 1, 3, 4, 6};
    const int32_t mods[] = {0, 2, 3, 5, 0, 1};
    zs_sched_config sc;
    memset(&sc, 0, sizeof(sc));
    sc.prefetch_bucket_size = 50000;
    sc.max_live_parameters = 1000000;
    sc.max_reuse_distance = 0;
    sc.arena_elems = 200000;
    zs_sched *sched = NULL;
    CHECK(zs_sched_create(plan, 4, offs, mods, &sc, NULL, &sched) == ZS_OK);
    if (sched) {
        for (int pass = 0; pass < 2; ++pass) {
            for (int32_t m = 0; m < 4; ++m) {
                CHECK(zs_sched_fetch(sched, m, NULL, NULL, NULL) == ZS_OK);
                CHECK(zs_sched_release(sched, m, NULL) == ZS_OK);
            }
            CHECK(zs_sched_end_pass(sched, NULL) == ZS_OK);
        }
        zs_sched_stats_t st;
        CHECK(zs_sched_stats(sched, &st) == ZS_OK);
        CHECK(st.passes == 2 && st.invalidations == 0);
        CHECK(st.elems_prefetched > 0);        /* the second pass prefetches */
        int64_t nlog = 0;
        CHECK(zs_sched_log(sched, NULL, 0, &nlog) == ZS_OK && nlog > 0);
        CHECK(zs_sched_fetch(sched, 4, NULL, NULL, NULL) == ZS_EINVAL);
        zs_sched_destroy(sched);
    }
    zs_free_plan(plan);
    if (failures) {
        fprintf(stderr, "%d check(s) failed\n", failures);
        return 1;
    }
    printf("ok\n");
    return 0;
}
