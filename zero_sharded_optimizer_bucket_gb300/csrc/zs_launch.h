// Host-side launchers of the libzs kernels (called by the C ABI in zs_api.cu
// after argument checks).  Each returns the launch status.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "zs_internal.h"

struct ZsAdamScalars {
    float lr, b1, b2, omb1, omb2, eps, wd, lr_wd, bc1, bc2;
    int adamw;
};

// Loss scale of the norm finish (see zs_loss_scaler); d_scale NULL: S = 1.
struct ZsScaleArgs {
    float *d_scale;
    int32_t *d_good;
    float factor, min_scale;
    int32_t window;
};

// One bucket: launch positions [tile0, tile0 + ntiles); position i works on
// tile d_order[i] (the plan's per-bucket largest-first permutation).
cudaError_t zsl_reduce_scatter(const ZsTile *d_tiles, const int32_t *d_order, int64_t tile0,
                               int64_t ntiles, const void *const *rank_ptrs, int N, int G, int dtype, uint16_t *gs,
                               uint16_t *gP, double *partials, cudaStream_t s);

// Tiles [tile0, tile0 + ntiles) (whole buckets from bucket0 on); rank k's
// buffer of bucket b at d_table[(b - bucket0) * N + k].
cudaError_t zsl_reduce_scatter_all(const ZsTile *d_tiles, int64_t tile0, int64_t ntiles,
                                   int32_t bucket0, const void *const *d_table, int N, int G,
                                   int dtype, uint16_t *gs, uint16_t *gP, double *partials,
                                   cudaStream_t s);

cudaError_t zsl_norm(const ZsTile *d_tiles, int64_t ntiles, int64_t n_level1, int dtype,
                     const uint16_t *gs, const uint16_t *gP, double *scratch, bool recompute,
                     float max_norm, float *d_norm, float *d_coef, int32_t *d_flags,
                     const ZsScaleArgs *scale, cudaStream_t s);

cudaError_t zsl_adam(int N, int dtype, int64_t S, int64_t s_lo, int64_t s_hi, int64_t p_lo, int64_t p_hi,
                     const ZsAdamScalars &c, const float *d_coef, const int32_t *d_flags,
                     const zs_shard_state &st, cudaStream_t s);

cudaError_t zsl_step2(const ZsTile *d_tiles, int64_t ntiles, int dtype, const ZsAdamScalars &c,
                      const float *d_coef, const int32_t *d_flags, const zs_shard_state &st,
                      uint16_t *flat_out, cudaStream_t s);

cudaError_t zsl_partition(const ZsTile *d_tiles, int64_t ntiles, int dtype, const float *W,
                          const zs_shard_state &st, cudaStream_t s);

// One gather launch covers the output range [out_lo, out_hi) of flat_out,
// made of at most ZS_GATHER_MAX parameters laid out back to back.
constexpr int ZS_GATHER_MAX = 128;   // keeps the launch arguments under 4 KB
struct ZsGatherEntry {
    int64_t out_off;    // first element of the parameter in flat_out
    int64_t shard_off;  // S_p
    int64_t ps;         // > 0
};
struct ZsGatherArgs {
    ZsGatherEntry e[ZS_GATHER_MAX];
    int32_t n;
    int32_t N;
    int64_t S;
    int64_t out_lo, out_hi;
};

// max_ctas caps the grid (0: the default, 8 CTAs per SM on either path)
// dependent: bulk-path launches are programmatic dependents of the previous
// kernel of the stream (back-to-back gathers lose the launch gap; the
// waiting CTAs hold their shared memory, so gathers that run beside other
// work are launched plainly)
cudaError_t zsl_gather(const ZsGatherArgs &a, const uint16_t *shards, uint16_t *flat_out,
                       cudaStream_t s, int max_ctas, bool dependent);
// Number of bounded waits of the bulk gather that gave up (synchronous).
cudaError_t zsl_bulk_wait_timeouts(int *count, bool reset);
// One bounded wait on an mbarrier nothing arrives on (gives up after limit_ns).
cudaError_t zsl_wait_timeout_test(int64_t limit_ns, cudaStream_t s);
