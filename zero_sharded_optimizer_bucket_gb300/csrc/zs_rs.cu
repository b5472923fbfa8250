// A2 reduce-scatter (with the A3 partial sums) and the A3 norm kernels.
//
// Reduce-scatter ([ZeRO-3 chapter] §6.2, avg-scatter of a full bucket):
// one CTA per tile.  A thread owns 8-element groups of destination slots
// aligned to 16 bytes in shard space; for each rank k in order 0..N-1 it
// loads the matching 8 gradients of rank k's bucket buffer (one 16-byte
// load when source and destination have the same phase, else two aligned
// loads and a lane shift), adds them to 8 float32 sums, then writes
// bf16_rne(sum / N).  The rank loop is sequential per element, so the
// result is bit-exact against the fixed-order definition.  Five CTAs of 256
// threads per SM (registers capped by the launch bounds) keep enough loads
// in flight to stream the N gradient buffers near the HBM read bandwidth.
#include "zs_device.cuh"
#include "zs_launch.h"

namespace zsk {

struct RankPtrs {
    const uint16_t *p[ZS_MAX_RANKS];
};

template <bool FROM_TABLE>
__global__ void __launch_bounds__(THREADS, 5)
rs_kernel(const ZsTile *__restrict__ tiles, int64_t tile0, RankPtrs ptrs,
          const uint16_t *const *__restrict__ table, int N, float fN,
          uint16_t *__restrict__ gs, uint16_t *__restrict__ gP, double *__restrict__ partials) {
    __shared__ const uint16_t *sp[ZS_MAX_RANKS];
    __shared__ double red[WARPS];
    __shared__ int bad;
    const int64_t t = tile0 + blockIdx.x;
    const ZsTile tile = tiles[t];
    if (threadIdx.x == 0) bad = 0;
    __syncthreads();
    for (int k = threadIdx.x; k < N; k += THREADS) {
        const uint16_t *q = FROM_TABLE ? table[(int64_t)tile.bucket * N + k] : ptrs.p[k];
        if (q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15u)) bad = 1;
        sp[k] = q;
    }
    __syncthreads();
    if (bad) {
        // an unusable rank pointer: read nothing, poison the norm so that
        // the update of this step is skipped
        if (threadIdx.x == 0 && partials) partials[t] = __longlong_as_double(0x7FF8000000000000LL);
        return;
    }
    uint16_t *__restrict__ out = tile.flat < 0 ? gP : gs;
    const int64_t D = tile.dst, G0 = D & ~int64_t(7);
    const int64_t ngroups = (D + tile.len - G0 + 7) >> 3;
    const int64_t delta = tile.src - D;
    const int q = (int)((G0 + delta) & 7);
    const int64_t vs = tile.src, ve = tile.src + tile.valid;
    // For N a power of two, 1/N is exact and s * (1/N) is the same single
    // rounding of the exact quotient as s / N, bit for bit; the multiply is
    // far cheaper than an IEEE division.  Other N divide.
    const bool pow2 = (N & (N - 1)) == 0;
    const float invN = 1.0f / fN;
    float sq32 = 0.0f;
    double sq64 = 0.0;
    for (int64_t gi = threadIdx.x; gi < ngroups; gi += THREADS) {
        const int64_t x0 = G0 + 8 * gi;
        const int64_t s0 = x0 + delta;
        const int64_t c0 = s0 >> 3;  // floor
        const int64_t lo = vs - s0, hi = ve - s0;
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        if (q == 0 && lo <= 0 && hi >= 8) {
            const int64_t off = 8 * c0;
#pragma unroll 8
            for (int k = 0; k < N; ++k) {
                const uint4 v = ldg16(sp[k] + off);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], bf2f(lane16(v, i)));
            }
        } else {
            const bool ld0 = (8 * c0 + 8 > vs) && (8 * c0 < ve);
            const bool ld1 = q != 0 && (8 * c0 + 16 > vs) && (8 * c0 + 8 < ve);
#pragma unroll 4
            for (int k = 0; k < N; ++k) {
                const uint4 z = make_uint4(0, 0, 0, 0);
                const uint4 a = ld0 ? ldg16(sp[k] + 8 * c0) : z;
                const uint4 b = ld1 ? ldg16(sp[k] + 8 * c0 + 8) : z;
                const uint4 v = mask8(shift8(a, b, q), lo, hi);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], bf2f(lane16(v, i)));
            }
        }
        uint32_t r[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) r[i] = f2bf(pow2 ? __fmul_rn(acc[i], invN) : __fdiv_rn(acc[i], fN));
        group_sq(r, sq32, sq64);
        if (x0 >= D && x0 + 8 <= D + tile.len) {
            *reinterpret_cast<uint4 *>(out + x0) = pack8(r);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (x0 + i >= D && x0 + i < D + tile.len) out[x0 + i] = (uint16_t)r[i];
        }
    }
    if (partials) {
        const double s = block_sum(__dadd_rn((double)sq32, sq64), red);
        if (threadIdx.x == 0) partials[t] = s;
    }
}

// Recompute the per-tile partial sums from the reduced gradients; the same
// group and thread mapping as rs_kernel, so the same bits.
__global__ void __launch_bounds__(THREADS)
norm_tiles_kernel(const ZsTile *__restrict__ tiles, const uint16_t *__restrict__ gs,
                  const uint16_t *__restrict__ gP, double *__restrict__ partials) {
    __shared__ double red[WARPS];
    const int64_t t = blockIdx.x;
    const ZsTile tile = tiles[t];
    const uint16_t *__restrict__ in = tile.flat < 0 ? gP : gs;
    const int64_t D = tile.dst, G0 = D & ~int64_t(7);
    const int64_t ngroups = (D + tile.len - G0 + 7) >> 3;
    float sq32 = 0.0f;
    double sq64 = 0.0;
    for (int64_t gi = threadIdx.x; gi < ngroups; gi += THREADS) {
        const int64_t x0 = G0 + 8 * gi;
        const uint4 v = mask8(ldg16(in + x0), D - x0, D + tile.len - x0);
        uint32_t r[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) r[i] = lane16(v, i);
        group_sq(r, sq32, sq64);
    }
    const double s = block_sum(__dadd_rn((double)sq32, sq64), red);
    if (threadIdx.x == 0) partials[t] = s;
}

// First level: block c sums partials [c*CH, (c+1)*CH) in a fixed order.
__global__ void __launch_bounds__(THREADS)
norm_level1_kernel(const double *__restrict__ partials, int64_t n, double *__restrict__ level1) {
    __shared__ double red[WARPS];
    const int64_t lo = (int64_t)blockIdx.x * ZS_LEVEL1_CHUNK;
    const int64_t hi = min(n, lo + ZS_LEVEL1_CHUNK);
    double v = 0.0;
    for (int64_t i = lo + threadIdx.x; i < hi; i += THREADS) v = __dadd_rn(v, partials[i]);
    const double s = block_sum(v, red);
    if (threadIdx.x == 0) level1[blockIdx.x] = s;
}

// Finish: total, norm = float(sqrt(total)), clip coefficient, flags.
__global__ void __launch_bounds__(THREADS)
norm_finish_kernel(const double *__restrict__ level1, int64_t n1, float max_norm,
                   float *__restrict__ d_norm, float *__restrict__ d_coef,
                   int32_t *__restrict__ d_flags) {
    __shared__ double red[WARPS];
    double v = 0.0;
    for (int64_t i = threadIdx.x; i < n1; i += THREADS) v = __dadd_rn(v, level1[i]);
    const double s = block_sum(v, red);
    if (threadIdx.x == 0) {
        const float norm = (float)sqrt(s);
        const bool finite = isfinite(norm);
        float coef = 1.0f;
        if (finite && max_norm > 0.0f) {
            const float c = __fdiv_rn(max_norm, __fadd_rn(norm, 1e-6f));
            coef = c < 1.0f ? c : 1.0f;
        }
        *d_norm = norm;
        *d_coef = coef;
        *d_flags = finite ? 0 : ZS_SKIP_NONFINITE;
    }
}

}  // namespace zsk

using namespace zsk;

cudaError_t zsl_reduce_scatter(const ZsTile *d_tiles, int64_t tile0, int64_t ntiles,
                               const void *const *rank_ptrs, int N, uint16_t *gs, uint16_t *gP,
                               double *partials, cudaStream_t s) {
    if (ntiles <= 0) return cudaSuccess;
    RankPtrs p;
    for (int k = 0; k < N; ++k) p.p[k] = static_cast<const uint16_t *>(rank_ptrs[k]);
    rs_kernel<false><<<(unsigned)ntiles, THREADS, 0, s>>>(d_tiles, tile0, p, nullptr, N, (float)N,
                                                          gs, gP, partials);
    return cudaGetLastError();
}

cudaError_t zsl_reduce_scatter_all(const ZsTile *d_tiles, int64_t ntiles,
                                   const void *const *d_table, int N, uint16_t *gs, uint16_t *gP,
                                   double *partials, cudaStream_t s) {
    if (ntiles <= 0) return cudaSuccess;
    RankPtrs p = {};
    rs_kernel<true><<<(unsigned)ntiles, THREADS, 0, s>>>(
        d_tiles, 0, p, reinterpret_cast<const uint16_t *const *>(d_table), N, (float)N, gs, gP,
        partials);
    return cudaGetLastError();
}

cudaError_t zsl_norm(const ZsTile *d_tiles, int64_t ntiles, int64_t n_level1, const uint16_t *gs,
                     const uint16_t *gP, double *scratch, bool recompute, float max_norm,
                     float *d_norm, float *d_coef, int32_t *d_flags, cudaStream_t s) {
    if (recompute && ntiles > 0)
        norm_tiles_kernel<<<(unsigned)ntiles, THREADS, 0, s>>>(d_tiles, gs, gP, scratch);
    norm_level1_kernel<<<(unsigned)n_level1, THREADS, 0, s>>>(scratch, ntiles, scratch + ntiles);
    norm_finish_kernel<<<1, THREADS, 0, s>>>(scratch + ntiles, n_level1, max_norm, d_norm, d_coef,
                                             d_flags);
    return cudaGetLastError();
}
