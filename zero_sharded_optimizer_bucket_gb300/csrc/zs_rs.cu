// A2 reduce-scatter (with the A3 partial sums) and the A3 norm kernels.
//
// Reduce-scatter ([ZeRO-3 chapter] §6.2, avg-scatter of a full bucket):
// one CTA per tile, a bucket's tiles launched largest first.  A thread owns 8-element chunks aligned to 16 bytes in
// the rank buffers; for each rank k in order 0..N-1 it loads the chunk of
// rank k's bucket buffer with one 16-byte load, adds the 8 values to 8
// float32 sums, then writes bf16_rne(sum / N) to the owners' shard slots
// (one 16-byte store; when shard and bucket have different phases the
// results are realigned once across neighbouring lanes).  The rank loop is sequential per element, so the
// result is bit-exact against the fixed-order definition.  Five CTAs of 256
// threads per SM (registers capped by the launch bounds) keep enough loads
// in flight to stream the N gradient buffers near the HBM read bandwidth.
#include <algorithm>
#include <atomic>

#include "zs_device.cuh"
#include "zs_launch.h"

namespace zsk {

struct RankPtrs {
    const uint16_t *p[ZS_MAX_RANKS];
};

constexpr int RS_CTAS_PER_SM = 5;

// FROM_TABLE: one launch over whole buckets (the fused step, a range of
// buckets), rank pointers from a device table, launch position i on tile i.
// Otherwise one bucket: rank pointers in the arguments, launch position i
// on tile order[i] (the bucket's tiles largest first, so that the launch
// does not end on a large tile that started late; in a launch over many
// buckets the tail comes once and the plain order, which mixes large and
// small tiles, keeps the CTA launch rate from mattering), and with
// prefetch != 0 the first pass fetched into L2 before the dependent wait.
template <bool FROM_TABLE, class T, bool GROUPED>
__global__ void __launch_bounds__(THREADS, RS_CTAS_PER_SM)
rs_kernel(const ZsTile *__restrict__ tiles, const int32_t *__restrict__ order, int64_t tile0,
          RankPtrs ptrs, int prefetch,
          const uint16_t *const *__restrict__ table, int32_t bucket0, int N, int G, float fN,
          uint16_t *__restrict__ gs, uint16_t *__restrict__ gP, double *__restrict__ partials) {
    __shared__ const uint16_t *sp[ZS_MAX_RANKS];
    __shared__ SqRed red;
    __shared__ int badw[WARPS];
    // the tile's results in destination order (the window of the tile norm)
    __shared__ __align__(16) uint16_t win[NORM_WIN_ELEMS];
    // the plan's tables (written by copies only, never by a kernel, so they
    // may be read before the wait below): this launch position's tile
    const int64_t t = FROM_TABLE ? tile0 + blockIdx.x : (int64_t)order[tile0 + blockIdx.x];
    const ZsTile tile = tiles[t];
    if (!FROM_TABLE && prefetch && tile.valid > 0 && threadIdx.x < N) {
        // A per-bucket launch is a programmatic dependent whose CTAs can be
        // placed while the previous kernel drains.  Meanwhile each of them
        // has the chunks that its first pass of the loop below reads (the
        // 256 chunks from the line-aligned first chunk, clipped to the
        // tile) fetched into L2, one bulk prefetch per rank.  A prefetch
        // changes no value any load can see: the L2 is the GPU's point of
        // coherence, and the loads still come after the wait.  Fetching
        // the whole tile instead measured slower: the extra requests
        // compete with the loads of the CTAs that start after the wait.
        // The host asks for it only when the bucket's CTAs fit in one wave
        // (with more waves, most CTAs start after the wait, and it measured
        // slower there too).
        const uint16_t *q = ptrs.p[threadIdx.x];
        if (q != nullptr && !(reinterpret_cast<uintptr_t>(q) & 15u)) {
            const int64_t lo = tile.src & ~int64_t(7);
            const int64_t first = ((tile.src >> 3) & ~int64_t(7)) * 8;
            const int64_t hi =
                min((tile.src + tile.valid + 7) & ~int64_t(7), first + 8 * int64_t(THREADS));
            asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;"
                         :
                         : "l"(__cvta_generic_to_global(q + lo)), "r"((uint32_t)(2 * (hi - lo)))
                         : "memory");
        }
    }
    // Wait until the previous kernel of the stream has finished and its
    // writes are visible (a no-op in an ordinary launch), then let the next
    // dependent launch start placing its CTAs, which wait the same way.
    asm volatile("griddepcontrol.wait;" : : : "memory");
    asm volatile("griddepcontrol.launch_dependents;" : : : "memory");
    // stage the rank pointers; one barrier, with a per-warp vote on their use
    int my_bad = 0;
    for (int k = threadIdx.x; k < N; k += THREADS) {
        const uint16_t *q =
            FROM_TABLE ? table[(int64_t)(tile.bucket - bucket0) * N + k] : ptrs.p[k];
        my_bad |= (q == nullptr || (reinterpret_cast<uintptr_t>(q) & 15u)) ? 1 : 0;
        sp[k] = q;
    }
    my_bad = __any_sync(0xFFFFFFFFu, my_bad);
    if ((threadIdx.x & 31) == 0) badw[threadIdx.x >> 5] = my_bad;
    __syncthreads();
    int bad = 0;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) bad |= badw[w];
    if (bad) {
        // an unusable rank pointer: read nothing, poison the norm so that
        // the update of this step is skipped
        if (threadIdx.x == 0 && partials) partials[t] = __longlong_as_double(0x7FF8000000000000LL);
        return;
    }
    uint16_t *__restrict__ out = tile.flat < 0 ? gP : gs;
    const int64_t D = tile.dst, V = tile.valid;
    const int64_t delta = tile.src - D;
    const int64_t vs = tile.src, ve = tile.src + V;
    // Work goes by 8-element chunks aligned in the SOURCE (the rank buffers):
    // one plain 16-byte load per rank and chunk.  The 8 results of a chunk
    // land at destination offset a = (-delta) mod 8 within an aligned group;
    // when a != 0 they are realigned once, after the rank loop: a lane's
    // last a results and the next lane's first 8-a results form one aligned
    // destination group (warp shuffle), stored as one 16-byte vector.
    const int a = (int)((-delta) & 7);
    const int64_t c_first = vs >> 3;
    const int64_t nchunks = V > 0 ? ((ve - 1) >> 3) - c_first + 1 : 0;
    const int lane = threadIdx.x & 31;
    // For N a power of two, 1/N is exact and s * (1/N) is the same single
    // rounding of the exact quotient as s / N, bit for bit; the multiply is
    // far cheaper than an IEEE division.  Other N divide.
    const bool pow2 = (N & (N - 1)) == 0;
    const float invN = 1.0f / fN;
    // the norm partial is formed from a shared-memory copy of the results
    const bool keep = partials != nullptr;
    const int64_t w0 = D & ~int64_t(7);
    // Chunks are numbered from c0, the tile's first chunk rounded down to a
    // multiple of 8: a warp's 32 chunks then start on a 128-byte boundary of
    // every rank buffer whose start is 128-byte aligned, so a warp's load of
    // one rank touches exactly four lines instead of five.  Lanes before the
    // tile's first chunk only take part in the shuffles.
    const int64_t c0 = c_first & ~int64_t(7);
    const int64_t nspan = nchunks > 0 ? c_first - c0 + nchunks : 0;
    // uniform trip count: every lane takes part in the shuffles
    for (int64_t base = 0; base < nspan; base += THREADS) {
        const int64_t gi = base + threadIdx.x;
        const int64_t c = c0 + gi;
        const bool act = c >= c_first && gi < nspan;
        const int64_t lo = vs - 8 * c, hi = ve - 8 * c;  // valid lanes [lo, hi)
        float acc[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
        if (act) {
            const uint16_t *const *__restrict__ p = sp;
            if (!GROUPED) {
                if (lo <= 0 && hi >= 8) {
#pragma unroll 8
                    for (int k = 0; k < N; ++k) {
                        const uint4 v = ldg16(p[k] + 8 * c);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], T::to_f32(lane16(v, i)));
                    }
                } else {
#pragma unroll 4
                    for (int k = 0; k < N; ++k) {
                        const uint4 v = mask8(ldg16(p[k] + 8 * c), lo, hi);
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], T::to_f32(lane16(v, i)));
                    }
                }
            } else if (lo <= 0 && hi >= 8 && (G & 3) == 0) {
                // HSDP, a full chunk and G a multiple of 4: each replica
                // group's G ranks in rank order (loads in batches of 4),
                // then the group sums in group order
                for (int q0 = 0; q0 < N; q0 += G) {
                    float in[8];
#pragma unroll
                    for (int i = 0; i < 8; ++i) in[i] = 0.0f;
                    for (int k0 = q0; k0 < q0 + G; k0 += 4) {
                        uint4 v[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) v[u] = ldg16(p[k0 + u] + 8 * c);
#pragma unroll
                        for (int u = 0; u < 4; ++u)
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                in[i] = __fadd_rn(in[i], T::to_f32(lane16(v[u], i)));
                    }
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], in[i]);
                }
            } else if (lo <= 0 && hi >= 8 && (N & 3) == 0) {
                // HSDP, a full chunk, other G with N a multiple of 4: loads
                // in batches of 4 ranks across group boundaries, no per-load
                // conditions; the group boundary is a warp-uniform counter
                float in[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) in[i] = 0.0f;
                int cnt = 0;
                for (int k0 = 0; k0 < N; k0 += 4) {
                    uint4 v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) v[u] = ldg16(p[k0 + u] + 8 * c);
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
#pragma unroll
                        for (int i = 0; i < 8; ++i)
                            in[i] = __fadd_rn(in[i], T::to_f32(lane16(v[u], i)));
                        if (++cnt == G) {
#pragma unroll
                            for (int i = 0; i < 8; ++i) {
                                acc[i] = __fadd_rn(acc[i], in[i]);
                                in[i] = 0.0f;
                            }
                            cnt = 0;
                        }
                    }
                }
            } else {
                // HSDP: each replica group's G ranks in rank order, then the
                // group sums in group order.  Loads go in batches of 4 ranks
                // whatever G is, so that short groups keep loads in flight;
                // the group boundary is a warp-uniform counter.
                const bool full = lo <= 0 && hi >= 8;
                float in[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) in[i] = 0.0f;
                int cnt = 0;
                for (int k0 = 0; k0 < N; k0 += 4) {
                    uint4 v[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        v[u] = make_uint4(0, 0, 0, 0);
                        if (k0 + u < N) {
                            v[u] = ldg16(p[k0 + u] + 8 * c);
                            if (!full) v[u] = mask8(v[u], lo, hi);
                        }
                    }
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        if (k0 + u < N) {
#pragma unroll
                            for (int i = 0; i < 8; ++i)
                                in[i] = __fadd_rn(in[i], T::to_f32(lane16(v[u], i)));
                            if (++cnt == G) {
#pragma unroll
                                for (int i = 0; i < 8; ++i) {
                                    acc[i] = __fadd_rn(acc[i], in[i]);
                                    in[i] = 0.0f;
                                }
                                cnt = 0;
                            }
                        }
                    }
                }
            }
        }
        uint32_t r[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
            r[i] = act ? T::from_f32(pow2 ? __fmul_rn(acc[i], invN) : __fdiv_rn(acc[i], fN)) : 0u;
        const int64_t y0 = 8 * c - delta;  // destination of lane 0 of the chunk
        if (a == 0) {
            if (act) {
                if (lo <= 0 && hi >= 8) {
                    *reinterpret_cast<uint4 *>(out + y0) = pack8(r);
                    if (keep) *reinterpret_cast<uint4 *>(win + (y0 - w0)) = pack8(r);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (i >= lo && i < hi) {
                            out[y0 + i] = (uint16_t)r[i];
                            if (keep) win[y0 + i - w0] = (uint16_t)r[i];
                        }
                }
            }
        } else {
            const uint4 w = pack8(r);
            uint4 wn;
            wn.x = __shfl_down_sync(0xFFFFFFFFu, w.x, 1);
            wn.y = __shfl_down_sync(0xFFFFFFFFu, w.y, 1);
            wn.z = __shfl_down_sync(0xFFFFFFFFu, w.z, 1);
            wn.w = __shfl_down_sync(0xFFFFFFFFu, w.w, 1);
            const bool next_act = __shfl_down_sync(0xFFFFFFFFu, (int)act, 1) != 0 && lane < 31;
            // my lanes [8-a, 8) and the next chunk's lanes [0, 8-a) all valid
            const bool vec = act && next_act && lo <= 8 - a && hi >= 16 - a;
            if (vec) {
                const uint4 sv = shift8(w, wn, 8 - a);
                *reinterpret_cast<uint4 *>(out + y0 + 8 - a) = sv;
                if (keep) *reinterpret_cast<uint4 *>(win + (y0 + 8 - a - w0)) = sv;
            }
            const bool prev_vec = __shfl_up_sync(0xFFFFFFFFu, (int)vec, 1) != 0 && lane > 0;
            if (act) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const bool head = i < 8 - a;  // stored by the previous lane's vector?
                    const bool done = head ? prev_vec : vec;
                    if (!done && i >= lo && i < hi) {
                        out[y0 + i] = (uint16_t)r[i];
                        if (keep) win[y0 + i - w0] = (uint16_t)r[i];
                    }
                }
            }
        }
    }
    // padding of the tile (beyond the valid prefix): zeros
    const int64_t p0 = D + V, p1 = D + tile.len;
    for (int64_t g = (p0 >> 3) + threadIdx.x; g <= ((p1 - 1) >> 3) && p1 > p0; g += THREADS) {
        const int64_t x0 = 8 * g;
        if (x0 >= p0 && x0 + 8 <= p1) {
            *reinterpret_cast<uint4 *>(out + x0) = make_uint4(0, 0, 0, 0);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (x0 + i >= p0 && x0 + i < p1) out[x0 + i] = 0;
        }
    }
    if (keep) {
        __syncthreads();   // the window is complete
        const int64_t ng = V > 0 ? ((D + V + 7) >> 3) - (D >> 3) : 0;
        const double s = tile_sumsq_cta<T>(win, ng, D - w0, D + V - w0, red);
        if (threadIdx.x == 0) partials[t] = s;
    }
}

// Recompute the per-tile partial sums from the reduced gradients: one warp
// per tile, persistent (warp w of the grid takes tiles w, w + warps, ...).
// Lane c plays the virtual threads c, c+32, ..., c+224 of the tile norm in
// that order, reading their groups of the tile's window straight from
// global memory (16-byte loads, coalesced across the lanes), and adds their
// pairs in column order; the butterfly across the lanes finishes the tile.
// On aligned tiles the groups of the next virtual thread are loaded before
// the current one is summed.  The same function of the stored values as the reduce-scatter's
// partials, so the same bits, with no shared memory and no block barrier.
constexpr int NORM_CTAS_PER_SM = 4;

template <class T>
__global__ void __launch_bounds__(THREADS, NORM_CTAS_PER_SM)
norm_tiles_kernel(const ZsTile *__restrict__ tiles, int64_t ntiles, const uint16_t *__restrict__ gs,
                  const uint16_t *__restrict__ gP, double *__restrict__ partials) {
    const int lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * WARPS;
    for (int64_t t = (int64_t)blockIdx.x * WARPS + (threadIdx.x >> 5); t < ntiles; t += nw) {
        const ZsTile tile = tiles[t];
        const int64_t D = tile.dst, V = tile.valid;
        const int64_t w0 = D & ~int64_t(7);
        const uint16_t *__restrict__ win = (tile.flat < 0 ? gP : gs) + w0;
        const int64_t ng = V > 0 ? ((D + V + 7) >> 3) - (D >> 3) : 0;
        const int64_t lo = D - w0, hi = D + V - w0;
        float ch = 0.0f, cl = 0.0f;
        bool ok = true;
        uint4 w[NORM_MAXG];
        if (((D | V) & 7) == 0 && ng <= 4 * NORM_VT) {
            // aligned tile (every Llama-shaped tile): the window is the values,
            // at most 4 groups per virtual thread, no masking; the groups of
            // the next virtual thread are in flight while one is summed
            uint4 q[2][4];
            int nq[2];
            auto load = [&](int m, uint4 (&o)[4]) {
                int c = 0;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const int64_t g = 32 * m + lane + (int64_t)NORM_VT * j;
                    o[j] = make_uint4(0, 0, 0, 0);
                    if (g < ng) {
                        o[j] = *reinterpret_cast<const uint4 *>(win + 8 * g);
                        c = j + 1;
                    }
                }
                return c;
            };
            nq[0] = load(0, q[0]);
#pragma unroll
            for (int m = 0; m < NORM_VT / 32; ++m) {
                if (m + 1 < NORM_VT / 32) nq[(m + 1) & 1] = load(m + 1, q[(m + 1) & 1]);
                const VtPair p = vt_sumsq<T>(q[m & 1], nq[m & 1]);
                ok = ok && p.ok;
                if (m == 0) {
                    ch = p.hi;
                    cl = p.lo;
                } else {
                    add22(ch, cl, p.hi, p.lo);
                }
            }
        } else {
#pragma unroll 1
            for (int m = 0; m < NORM_VT / 32; ++m) {
                const int n = vt_groups(win, 32 * m + lane, ng, lo, hi, w);
                const VtPair p = vt_sumsq<T>(w, n);
                ok = ok && p.ok;
                if (m == 0) {
                    ch = p.hi;
                    cl = p.lo;
                } else {
                    add22(ch, cl, p.hi, p.lo);
                }
            }
        }
        double s;
        if (__all_sync(0xFFFFFFFFu, ok)) {
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float h2 = __shfl_xor_sync(0xFFFFFFFFu, ch, off);
                const float l2 = __shfl_xor_sync(0xFFFFFFFFu, cl, off);
                add22(ch, cl, h2, l2);
            }
            s = __dadd_rn((double)ch, (double)cl);
        } else {
            // float64 for the whole tile, the same groups and tree
            double c = 0.0;
#pragma unroll 1
            for (int m = 0; m < NORM_VT / 32; ++m) {
                const int k = vt_groups(win, 32 * m + lane, ng, lo, hi, w);
                const double f = vt_sumsq_f64<T>(w, k);
                c = m == 0 ? f : __dadd_rn(c, f);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) c = __dadd_rn(c, __shfl_xor_sync(0xFFFFFFFFu, c, off));
            s = c;
        }
        if (lane == 0) partials[t] = s;
    }
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

// Finish: total, norm = float(sqrt(total)) / S, clip coefficient / S,
// flags; then the loss-scale update when a scaler is given.  S = 1 without
// one, which leaves every result bit-identical to the unscaled formula.
__global__ void __launch_bounds__(THREADS)
norm_finish_kernel(const double *__restrict__ level1, int64_t n1, float max_norm,
                   float *__restrict__ d_norm, float *__restrict__ d_coef,
                   int32_t *__restrict__ d_flags, ZsScaleArgs sc) {
    __shared__ double red[WARPS];
    double v = 0.0;
    for (int64_t i = threadIdx.x; i < n1; i += THREADS) v = __dadd_rn(v, level1[i]);
    const double s = block_sum(v, red);
    if (threadIdx.x == 0) {
        const float S = sc.d_scale ? *sc.d_scale : 1.0f;
        const float norm = __fdiv_rn((float)sqrt(s), S);
        const bool finite = isfinite(norm);
        float coef = 1.0f;
        if (finite) {
            float clip = 1.0f;
            if (max_norm > 0.0f) {
                const float c = __fdiv_rn(max_norm, __fadd_rn(norm, 1e-6f));
                clip = c < 1.0f ? c : 1.0f;
            }
            coef = __fdiv_rn(clip, S);
        }
        *d_norm = norm;
        *d_coef = coef;
        *d_flags = finite ? 0 : ZS_SKIP_NONFINITE;
        if (sc.d_scale && sc.window > 0) {
            if (!finite) {
                const float d = __fdiv_rn(S, sc.factor);
                *sc.d_scale = d > sc.min_scale ? d : sc.min_scale;
                *sc.d_good = 0;
            } else {
                const int32_t g = *sc.d_good + 1;
                if (g >= sc.window) {
                    *sc.d_scale = __fmul_rn(S, sc.factor);
                    *sc.d_good = 0;
                } else {
                    *sc.d_good = g;
                }
            }
        }
    }
}

}  // namespace zsk

using namespace zsk;

// SM count of the current device, read once per device (atomic: host
// threads may launch at once).
static cudaError_t sm_count(int *out) {
    static std::atomic<int> sms_of[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int sms = sms_of[dev].load(std::memory_order_relaxed);
    if (sms <= 0) {
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        if (sms <= 0) sms = 1;
        sms_of[dev].store(sms, std::memory_order_relaxed);
    }
    *out = sms;
    return cudaSuccess;
}

// Per-bucket launches go out as programmatic dependents of the previous
// kernel in the stream: back-to-back buckets then lose the launch gap
// between them.  Stream order is kept: each CTA first waits for the
// previous kernel (griddepcontrol.wait in rs_kernel).
template <bool FROM_TABLE, class T, bool GROUPED>
static cudaError_t launch_rs_pdl(const ZsTile *d_tiles, const int32_t *d_order, int64_t tile0,
                                 int64_t ntiles,
                                 const RankPtrs &p, const uint16_t *const *tbl, int N, int G,
                                 uint16_t *gs, uint16_t *gP, double *partials, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ntiles);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int sms = 0;
    const cudaError_t e = sm_count(&sms);
    if (e != cudaSuccess) return e;
    const int prefetch = ntiles <= (int64_t)sms * RS_CTAS_PER_SM ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, rs_kernel<FROM_TABLE, T, GROUPED>, d_tiles, d_order, tile0, p,
                              prefetch, tbl, 0, N, G,
                              (float)N, gs, gP, partials);
}

template <class T>
static cudaError_t launch_rs(const ZsTile *d_tiles, const int32_t *d_order, int64_t tile0,
                             int64_t ntiles,
                             const RankPtrs &p, const void *const *d_table, int32_t bucket0, int N,
                             int G, uint16_t *gs,
                             uint16_t *gP, double *partials, cudaStream_t s) {
    const auto *tbl = reinterpret_cast<const uint16_t *const *>(d_table);
    const dim3 g((unsigned)ntiles), b(THREADS);
    if (d_table) {
        if (G == N) rs_kernel<true, T, false><<<g, b, 0, s>>>(d_tiles, nullptr, tile0, p, 0, tbl, bucket0, N, G, (float)N, gs, gP, partials);
        else rs_kernel<true, T, true><<<g, b, 0, s>>>(d_tiles, nullptr, tile0, p, 0, tbl, bucket0, N, G, (float)N, gs, gP, partials);
        return cudaGetLastError();
    }
    const cudaError_t e =
        G == N ? launch_rs_pdl<false, T, false>(d_tiles, d_order, tile0, ntiles, p, nullptr, N, G, gs, gP, partials, s)
               : launch_rs_pdl<false, T, true>(d_tiles, d_order, tile0, ntiles, p, nullptr, N, G, gs, gP, partials, s);
    return e != cudaSuccess ? e : cudaGetLastError();
}

cudaError_t zsl_reduce_scatter(const ZsTile *d_tiles, const int32_t *d_order, int64_t tile0,
                               int64_t ntiles, const void *const *rank_ptrs, int N, int G, int dtype, uint16_t *gs,
                               uint16_t *gP, double *partials, cudaStream_t s) {
    if (ntiles <= 0) return cudaSuccess;
    RankPtrs p;
    for (int k = 0; k < N; ++k) p.p[k] = static_cast<const uint16_t *>(rank_ptrs[k]);
    return dtype == ZS_DTYPE_FP16
               ? launch_rs<FP16T>(d_tiles, d_order, tile0, ntiles, p, nullptr, 0, N, G, gs, gP, partials, s)
               : launch_rs<BF16T>(d_tiles, d_order, tile0, ntiles, p, nullptr, 0, N, G, gs, gP, partials, s);
}

cudaError_t zsl_reduce_scatter_all(const ZsTile *d_tiles, int64_t tile0, int64_t ntiles,
                                   int32_t bucket0, const void *const *d_table, int N, int G,
                                   int dtype, uint16_t *gs, uint16_t *gP, double *partials,
                                   cudaStream_t s) {
    if (ntiles <= 0) return cudaSuccess;
    RankPtrs p = {};
    return dtype == ZS_DTYPE_FP16
               ? launch_rs<FP16T>(d_tiles, nullptr, tile0, ntiles, p, d_table, bucket0, N, G, gs, gP, partials, s)
               : launch_rs<BF16T>(d_tiles, nullptr, tile0, ntiles, p, d_table, bucket0, N, G, gs, gP, partials, s);
}

cudaError_t zsl_norm(const ZsTile *d_tiles, int64_t ntiles, int64_t n_level1, int dtype,
                     const uint16_t *gs, const uint16_t *gP, double *scratch, bool recompute,
                     float max_norm, float *d_norm, float *d_coef, int32_t *d_flags,
                     const ZsScaleArgs *scale, cudaStream_t s) {
    if (recompute && ntiles > 0) {
        // persistent grid: NORM_CTAS_PER_SM CTAs on every SM
        int sms = 0;
        const cudaError_t e = sm_count(&sms);
        if (e != cudaSuccess) return e;
        const int64_t warps = (ntiles + WARPS - 1) / WARPS;
        const int64_t grid = std::min<int64_t>(warps, (int64_t)sms * NORM_CTAS_PER_SM);
        if (dtype == ZS_DTYPE_FP16)
            norm_tiles_kernel<FP16T><<<(unsigned)grid, THREADS, 0, s>>>(d_tiles, ntiles, gs, gP,
                                                                         scratch);
        else
            norm_tiles_kernel<BF16T><<<(unsigned)grid, THREADS, 0, s>>>(d_tiles, ntiles, gs, gP,
                                                                         scratch);
    }
    norm_level1_kernel<<<(unsigned)n_level1, THREADS, 0, s>>>(scratch, ntiles, scratch + ntiles);
    ZsScaleArgs sc = {};
    if (scale) sc = *scale;
    norm_finish_kernel<<<1, THREADS, 0, s>>>(scratch + ntiles, n_level1, max_norm, d_norm, d_coef,
                                             d_flags, sc);
    return cudaGetLastError();
}

