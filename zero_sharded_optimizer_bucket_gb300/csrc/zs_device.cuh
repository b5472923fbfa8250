// Device helpers shared by the libzs kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "zs_internal.h"

namespace zsk {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;

// bf16 bit pattern -> float (exact: the bits become the upper half)
__device__ __forceinline__ float bf2f(uint32_t b) { return __uint_as_float(b << 16); }

// float -> bf16 bit pattern, round to nearest even
__device__ __forceinline__ uint32_t f2bf(float x) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
}

__device__ __forceinline__ uint32_t lane16(const uint4 &v, int i) {
    const uint32_t w = (i < 2) ? v.x : (i < 4) ? v.y : (i < 6) ? v.z : v.w;
    return (i & 1) ? (w >> 16) : (w & 0xFFFFu);
}

__device__ __forceinline__ uint4 pack8(const uint32_t r[8]) {
    return make_uint4(r[0] | (r[1] << 16), r[2] | (r[3] << 16), r[4] | (r[5] << 16),
                      r[6] | (r[7] << 16));
}

// The 8 bf16 lanes q..q+7 of the 16-lane concatenation (a, b), q in 0..7.
// q is uniform over a tile, so the selects below do not diverge.
__device__ __forceinline__ uint4 shift8(const uint4 &a, const uint4 &b, int q) {
    const uint32_t w[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    const int s = q >> 1;
    uint32_t u[5];
#pragma unroll
    for (int j = 0; j < 5; ++j) {
        // w[j + s] with s in 0..3, without dynamic register indexing
        const uint32_t x0 = w[j], x1 = (j + 1 < 8) ? w[j + 1] : 0u;
        const uint32_t x2 = (j + 2 < 8) ? w[j + 2] : 0u, x3 = (j + 3 < 8) ? w[j + 3] : 0u;
        u[j] = (s == 0) ? x0 : (s == 1) ? x1 : (s == 2) ? x2 : x3;
    }
    if (q & 1) {
        return make_uint4(__funnelshift_r(u[0], u[1], 16), __funnelshift_r(u[1], u[2], 16),
                          __funnelshift_r(u[2], u[3], 16), __funnelshift_r(u[3], u[4], 16));
    }
    return make_uint4(u[0], u[1], u[2], u[3]);
}

// Zero the lanes outside [lo, hi) (lane indices, any integers).
__device__ __forceinline__ uint4 mask8(const uint4 &v, int64_t lo, int64_t hi) {
    uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        if (i < lo || i >= hi) w[i >> 1] &= (i & 1) ? 0x0000FFFFu : 0xFFFF0000u;
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// 16-bit storage types: bit pattern <-> float.
struct BF16T {
    static __device__ __forceinline__ float to_f32(uint32_t b) { return bf2f(b); }
    static __device__ __forceinline__ uint32_t from_f32(float x) { return f2bf(x); }
    // largest |x| (bits & 0x7FFF) of a group summed in the float32 pair:
    // below 2^60 (no square or partial sum of a thread overflows) and, unless
    // all are zero, at least 2^-40 (squares too small to be exact in float32
    // then weigh below 2^-69 of the group's); Inf and NaN excluded
    static __device__ __forceinline__ bool sq_exact(uint32_t mx) {
        return mx < 0x5D80u && (mx == 0u || mx >= 0x2B80u);
    }
};
struct FP16T {
    static __device__ __forceinline__ float to_f32(uint32_t b) {
        return __half2float(__ushort_as_half((unsigned short)b));
    }
    static __device__ __forceinline__ uint32_t from_f32(float x) {
        return (uint32_t)__half_as_ushort(__float2half_rn(x));
    }
    // finite binary16 squares (<= 65504^2, >= 2^-48) are exact in float32;
    // Inf and NaN go to the float64 sum
    static __device__ __forceinline__ bool sq_exact(uint32_t mx) { return mx < 0x7C00u; }
};

// Norm accumulators of one thread: the sum of squares of its values kept
// without rounding error as the float32 pair hi + lo (a double-float), and
// a float64 sum for groups outside the pair's exact range.
struct SqAcc {
    float hi = 0.0f, lo = 0.0f;
    double d = 0.0;
};

// (hi, lo) += v*v with no rounding error: v*v is exact in float32 (a 16-bit
// value has at most 11 significant bits, its square at most 22), s is the
// rounded sum and the TwoSum error term e is exact, so hi + lo gains exactly
// v*v up to the rounding of lo itself (relative 2^-48 of the sum).  The
// products are formed by fused multiply-adds, which equal the separately
// rounded operations here because v*v is exact.
__device__ __forceinline__ void sq_add_exact(float v, SqAcc &a) {
    const float s = __fmaf_rn(v, v, a.hi);
    const float bv = __fsub_rn(s, a.hi);
    const float av = __fsub_rn(s, bv);
    const float e = __fadd_rn(__fsub_rn(a.hi, av), __fmaf_rn(v, v, -bv));
    a.hi = s;
    a.lo = __fadd_rn(a.lo, e);
}

// Double-float addition (hi, lo) += (hi2, lo2): TwoSum of the heads, the
// tails added to its error, renormalised (Fast2Sum); relative error about
// 2^-46.
__device__ __forceinline__ void add22(float &hi, float &lo, float hi2, float lo2) {
    const float s = __fadd_rn(hi, hi2);
    const float bv = __fsub_rn(s, hi);
    const float av = __fsub_rn(s, bv);
    float e = __fadd_rn(__fsub_rn(hi, av), __fsub_rn(hi2, bv));
    e = __fadd_rn(e, __fadd_rn(lo, lo2));
    hi = __fadd_rn(s, e);
    lo = __fsub_rn(e, __fsub_rn(hi, s));
}

// Sum of squares of 8 16-bit values into a thread's norm accumulators, in
// element order.  A group whose largest |x| keeps every square and every
// partial sum of the thread inside float32's range (T::sq_exact) goes into
// the exact pair; any other group (huge or tiny values, Inf, NaN) into the
// float64 sum.  The result depends only on the 8 inputs and the order of
// the calls, so every kernel that makes the same calls gets the same bits.
template <class T>
__device__ __forceinline__ void group_sq(const uint32_t r[8], SqAcc &acc) {
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) mx = max(mx, r[i] & 0x7FFFu);
    if (!T::sq_exact(mx)) {
        double s = 0.0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const double v = (double)T::to_f32(r[i]);
            s = __dadd_rn(s, __dmul_rn(v, v));
        }
        acc.d = __dadd_rn(acc.d, s);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) sq_add_exact(T::to_f32(r[i]), acc);
    }
}

// Shared memory of block_sum_sq.
struct SqRed {
    float hi[WARPS], lo[WARPS];
    double d[WARPS];
    int ok[WARPS];
};

// Deterministic block sum of the threads' norm accumulators; the result is
// valid in thread 0.  A warp whose threads all have d == 0 and hi below
// 2^119 sums the pairs by double-float additions (fixed butterfly): 256
// such pairs cannot overflow.  Any other warp sums hi + lo + d in float64.
// Thread 0 adds the warps in order, by double-float additions when every
// warp took that path (converting once), else in float64.  GB300 runs
// float64 at a small fraction of the float32 rate, so the common case keeps
// the float64 pipe out of the reduction; the pair arithmetic keeps the
// partial about as accurate as float64 would.  Every choice and rounding
// depends only on the accumulators.
__device__ __forceinline__ double block_sum_sq(const SqAcc &a, SqRed &red) {
    const bool ok = a.d == 0.0 && a.hi < 0x1p119f;   // false for NaN
    const bool wok = __all_sync(0xFFFFFFFFu, ok);
    float hi = a.hi, lo = a.lo;
    double d = 0.0;
    if (wok) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float h2 = __shfl_xor_sync(0xFFFFFFFFu, hi, off);
            const float l2 = __shfl_xor_sync(0xFFFFFFFFu, lo, off);
            add22(hi, lo, h2, l2);
        }
    } else {
        d = __dadd_rn(__dadd_rn((double)a.hi, (double)a.lo), a.d);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1)
            d = __dadd_rn(d, __shfl_xor_sync(0xFFFFFFFFu, d, off));
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
        red.hi[warp] = hi;
        red.lo[warp] = lo;
        red.d[warp] = d;
        red.ok[warp] = wok;
    }
    __syncthreads();
    double s = 0.0;
    if (threadIdx.x == 0) {
        bool all = true;
        for (int w = 0; w < WARPS; ++w) all = all && red.ok[w];
        if (all) {
            float h = 0.0f, l = 0.0f;
            for (int w = 0; w < WARPS; ++w) add22(h, l, red.hi[w], red.lo[w]);
            s = __dadd_rn((double)h, (double)l);
        } else {
            for (int w = 0; w < WARPS; ++w)
                s = __dadd_rn(s, red.ok[w] ? __dadd_rn((double)red.hi[w], (double)red.lo[w])
                                           : red.d[w]);
        }
    }
    return s;
}

// Deterministic block sum (fixed butterfly per warp, warps in order);
// the result is valid in thread 0.
__device__ __forceinline__ double block_sum(double v, double *red /* [WARPS] */) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v = __dadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, off));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) red[warp] = v;
    __syncthreads();
    double s = 0.0;
    if (threadIdx.x == 0) {
        for (int w = 0; w < WARPS; ++w) s = __dadd_rn(s, red[w]);
    }
    return s;
}

struct AdamC {
    float lr, b1, b2, omb1, omb2, eps, wd, lr_wd, bc1, bc2;
    int adamw;
};

// One Adam(W) update in float32, each operation rounded, no contraction:
//   g = grad*coef; AdamW: p -= (lr*wd)*p | L2: g += wd*p
//   m = b1*m + (1-b1)*g; v = b2*v + (1-b2)*(g*g)
//   p -= lr * ((m/bc1) / (sqrt(v/bc2) + eps))
__device__ __forceinline__ void adam_elem(float &p, float &m, float &v, float grad, float coef,
                                          const AdamC &c) {
    float g = __fmul_rn(grad, coef);
    if (c.adamw)
        p = __fsub_rn(p, __fmul_rn(c.lr_wd, p));
    else
        g = __fadd_rn(g, __fmul_rn(c.wd, p));
    m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.omb1, g));
    v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(c.omb2, __fmul_rn(g, g)));
    const float mh = __fdiv_rn(m, c.bc1);
    const float vh = __fdiv_rn(v, c.bc2);
    const float den = __fadd_rn(__fsqrt_rn(vh), c.eps);
    p = __fsub_rn(p, __fmul_rn(c.lr, __fdiv_rn(mh, den)));
}

__device__ __forceinline__ uint4 ldg16(const uint16_t *p) {
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

}  // namespace zsk
