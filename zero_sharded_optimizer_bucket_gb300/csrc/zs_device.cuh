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
    // largest |x| (bits & 0x7FFF) for which the squares of 8 values neither
    // overflow float32 (|x| < 2^60) nor all underflow (|x| >= 2^-64)
    static __device__ __forceinline__ bool sq_in_f32(uint32_t mx) {
        return mx < 0x5D80u && (mx == 0u || mx >= 0x1F80u);
    }
};
struct FP16T {
    static __device__ __forceinline__ float to_f32(uint32_t b) {
        return __half2float(__ushort_as_half((unsigned short)b));
    }
    static __device__ __forceinline__ uint32_t from_f32(float x) {
        return (uint32_t)__half_as_ushort(__float2half_rn(x));
    }
    // binary16 squares (<= 65504^2, >= 2^-48) always fit float32
    static __device__ __forceinline__ bool sq_in_f32(uint32_t) { return true; }
};

// Sum of squares of 8 16-bit values for the norm partial.  In float32 when
// that can neither overflow nor lose the whole group to underflow, in
// float64 otherwise (Inf / NaN propagate either way).  Fixed order, no
// contraction: the value depends only on the 8 inputs, so every kernel that
// calls it gets the same bits.
template <class T>
__device__ __forceinline__ void group_sq(const uint32_t r[8], float &acc32, double &acc64) {
    uint32_t mx = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) mx = max(mx, r[i] & 0x7FFFu);
    if (!T::sq_in_f32(mx)) {
        double s = 0.0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const double v = (double)T::to_f32(r[i]);
            s = __dadd_rn(s, __dmul_rn(v, v));
        }
        acc64 = __dadd_rn(acc64, s);
    } else {
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const float v = T::to_f32(r[i]);
            s = __fadd_rn(s, __fmul_rn(v, v));
        }
        acc32 = __fadd_rn(acc32, s);
    }
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
