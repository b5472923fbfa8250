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
    // largest |x| (bits & 0x7FFF) of a thread whose squares the norm sums in
    // float32 without error: all zero, or in [2^-40, 2^56) (squares too
    // small to be exact then weigh below 2^-69 of the largest; 256 thread
    // sums below 2^119 cannot overflow); Inf and NaN excluded
    static __device__ __forceinline__ bool sq_exact(uint32_t mx) {
        return mx < 0x5B80u && (mx == 0u || mx >= 0x2B80u);
    }
    // 2^(2E + 7), E = floor(log2 of the largest |x|) (mx a normal value)
    static __device__ __forceinline__ float sq_bound(uint32_t mx) {
        const int E = (int)(mx >> 7) - 127;
        return __int_as_float((2 * E + 7 + 127) << 23);
    }
};
struct FP16T {
    static __device__ __forceinline__ float to_f32(uint32_t b) {
        return __half2float(__ushort_as_half((unsigned short)b));
    }
    static __device__ __forceinline__ uint32_t from_f32(float x) {
        return (uint32_t)__half_as_ushort(__float2half_rn(x));
    }
    // finite binary16 values (squares in [2^-48, 65504^2], exact in float32)
    static __device__ __forceinline__ bool sq_exact(uint32_t mx) { return mx < 0x7C00u; }
    // 2^(2E + 7), E = floor(log2 of the largest |x|) (mx nonzero; a
    // subnormal's value is mx * 2^-24)
    static __device__ __forceinline__ float sq_bound(uint32_t mx) {
        const int ef = (int)(mx >> 10);
        const int E = ef ? ef - 15 : (31 - __clz((int)mx)) - 24;
        return __int_as_float((2 * E + 7 + 127) << 23);
    }
};

// ------------------------------------------------------------ the norm --
// The partial sum of squares of one tile is a function of the tile's stored
// values alone, so that every kernel that forms it, from any thread
// arrangement, gets the same bits:
//  * the window: the 16-byte aligned run [w0, w0 + 8*n_groups) around the
//    tile's values [dst, dst + valid), w0 = dst & ~7, cut into 8-element
//    groups; values outside [dst, dst + valid) count as 0;
//  * group g belongs to virtual thread g mod 256, which takes its groups in
//    increasing g (at most NORM_MAXG) and sums the squares of their values
//    with vt_sumsq below into a float32 pair hi + lo;
//  * the 256 pairs are added as double-floats: column c = 0..31 adds the
//    pairs of virtual threads c, c+32, ..., c+224 in that order, then the
//    32 columns are added by a butterfly (xor 16, 8, 4, 2, 1), and the
//    result is hi + lo in float64.
// When a virtual thread's values leave the exact range (|x| >= 2^56, Inf,
// NaN, or nonzero values all below 2^-40 in bf16), the whole tile is summed
// in float64 instead, with the same assignment of groups and the same tree
// (vt_sumsq_f64 below, and the float64 branch of the tile sums).
constexpr int NORM_VT = 256;                                   // virtual threads of a tile
constexpr int NORM_MAXG = (int)((ZS_TILE_ELEMS + 14) / 8 + NORM_VT - 1) / NORM_VT;  // 5
constexpr int NORM_WIN_ELEMS = (int)ZS_TILE_ELEMS + 16;        // window buffer (elements)

// two float32 in one 64-bit register, as the paired instructions take them
__device__ __forceinline__ unsigned long long f2pack(float a, float b) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ void f2unpack(unsigned long long r, float &a, float &b) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(a), "=f"(b) : "l"(r));
}

// Double-float addition (hi, lo) += (hi2, lo2): TwoSum of the heads, the
// tails added to its error, renormalised (Fast2Sum).
__device__ __forceinline__ void add22(float &hi, float &lo, float hi2, float lo2) {
    const float s = __fadd_rn(hi, hi2);
    const float bv = __fsub_rn(s, hi);
    const float av = __fsub_rn(s, bv);
    float e = __fadd_rn(__fsub_rn(hi, av), __fsub_rn(hi2, bv));
    e = __fadd_rn(e, __fadd_rn(lo, lo2));
    hi = __fadd_rn(s, e);
    lo = __fsub_rn(e, __fsub_rn(hi, s));
}

struct VtPair {
    float hi, lo;
    bool ok;
};

// Sum of squares of one virtual thread's groups w[0..n) (16-bit patterns,
// two per word, element 2j in the low half of word j; masked values 0),
// without rounding error up to about 2^-32 of the sum.  The even and the
// odd elements go to two accumulators, advanced together by Blackwell's
// paired float32 instructions.  Each accumulator starts at B, a power of two
// above 32 * max^2 (max the largest |x| of the thread), so it stays in
// [B, 2B) while it gains the squares (at most 20 per accumulator).  Then
// for a square x*x (exact in float32: at most 22 significant bits):
//   s = x*x + h;  d = h - s (exact, Sterbenz);  e = x*x + d (the exact
//   rounding error of s);  l = l + e;  h = s
// and h - B is exact at the end: four float32 operations per value.
template <class T, int NG>
__device__ __forceinline__ VtPair vt_sumsq(const uint4 (&w)[NG], int n) {
    uint32_t m2 = 0;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        if (g < n) {
            m2 = __vmaxu2(m2, w[g].x & 0x7FFF7FFFu);
            m2 = __vmaxu2(m2, w[g].y & 0x7FFF7FFFu);
            m2 = __vmaxu2(m2, w[g].z & 0x7FFF7FFFu);
            m2 = __vmaxu2(m2, w[g].w & 0x7FFF7FFFu);
        }
    }
    const uint32_t mx = max(m2 & 0xFFFFu, m2 >> 16);
    VtPair p;
    p.hi = 0.0f;
    p.lo = 0.0f;
    p.ok = T::sq_exact(mx);
    if (!p.ok || mx == 0u) return p;
    const float B = T::sq_bound(mx);
    const unsigned long long BB = f2pack(B, B);
    unsigned long long h = BB, l = 0;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        if (g < n) {
            const uint32_t x[4] = {w[g].x, w[g].y, w[g].z, w[g].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const unsigned long long v = f2pack(T::to_f32(x[j] & 0xFFFFu), T::to_f32(x[j] >> 16));
                unsigned long long s, dd, e;
                asm("fma.rn.f32x2 %0, %1, %1, %2;" : "=l"(s) : "l"(v), "l"(h));
                asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(dd) : "l"(h), "l"(s));
                asm("fma.rn.f32x2 %0, %1, %1, %2;" : "=l"(e) : "l"(v), "l"(dd));
                asm("add.rn.f32x2 %0, %1, %2;" : "=l"(l) : "l"(l), "l"(e));
                h = s;
            }
        }
    }
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(h) : "l"(h), "l"(BB));   // exact
    float he, ho, le, lo;
    f2unpack(h, he, ho);
    f2unpack(l, le, lo);
    // renormalise each pair (|l| is far below h: Fast2Sum), then add them
    float s = __fadd_rn(he, le);
    le = __fsub_rn(le, __fsub_rn(s, he));
    he = s;
    s = __fadd_rn(ho, lo);
    lo = __fsub_rn(lo, __fsub_rn(s, ho));
    ho = s;
    add22(he, le, ho, lo);
    p.hi = he;
    p.lo = le;
    return p;
}

// Float64 sum of squares of one virtual thread's groups, in order.
template <class T, int NG>
__device__ __forceinline__ double vt_sumsq_f64(const uint4 (&w)[NG], int n) {
    double s = 0.0;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
        if (g < n) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const double x = (double)T::to_f32(lane16(w[g], i));
                s = __dadd_rn(s, __dmul_rn(x, x));
            }
        }
    }
    return s;
}

// Group g of a window held at win (global or shared memory, 16-byte
// aligned), the values outside window positions [lo, hi) set to 0.
__device__ __forceinline__ uint4 win_group(const uint16_t *win, int64_t g, int64_t lo, int64_t hi) {
    uint4 v = *reinterpret_cast<const uint4 *>(win + 8 * g);
    if (8 * g < lo || 8 * g + 8 > hi) v = mask8(v, lo - 8 * g, hi - 8 * g);
    return v;
}

// Virtual thread vt's groups of a window with n_groups groups.
__device__ __forceinline__ int vt_groups(const uint16_t *win, int vt, int64_t n_groups, int64_t lo,
                                         int64_t hi, uint4 (&w)[NORM_MAXG]) {
    int n = 0;
#pragma unroll
    for (int j = 0; j < NORM_MAXG; ++j) {
        const int64_t g = vt + (int64_t)NORM_VT * j;
        w[j] = make_uint4(0, 0, 0, 0);
        if (g < n_groups) {
            w[j] = win_group(win, g, lo, hi);
            n = j + 1;
        }
    }
    return n;
}

// Shared memory of the tile norm in a CTA of NORM_VT threads.
struct SqRed {
    union {
        struct {
            float hi[NORM_VT], lo[NORM_VT];
        } p;
        double d[NORM_VT];
    } u;
};

// The tile norm in a CTA of NORM_VT threads, thread t being virtual thread
// t, from the window at win (written by this CTA before a barrier, or
// read-only memory).  All threads call it; the result is valid in thread 0.
template <class T>
__device__ __forceinline__ double tile_sumsq_cta(const uint16_t *win, int64_t n_groups, int64_t lo,
                                                 int64_t hi, SqRed &red) {
    const int t = threadIdx.x;
    uint4 w[NORM_MAXG];
    const int n = vt_groups(win, t, n_groups, lo, hi, w);
    const VtPair p = vt_sumsq<T>(w, n);
    red.u.p.hi[t] = p.hi;
    red.u.p.lo[t] = p.lo;
    double s = 0.0;
    if (__syncthreads_and(p.ok)) {
        if (t < 32) {
            float h = red.u.p.hi[t], l = red.u.p.lo[t];
#pragma unroll
            for (int m = 1; m < NORM_VT / 32; ++m) add22(h, l, red.u.p.hi[32 * m + t], red.u.p.lo[32 * m + t]);
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float h2 = __shfl_xor_sync(0xFFFFFFFFu, h, off);
                const float l2 = __shfl_xor_sync(0xFFFFFFFFu, l, off);
                add22(h, l, h2, l2);
            }
            s = __dadd_rn((double)h, (double)l);
        }
        return s;
    }
    // float64 for the whole tile
    const double f = vt_sumsq_f64<T>(w, n);
    __syncthreads();            // every thread has read the pairs
    red.u.d[t] = f;
    __syncthreads();
    if (t < 32) {
        double c = red.u.d[t];
#pragma unroll
        for (int m = 1; m < NORM_VT / 32; ++m) c = __dadd_rn(c, red.u.d[32 * m + t]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) c = __dadd_rn(c, __shfl_xor_sync(0xFFFFFFFFu, c, off));
        s = c;
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

// ------------------------------------------------- shared memory, TMA --
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Waits for the phase of parity `parity` of the mbarrier at shared address
// bar to complete; false when limit_ns pass first (the clock is read every
// 64 polls; a poll count far beyond any such time is a second bound).
__device__ inline bool mbar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = global_ns();
    for (long long i = 0; i < (1ll << 34); ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar), "r"(parity)
            : "memory");
        if (done) return true;
        if ((i & 63) == 63 && global_ns() - t0 > limit_ns) return false;
    }
    return false;
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
