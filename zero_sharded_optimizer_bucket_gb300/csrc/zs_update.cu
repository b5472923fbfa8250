// A4 Adam(W) + bf16 cast, the fused pass 2 (Adam + cast + gathered write),
// and the A1 partition copy.
//
// The optimizer sees only each rank's fp32 partition and writes the 16-bit
// shard back ([ZeRO-3 chapter] §6.3); per element it is a pure stream of
// 14 bytes read (bf16 grad + fp32 master, m, v) and 14 bytes written
// (fp32 master, m, v + bf16 shard), 16-byte vectors throughout.
#include "zs_device.cuh"
#include "zs_launch.h"

namespace zsk {

struct StatePtrs {
    const uint16_t *g;
    uint16_t *param;
    float *p, *m, *v;
};

__device__ __forceinline__ StatePtrs pick(const zs_shard_state &st, bool persistent) {
    StatePtrs s;
    if (persistent) {
        s.g = static_cast<const uint16_t *>(st.persist_grads);
        s.param = static_cast<uint16_t *>(st.persist_params);
        s.p = st.p_master;
        s.m = st.p_exp_avg;
        s.v = st.p_exp_avg_sq;
    } else {
        s.g = static_cast<const uint16_t *>(st.grad_shards);
        s.param = static_cast<uint16_t *>(st.param_shards);
        s.p = st.master;
        s.m = st.exp_avg;
        s.v = st.exp_avg_sq;
    }
    return s;
}

__device__ __forceinline__ void load8f(const float *a, float o[8]) {
    const float4 x = *reinterpret_cast<const float4 *>(a);
    const float4 y = *reinterpret_cast<const float4 *>(a + 4);
    o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w;
    o[4] = y.x; o[5] = y.y; o[6] = y.z; o[7] = y.w;
}

__device__ __forceinline__ void store8f(float *a, const float o[8]) {
    *reinterpret_cast<float4 *>(a) = make_float4(o[0], o[1], o[2], o[3]);
    *reinterpret_cast<float4 *>(a + 4) = make_float4(o[4], o[5], o[6], o[7]);
}

// 8 aligned elements at off: Adam on all of them, bf16 results in r.
template <class T, bool SHARD = true>
__device__ __forceinline__ void adam8(const StatePtrs &s, int64_t off, float coef, const AdamC &c,
                                      uint32_t r[8]) {
    const uint4 gv = ldg16(s.g + off);
    float p[8], m[8], v[8];
    load8f(s.p + off, p);
    load8f(s.m + off, m);
    load8f(s.v + off, v);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        adam_elem(p[i], m[i], v[i], T::to_f32(lane16(gv, i)), coef, c);
        r[i] = T::from_f32(p[i]);
    }
    store8f(s.p + off, p);
    store8f(s.m + off, m);
    store8f(s.v + off, v);
    // SHARD false: no shard buffer, the parameters live only in the replica
    if (SHARD) *reinterpret_cast<uint4 *>(s.param + off) = pack8(r);
}

template <class T, bool SHARD = true>
__device__ __forceinline__ uint32_t adam1(const StatePtrs &s, int64_t x, float coef,
                                          const AdamC &c) {
    float p = s.p[x], m = s.m[x], v = s.v[x];
    adam_elem(p, m, v, T::to_f32(s.g[x]), coef, c);
    const uint32_t r = T::from_f32(p);
    s.p[x] = p;
    s.m[x] = m;
    s.v[x] = v;
    if (SHARD) s.param[x] = (uint16_t)r;
    return r;
}

// Unfused Adam over one sub-group: blockIdx.y < N walks shard row y,
// columns [s_lo, s_lo + W); blockIdx.y == N walks persistent [p_lo, p_lo + PW).
template <class T>
__global__ void __launch_bounds__(THREADS)
adam_kernel(int N, int64_t S, int64_t s_lo, int64_t W, int64_t p_lo, int64_t PW, AdamC c,
            const float *__restrict__ d_coef, const int32_t *__restrict__ d_flags,
            zs_shard_state st) {
    if (*d_flags & ZS_SKIP_NONFINITE) return;
    const float coef = *d_coef;
    const bool pers = (int)blockIdx.y == N;
    const StatePtrs s = pick(st, pers);
    const int64_t base = pers ? p_lo : (int64_t)blockIdx.y * S + s_lo;
    const int64_t units = (pers ? PW : W) >> 3;
    for (int64_t u = (int64_t)blockIdx.x * THREADS + threadIdx.x; u < units;
         u += (int64_t)gridDim.x * THREADS) {
        uint32_t r[8];
        adam8<T>(s, base + 8 * u, coef, c, r);
    }
}

// Fused pass 2: Adam + cast on one tile, and the cast parameters also
// written at their place in model flat space (the all-gather of the next
// forward pass, [ZeRO-3 chapter] §5.2), straight from registers.
template <class T, bool SHARD>
__global__ void __launch_bounds__(THREADS)
step2_kernel(const ZsTile *__restrict__ tiles, AdamC c, const float *__restrict__ d_coef,
             const int32_t *__restrict__ d_flags, zs_shard_state st,
             uint16_t *__restrict__ flat_out, int a0) {
    if (*d_flags & ZS_SKIP_NONFINITE) return;
    const float coef = *d_coef;
    const ZsTile tile = tiles[blockIdx.x];
    const bool pers = tile.flat < 0;
    const StatePtrs s = pick(st, pers);
    const int64_t D = tile.dst, G0 = D & ~int64_t(7), L = tile.len;
    const int64_t ngroups = (D + L - G0 + 7) >> 3;
    const int64_t fdelta = tile.flat - D;
    const int fq = (int)((a0 + G0 + fdelta) & 7);
    const int lane = threadIdx.x & 31;
    // uniform trip count: every lane takes part in the shuffles below
    for (int64_t base = 0; base < ngroups; base += THREADS) {
        const int64_t gi = base + threadIdx.x;
        const bool act = gi < ngroups;
        const int64_t x0 = G0 + 8 * gi;
        uint32_t r[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) r[i] = 0u;
        if (act) {
            // persistent parameters are always stored whole; shard tiles
            // skip the shard store when SHARD is false (tile-uniform branch)
            if (x0 >= D && x0 + 8 <= D + L) {
                if (pers) adam8<T, true>(s, x0, coef, c, r);
                else adam8<T, SHARD>(s, x0, coef, c, r);
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (x0 + i >= D && x0 + i < D + L)
                        r[i] = pers ? adam1<T, true>(s, x0 + i, coef, c)
                                    : adam1<T, SHARD>(s, x0 + i, coef, c);
            }
        }
        if (pers) continue;
        // slots i with li0 + i in [0, flat_len) go to model flat space
        const int64_t li0 = x0 - D;
        const int64_t lo = -li0, hi = tile.flat_len - li0;
        if (fq == 0) {
            if (act) {
                if (lo <= 0 && hi >= 8) {
                    *reinterpret_cast<uint4 *>(flat_out + x0 + fdelta) = pack8(r);
                } else {
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        if (i >= lo && i < hi) flat_out[x0 + i + fdelta] = (uint16_t)r[i];
                }
            }
        } else {
            // the group's flat positions start fq past a 16-byte boundary:
            // slots [8-fq, 8) of this lane and [0, 8-fq) of the next lane
            // make one aligned 16-byte store
            const uint4 w = pack8(r);
            uint4 wn;
            wn.x = __shfl_down_sync(0xFFFFFFFFu, w.x, 1);
            wn.y = __shfl_down_sync(0xFFFFFFFFu, w.y, 1);
            wn.z = __shfl_down_sync(0xFFFFFFFFu, w.z, 1);
            wn.w = __shfl_down_sync(0xFFFFFFFFu, w.w, 1);
            const bool next_act = __shfl_down_sync(0xFFFFFFFFu, (int)act, 1) != 0 && lane < 31;
            const bool vec = act && next_act && lo <= 8 - fq && hi >= 16 - fq;
            if (vec)
                *reinterpret_cast<uint4 *>(flat_out + x0 + fdelta + 8 - fq) = shift8(w, wn, 8 - fq);
            const bool prev_vec = __shfl_up_sync(0xFFFFFFFFu, (int)vec, 1) != 0 && lane > 0;
            if (act) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const bool done = (i < 8 - fq) ? prev_vec : vec;
                    if (!done && i >= lo && i < hi) flat_out[x0 + i + fdelta] = (uint16_t)r[i];
                }
            }
        }
    }
}

// Partition copy: dst <- W[win + i] (0 beyond valid), moments zero, bf16 shard.
template <class T>
__global__ void __launch_bounds__(THREADS)
partition_kernel(const ZsTile *__restrict__ tiles, const float *__restrict__ W, zs_shard_state st) {
    const ZsTile tile = tiles[blockIdx.x];
    const bool pers = tile.flat < 0;
    const StatePtrs s = pick(st, pers);
    const int64_t D = tile.dst, G0 = D & ~int64_t(7), L = tile.len;
    const int64_t ngroups = (D + L - G0 + 7) >> 3;
    for (int64_t gi = threadIdx.x; gi < ngroups; gi += THREADS) {
        const int64_t x0 = G0 + 8 * gi;
        float w[8];
        uint32_t r[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t li = x0 + i - D;
            w[i] = (li >= 0 && li < tile.valid) ? __ldg(W + tile.win + li) : 0.0f;
            r[i] = T::from_f32(w[i]);
        }
        if (x0 >= D && x0 + 8 <= D + L) {
            const float z[8] = {0, 0, 0, 0, 0, 0, 0, 0};
            store8f(s.p + x0, w);
            store8f(s.m + x0, z);
            store8f(s.v + x0, z);
            *reinterpret_cast<uint4 *>(s.param + x0) = pack8(r);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int64_t x = x0 + i;
                if (x >= D && x < D + L) {
                    s.p[x] = w[i];
                    s.m[x] = 0.0f;
                    s.v[x] = 0.0f;
                    s.param[x] = (uint16_t)r[i];
                }
            }
        }
    }
}

__host__ AdamC to_device(const ZsAdamScalars &a) {
    AdamC c;
    c.lr = a.lr; c.b1 = a.b1; c.b2 = a.b2; c.omb1 = a.omb1; c.omb2 = a.omb2; c.eps = a.eps;
    c.wd = a.wd; c.lr_wd = a.lr_wd; c.bc1 = a.bc1; c.bc2 = a.bc2; c.adamw = a.adamw;
    return c;
}

}  // namespace zsk

using namespace zsk;

cudaError_t zsl_adam(int N, int dtype, int64_t S, int64_t s_lo, int64_t s_hi, int64_t p_lo,
                     int64_t p_hi, const ZsAdamScalars &a, const float *d_coef,
                     const int32_t *d_flags, const zs_shard_state &st, cudaStream_t s) {
    const int64_t W = s_hi - s_lo, PW = p_hi - p_lo;
    if ((W <= 0 || N == 0) && PW <= 0) return cudaSuccess;
    const int64_t units = (W > PW ? W : PW) / 8;
    int64_t x = (units + THREADS - 1) / THREADS;
    const int64_t cap = 2048 / (N + 1) + 1;
    if (x > cap) x = cap;
    if (x < 1) x = 1;
    dim3 grid((unsigned)x, (unsigned)(N + 1));
    if (dtype == ZS_DTYPE_FP16)
        adam_kernel<FP16T><<<grid, THREADS, 0, s>>>(N, S, s_lo, W, p_lo, PW, to_device(a), d_coef,
                                                    d_flags, st);
    else
        adam_kernel<BF16T><<<grid, THREADS, 0, s>>>(N, S, s_lo, W, p_lo, PW, to_device(a), d_coef,
                                                    d_flags, st);
    return cudaGetLastError();
}

cudaError_t zsl_step2(const ZsTile *d_tiles, int64_t ntiles, int dtype, const ZsAdamScalars &a,
                      const float *d_coef, const int32_t *d_flags, const zs_shard_state &st,
                      uint16_t *flat_out, cudaStream_t s) {
    if (ntiles <= 0) return cudaSuccess;
    const int a0 = (int)((reinterpret_cast<uintptr_t>(flat_out) >> 1) & 7);
    const dim3 g((unsigned)ntiles), b(THREADS);
    const AdamC c = to_device(a);
    if (dtype == ZS_DTYPE_FP16) {
        if (st.param_shards) step2_kernel<FP16T, true><<<g, b, 0, s>>>(d_tiles, c, d_coef, d_flags, st, flat_out, a0);
        else step2_kernel<FP16T, false><<<g, b, 0, s>>>(d_tiles, c, d_coef, d_flags, st, flat_out, a0);
    } else {
        if (st.param_shards) step2_kernel<BF16T, true><<<g, b, 0, s>>>(d_tiles, c, d_coef, d_flags, st, flat_out, a0);
        else step2_kernel<BF16T, false><<<g, b, 0, s>>>(d_tiles, c, d_coef, d_flags, st, flat_out, a0);
    }
    return cudaGetLastError();
}

cudaError_t zsl_partition(const ZsTile *d_tiles, int64_t ntiles, int dtype, const float *W,
                          const zs_shard_state &st, cudaStream_t s) {
    if (ntiles <= 0) return cudaSuccess;
    if (dtype == ZS_DTYPE_FP16)
        partition_kernel<FP16T><<<(unsigned)ntiles, THREADS, 0, s>>>(d_tiles, W, st);
    else
        partition_kernel<BF16T><<<(unsigned)ntiles, THREADS, 0, s>>>(d_tiles, W, st);
    return cudaGetLastError();
}
