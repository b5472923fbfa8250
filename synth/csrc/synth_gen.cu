// Synthetic-input generator on the GPU: the same Philox4x32-10 draws and
// value mappings as synth/philox.py, written into device buffers.  Test and
// benchmark infrastructure; holds no arithmetic of the ZeRO-3 step.
//
// Philox4x32-10 from its published definition (Salmon et al., SC'11):
// counter (c0..c3), key (k0, k1); ten rounds of
//   (hi0, lo0) = M0 * c0, (hi1, lo1) = M1 * c2,
//   c = (hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0),  k += (W0, W1)
// Counter layout: (index lo, index hi, sub, stream), key: (seed lo, seed hi).
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace {

constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
constexpr int THREADS = 256;

__device__ __forceinline__ uint4 philox(uint64_t idx, uint32_t sub, uint32_t stream, uint32_t k0,
                                        uint32_t k1) {
    uint32_t c0 = (uint32_t)idx, c1 = (uint32_t)(idx >> 32), c2 = sub, c3 = stream;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(M0, c0), lo0 = M0 * c0;
        const uint32_t hi1 = __umulhi(M1, c2), lo1 = M1 * c2;
        const uint32_t n0 = hi1 ^ c1 ^ k0, n2 = hi0 ^ c3 ^ k1;
        c0 = n0;
        c1 = lo1;
        c2 = n2;
        c3 = lo0;
        k0 += W0;
        k1 += W1;
    }
    return make_uint4(c0, c1, c2, c3);
}

// Irwin-Hall of the 8 16-bit halves: exact integer in [-524280, 524280]
__device__ __forceinline__ float normal(uint4 w, float c) {
    const uint32_t s = (w.x & 0xFFFFu) + (w.x >> 16) + (w.y & 0xFFFFu) + (w.y >> 16) +
                       (w.z & 0xFFFFu) + (w.z >> 16) + (w.w & 0xFFFFu) + (w.w >> 16);
    const int32_t z = 2 * (int32_t)s - 8 * 65535;
    return __fmul_rn((float)z, c);
}

constexpr uint32_t STREAM_GRAD = 1, STREAM_OUTLIER = 2;

__global__ void grad_kernel(uint16_t *out, int64_t start, int64_t count, uint32_t k0, uint32_t k1,
                            uint32_t sub, float c, uint32_t othr, float oscale) {
    for (int64_t i = (int64_t)blockIdx.x * THREADS + threadIdx.x; i < count;
         i += (int64_t)gridDim.x * THREADS) {
        const uint64_t idx = (uint64_t)(start + i);
        float v = normal(philox(idx, sub, STREAM_GRAD, k0, k1), c);
        if (othr != 0u && philox(idx, sub, STREAM_OUTLIER, k0, k1).x < othr) v = __fmul_rn(v, oscale);
        out[i] = (uint16_t)(__float_as_uint(v) >> 16);
    }
}

__global__ void normal_kernel(float *out, int64_t start, int64_t count, uint32_t k0, uint32_t k1,
                              uint32_t sub, uint32_t stream, float c) {
    for (int64_t i = (int64_t)blockIdx.x * THREADS + threadIdx.x; i < count;
         i += (int64_t)gridDim.x * THREADS)
        out[i] = normal(philox((uint64_t)(start + i), sub, stream, k0, k1), c);
}

// fp16: floor(z / 512) * 2^e, exactly representable in binary16
__global__ void grad_fp16_kernel(uint16_t *out, int64_t start, int64_t count, uint32_t k0,
                                 uint32_t k1, uint32_t sub, int e, uint32_t othr, int oe) {
    for (int64_t i = (int64_t)blockIdx.x * THREADS + threadIdx.x; i < count;
         i += (int64_t)gridDim.x * THREADS) {
        const uint64_t idx = (uint64_t)(start + i);
        const uint4 w = philox(idx, sub, STREAM_GRAD, k0, k1);
        const int32_t s = (int32_t)((w.x & 0xFFFFu) + (w.x >> 16) + (w.y & 0xFFFFu) + (w.y >> 16) +
                                    (w.z & 0xFFFFu) + (w.z >> 16) + (w.w & 0xFFFFu) + (w.w >> 16));
        const int32_t z = 2 * s - 8 * 65535;
        const int32_t k = (z >= 0) ? (z / 512) : -((-z + 511) / 512);  // floor(z / 512)
        int ee = e;
        if (othr != 0u && philox(idx, sub, STREAM_OUTLIER, k0, k1).x < othr) ee += oe;
        const float v = ldexpf((float)k, ee);
        out[i] = __half_as_ushort(__float2half_rn(v));
    }
}

// Stand-in compute for scheduling experiments: every thread runs `iters`
// dependent FMAs on registers (bounded loop, no memory waits) and one thread
// writes the result so the work is kept.
__global__ void busy_kernel(int64_t iters, float *sink) {
    float x = (float)threadIdx.x * 1e-3f, y = 1.0000001f;
    for (int64_t i = 0; i < iters; ++i) x = fmaf(x, y, 1e-7f);
    if (threadIdx.x == 0 && blockIdx.x == 0 && x == -1.0f) *sink = x;
}

unsigned blocks_for(int64_t count) {
    int64_t b = (count + THREADS - 1) / THREADS;
    if (b > 152 * 16) b = 152 * 16;
    return (unsigned)(b < 1 ? 1 : b);
}

}  // namespace

extern "C" {

// out[i] = gradient value (bf16 bits, truncated) at index start + i.
int zsg_fill_grad_bf16(void *out, int64_t start, int64_t count, uint64_t seed, uint32_t sub,
                       float c, uint32_t outlier_thr, float outlier_scale, void *stream) {
    if (count <= 0) return 0;
    grad_kernel<<<blocks_for(count), THREADS, 0, (cudaStream_t)stream>>>(
        static_cast<uint16_t *>(out), start, count, (uint32_t)seed, (uint32_t)(seed >> 32), sub, c,
        outlier_thr, outlier_scale);
    return (int)cudaGetLastError();
}

// out[i] = fp16 gradient value (binary16 bits, exact) at index start + i.
int zsg_fill_grad_fp16(void *out, int64_t start, int64_t count, uint64_t seed, uint32_t sub,
                       int log2_scale, uint32_t outlier_thr, int outlier_log2, void *stream) {
    if (count <= 0) return 0;
    grad_fp16_kernel<<<blocks_for(count), THREADS, 0, (cudaStream_t)stream>>>(
        static_cast<uint16_t *>(out), start, count, (uint32_t)seed, (uint32_t)(seed >> 32), sub,
        log2_scale, outlier_thr, outlier_log2);
    return (int)cudaGetLastError();
}

// Busy compute of `iters` FMA steps per thread on `blocks` CTAs of
// `threads` threads (a multiple of 32, at most 256).  With one warp per SM
// the dependent chain takes time while leaving the SM's issue slots and the
// memory system to other streams, the way tensor-core compute does.
int zsg_busy(int64_t iters, int blocks, int threads, float *sink, void *stream) {
    if (iters <= 0 || blocks <= 0 || threads <= 0 || threads > THREADS || threads % 32) return 0;
    busy_kernel<<<blocks, threads, 0, (cudaStream_t)stream>>>(iters, sink);
    return (int)cudaGetLastError();
}

// out[i] = normal value (float32) of stream `stream_tag` at index start + i.
int zsg_fill_normal_f32(float *out, int64_t start, int64_t count, uint64_t seed, uint32_t sub,
                        uint32_t stream_tag, float c, void *stream) {
    if (count <= 0) return 0;
    normal_kernel<<<blocks_for(count), THREADS, 0, (cudaStream_t)stream>>>(
        out, start, count, (uint32_t)seed, (uint32_t)(seed >> 32), sub, stream_tag, c);
    return (int)cudaGetLastError();
}

}  // extern "C"
