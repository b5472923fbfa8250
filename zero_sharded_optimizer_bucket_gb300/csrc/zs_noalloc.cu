// zs_grad_norm_noalloc: the gradient norm for callers that cannot allocate.
//
// zs_grad_norm needs a norm_scratch buffer from its caller.  Some callers
// have no way to get one: a plugin that a host framework hands only its
// input and output buffers (the framework owns all device memory and offers
// no scratch), or a step loop that must not call cudaMalloc because
// cudaMalloc can synchronise the whole device.  This entry point keeps the
// scratch in a fixed array of this library instead, so it allocates nothing.
//
// The array is ZS_NOALLOC_NORM_MAX_SCRATCH doubles (8 MiB) in device memory,
// held by every GPU that loads the library until the process exits.  Its
// address is looked up once per device (cudaGetSymbolAddress, with that
// device current) on the first call made on that device.
#include <cstdint>
#include <mutex>

#include "zs_launch.h"

static __device__ __align__(256) double g_norm_scratch[ZS_NOALLOC_NORM_MAX_SCRATCH];

namespace {

constexpr int kMaxDevices = 256;
std::mutex g_mu;
double *g_scratch_addr[kMaxDevices] = {};

// Device address of g_norm_scratch on the current device.  The name of the
// array in host code is only a host-side stand-in, never a device address.
zs_status scratch_address(double **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return zs_fail(ZS_ECUDA, "zs_grad_norm_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return zs_fail(ZS_EINVAL, "zs_grad_norm_noalloc: device %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_addr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_norm_scratch);
        if (e != cudaSuccess || !p)
            return zs_fail(ZS_ECUDA, "zs_grad_norm_noalloc: cudaGetSymbolAddress: %s",
                           cudaGetErrorString(e));
        g_scratch_addr[dev] = static_cast<double *>(p);
    }
    *out = g_scratch_addr[dev];
    return ZS_OK;
}

bool aligned(const void *p, uintptr_t a) {
    return p && (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0;
}

}  // namespace

extern "C" zs_status zs_grad_norm_noalloc(const zs_plan *P, const void *grad_shards,
                                          const void *persist_grads, float max_norm,
                                          float *d_norm, float *d_clip_coef, int32_t *d_flags,
                                          void *stream) {
    const char *fn = "zs_grad_norm_noalloc";
    if (!P) return zs_fail(ZS_EINVAL, "%s: NULL plan", fn);
    const int64_t ntiles = (int64_t)P->tiles.size();
    const int64_t need = ntiles + P->n_level1;
    if (need > ZS_NOALLOC_NORM_MAX_SCRATCH)
        return zs_fail(ZS_EINVAL,
                       "%s: the plan needs %lld doubles of norm scratch but the built-in array "
                       "holds %lld (about %lld tiles of 8192 elements); use zs_grad_norm with a "
                       "scratch buffer of norm_scratch_elems doubles",
                       fn, (long long)need, (long long)ZS_NOALLOC_NORM_MAX_SCRATCH,
                       (long long)(ZS_NOALLOC_NORM_MAX_SCRATCH - ZS_NOALLOC_NORM_MAX_SCRATCH / 4096));
    if (ntiles > 0 && !P->d_tiles)
        return zs_fail(ZS_ESTATE, "%s: plan not uploaded (call zs_plan_upload first)", fn);
    if (!aligned(d_norm, 4) || !aligned(d_clip_coef, 4) || !aligned(d_flags, 4))
        return zs_fail(ZS_EINVAL, "%s: device scalar pointers must be non-NULL and 4-byte aligned",
                       fn);
    if (P->S > 0 && !aligned(grad_shards, 16))
        return zs_fail(ZS_EINVAL, "%s: grad_shards NULL or not 16-byte aligned", fn);
    if (P->Pn_alloc > 0 && !aligned(persist_grads, 16))
        return zs_fail(ZS_EINVAL, "%s: persist_grads NULL or not 16-byte aligned", fn);
    double *scratch = nullptr;
    zs_status r = scratch_address(&scratch);
    if (r) return r;
    // every scratch element read below is written first by the same call
    // (one partial per tile, one first-level sum per block), so what an
    // earlier call left in the array does not matter
    const cudaError_t e = zsl_norm(P->d_tiles, ntiles, P->n_level1, P->cfg.dtype,
                                   static_cast<const uint16_t *>(grad_shards),
                                   static_cast<const uint16_t *>(persist_grads), scratch, true,
                                   max_norm, d_norm, d_clip_coef, d_flags, nullptr,
                                   (cudaStream_t)stream);
    if (e != cudaSuccess)
        return zs_fail(ZS_ECUDA, "%s: %s (%s)", fn, cudaGetErrorName(e), cudaGetErrorString(e));
    zs_clear_error();
    return ZS_OK;
}
