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
// address is looked up (cudaGetSymbolAddress, with that device current) on
// the first call made on a device, and again on the first call after the
// device's context was destroyed and created anew (cudaDeviceReset), when
// the module holding the array is loaded again, possibly elsewhere.  The
// cache is keyed on the context's process-unique id (cuCtxGetId), which a
// new context never shares with an old one.
#include <cuda.h>

#include <cstdint>
#include <mutex>

#include "zs_launch.h"

static __device__ __align__(256) double g_norm_scratch[ZS_NOALLOC_NORM_MAX_SCRATCH];

namespace {

constexpr int kMaxDevices = 256;
std::mutex g_mu;

struct DeviceScratch {
    unsigned long long ctx_id;  // context the address belongs to (0: none yet)
    double *addr;
};
DeviceScratch g_scratch[kMaxDevices] = {};

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long *);
CtxGetCurrentFn g_ctx_get_current = nullptr;
CtxGetIdFn g_ctx_get_id = nullptr;

// The driver's context queries, through the runtime (no link-time
// dependency on the driver library).  Called with g_mu held.
zs_status resolve_driver_entry_points() {
    if (g_ctx_get_current && g_ctx_get_id) return ZS_OK;
    cudaDriverEntryPointQueryResult q1 = cudaDriverEntryPointSymbolNotFound, q2 = q1;
    void *f1 = nullptr, *f2 = nullptr;
    const cudaError_t e1 =
        cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &f1, 12000, cudaEnableDefault, &q1);
    const cudaError_t e2 =
        cudaGetDriverEntryPointByVersion("cuCtxGetId", &f2, 12000, cudaEnableDefault, &q2);
    if (e1 != cudaSuccess || e2 != cudaSuccess || q1 != cudaDriverEntryPointSuccess ||
        q2 != cudaDriverEntryPointSuccess || !f1 || !f2)
        return zs_fail(ZS_ECUDA, "zs_grad_norm_noalloc: driver context queries unavailable (%s)",
                       cudaGetErrorString(e1 != cudaSuccess ? e1 : e2));
    g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(f1);
    g_ctx_get_id = reinterpret_cast<CtxGetIdFn>(f2);
    return ZS_OK;
}

// Device address of g_norm_scratch in the current device's current context.
// The name of the array in host code is only a host-side stand-in, never a
// device address.
zs_status scratch_address(double **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return zs_fail(ZS_ECUDA, "zs_grad_norm_noalloc: cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return zs_fail(ZS_EINVAL, "zs_grad_norm_noalloc: device %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_mu);
    zs_status r = resolve_driver_entry_points();
    if (r) return r;
    CUcontext ctx = nullptr;
    if (g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx) {
        // no context current on this thread yet: make the device's primary
        // context current (cudaSetDevice initialises it; nothing is allocated)
        e = cudaSetDevice(dev);
        if (e != cudaSuccess || g_ctx_get_current(&ctx) != CUDA_SUCCESS || !ctx)
            return zs_fail(ZS_ECUDA, "zs_grad_norm_noalloc: no CUDA context on device %d (%s)",
                           dev, cudaGetErrorString(e));
    }
    unsigned long long id = 0;
    if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS || id == 0)
        return zs_fail(ZS_ECUDA, "zs_grad_norm_noalloc: cuCtxGetId failed on device %d", dev);
    DeviceScratch &ds = g_scratch[dev];
    if (ds.ctx_id != id || !ds.addr) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_norm_scratch);
        if (e != cudaSuccess || !p)
            return zs_fail(ZS_ECUDA, "zs_grad_norm_noalloc: cudaGetSymbolAddress: %s",
                           cudaGetErrorString(e));
        ds.addr = static_cast<double *>(p);
        ds.ctx_id = id;
    }
    *out = ds.addr;
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
