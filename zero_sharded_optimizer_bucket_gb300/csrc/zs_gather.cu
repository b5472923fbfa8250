// A5 all_gather_coalesced: repack shard space into the flat buffer of a
// gather group ([ZeRO-3 chapter] §5.2: shards sorted by ds_id, one flat
// buffer, per-parameter views).
//
// Two paths.  When every run (rank r's shard of one parameter, landing at
// out_off + r*ps) is 16-byte aligned at both ends in both buffers, TMA bulk
// copies move the bytes (gather_bulk_kernel below).  Otherwise the SM path:
// output-centric, a thread owns a group of 8 output slots aligned to 16
// bytes in the output's address space.  When the 8 slots come from one
// rank's shard of one parameter they are one contiguous run of shard space:
// one 16-byte load (two and a lane shift when the phases differ) and one
// 16-byte store.  Slots that straddle a shard boundary are assembled one by
// one.
#include <atomic>

#include "zs_device.cuh"
#include "zs_launch.h"

namespace zsk {

__global__ void __launch_bounds__(THREADS)
gather_kernel(ZsGatherArgs a, const uint16_t *__restrict__ shards, uint16_t *__restrict__ out,
              int a0) {
    __shared__ ZsGatherEntry e[ZS_GATHER_MAX];
    for (int i = threadIdx.x; i < a.n; i += THREADS) e[i] = a.e[i];
    __syncthreads();
    const int64_t g_first = (a0 + a.out_lo) >> 3, g_last = (a0 + a.out_hi - 1) >> 3;
    for (int64_t g = g_first + (int64_t)blockIdx.x * THREADS + threadIdx.x; g <= g_last;
         g += (int64_t)gridDim.x * THREADS) {
        const int64_t f0 = 8 * g - a0;
        const int64_t fa = f0 > a.out_lo ? f0 : a.out_lo;
        int lo = 0, hi = a.n - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (e[mid].out_off <= fa) lo = mid; else hi = mid - 1;
        }
        int idx = lo;
        int64_t el = fa - e[idx].out_off;
        int64_t r = el / e[idx].ps;
        int64_t j = el - r * e[idx].ps;
        const bool full = f0 >= a.out_lo && f0 + 8 <= a.out_hi;
        if (full && j + 8 <= e[idx].ps) {
            const int64_t src = r * a.S + e[idx].shard_off + j;
            const int q = (int)(src & 7);
            const int64_t c0 = src >> 3;
            uint4 v = ldg16(shards + 8 * c0);
            if (q) v = shift8(v, ldg16(shards + 8 * c0 + 8), q);
            *reinterpret_cast<uint4 *>(out + f0) = v;
            continue;
        }
        uint32_t rv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int64_t f = f0 + i;
            rv[i] = 0u;
            if (f < a.out_lo || f >= a.out_hi) continue;
            rv[i] = shards[r * a.S + e[idx].shard_off + j];
            if (++j == e[idx].ps) {
                j = 0;
                if (++r == a.N) {
                    r = 0;
                    if (idx + 1 < a.n) ++idx;
                }
            }
        }
        if (full) {
            *reinterpret_cast<uint4 *>(out + f0) = pack8(rv);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i)
                if (f0 + i >= a.out_lo && f0 + i < a.out_hi) out[f0 + i] = (uint16_t)rv[i];
        }
    }
}

// ---------------------------------------------------------------------------
// Bulk-copy path.  When every run of the launch (rank r's shard of one
// parameter, ps elements, landing at out_off + r*ps) starts and ends on a
// 16-byte boundary in both buffers, the gather is a list of aligned memcpy
// pieces.  One thread per CTA drives the TMA engine: it loads a chunk of
// the output (BULK_CHUNK bytes, one or more pieces) from shard space into a
// shared-memory stage with cp.async.bulk, waits on the stage's mbarrier,
// and writes the chunk back to flat_out with one bulk store.  BULK_STAGES
// chunks are in flight per CTA, so a CTA per SM keeps HBM busy while the
// SMs' warps stay free for other kernels.
#ifndef ZS_BULK_STAGES
#define ZS_BULK_STAGES 3
#endif
#ifndef ZS_BULK_CHUNK
#define ZS_BULK_CHUNK 32768
#endif
constexpr int BULK_STAGES = ZS_BULK_STAGES;
constexpr int BULK_CHUNK = ZS_BULK_CHUNK;              // bytes per chunk (multiple of 16)
constexpr int64_t BULK_CHUNK_ELEMS = BULK_CHUNK / 2;
constexpr int BULK_SMEM = BULK_STAGES * BULK_CHUNK;
constexpr int BULK_SMEM_ALLOC = BULK_SMEM + 8 * BULK_STAGES;   // + mbarriers
constexpr uint64_t BULK_WAIT_NS = 1000000000ull;       // one wait gives up after 1 s

__device__ int g_bulk_wait_timeouts;                    // waits that gave up

// Issues the loads of chunk c (output elements [f, f_end)) into stage buffer
// dst, completing on mbarrier bar; returns the chunk's bytes.
__device__ uint32_t bulk_load_chunk(const ZsGatherArgs &a, const uint16_t *shards, int64_t c,
                                    uint32_t dst, uint32_t bar) {
    int64_t f = a.out_lo + c * BULK_CHUNK_ELEMS;
    const int64_t f_end = min(f + BULK_CHUNK_ELEMS, a.out_hi);
    const uint32_t bytes = (uint32_t)(2 * (f_end - f));
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :
                 : "r"(bar), "r"(bytes)
                 : "memory");
    int lo = 0, hi = a.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (a.e[mid].out_off <= f) lo = mid; else hi = mid - 1;
    }
    int idx = lo;
    int64_t r = (f - a.e[idx].out_off) / a.e[idx].ps;
    int64_t j = (f - a.e[idx].out_off) - r * a.e[idx].ps;
    uint32_t at = dst;
    while (f < f_end) {
        const int64_t len = min(f_end - f, a.e[idx].ps - j);
        const uint16_t *src = shards + r * a.S + a.e[idx].shard_off + j;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, "
            "[%3];"
            :
            : "r"(at), "l"(src), "r"((uint32_t)(2 * len)), "r"(bar)
            : "memory");
        at += (uint32_t)(2 * len);
        f += len;
        j += len;
        if (j == a.e[idx].ps) {
            j = 0;
            if (++r == a.N) {
                r = 0;
                ++idx;
            }
        }
    }
    return bytes;
}

__global__ void __launch_bounds__(32)
gather_bulk_kernel(ZsGatherArgs a, const uint16_t *__restrict__ shards, uint16_t *__restrict__ out) {
    // dynamic shared memory only: BULK_STAGES chunk buffers, then the
    // stages' mbarriers
    extern __shared__ __align__(128) uint8_t stage[];
    if (threadIdx.x != 0) return;
    // When launched as a programmatic dependent: wait until the previous
    // kernel of the stream has finished and its writes (the parameter
    // shards) are visible, then let the next gather start placing its CTAs,
    // which wait the same way; back-to-back gathers then lose the launch
    // gap.  In an ordinary launch both instructions have no effect.
    asm volatile("griddepcontrol.wait;" : : : "memory");
    asm volatile("griddepcontrol.launch_dependents;" : : : "memory");
    const uint32_t base = smem_u32(stage);
    if (base & 15) {                     // bulk copies need 16-byte aligned buffers
        atomicAdd(&g_bulk_wait_timeouts, 1);
        return;
    }
    // shared-window address of stage s's mbarrier (computed as an integer:
    // the barriers lie past the chunk buffers in the dynamic allocation)
    auto bar = [base](int64_t s) { return base + (uint32_t)(BULK_SMEM + 8 * s); };
    const int64_t n_chunks = (a.out_hi - a.out_lo + BULK_CHUNK_ELEMS - 1) / BULK_CHUNK_ELEMS;
    if ((int64_t)blockIdx.x >= n_chunks) return;
    const int64_t mine = (n_chunks - blockIdx.x + gridDim.x - 1) / gridDim.x;
    for (int s = 0; s < BULK_STAGES; ++s)
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" : : "r"(bar(s)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" : : : "memory");
    asm volatile("fence.proxy.async.shared::cta;" : : : "memory");
    uint32_t bytes[BULK_STAGES];
    const int64_t pre = mine < BULK_STAGES ? mine : BULK_STAGES;
    for (int64_t k = 0; k < pre; ++k)
        bytes[k] = bulk_load_chunk(a, shards, blockIdx.x + k * gridDim.x,
                                   base + (uint32_t)(k * BULK_CHUNK), bar(k));
    int64_t issued = pre;
    bool ok = true;
    for (int64_t k = 0; k < mine; ++k) {
        const int s = (int)(k % BULK_STAGES);
        if (!mbar_wait(bar(s), (uint32_t)((k / BULK_STAGES) & 1), BULK_WAIT_NS)) {
            ok = false;
            break;
        }
        const int64_t c = blockIdx.x + k * gridDim.x;
        uint16_t *dst = out + a.out_lo + c * BULK_CHUNK_ELEMS;
        asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                     :
                     : "l"(dst), "r"(base + (uint32_t)(s * BULK_CHUNK)), "r"(bytes[s])
                     : "memory");
        asm volatile("cp.async.bulk.commit_group;" : : : "memory");
        if (issued < mine) {
            // the stage is free again once the store has read it
            asm volatile("cp.async.bulk.wait_group.read 0;" : : : "memory");
            bytes[s] = bulk_load_chunk(a, shards, blockIdx.x + issued * gridDim.x,
                                       base + (uint32_t)(s * BULK_CHUNK), bar(s));
            ++issued;
        }
    }
    if (!ok) {
        // a wait gave up: count it and let the loads already issued land
        // (each wait again bounded) before the CTA's shared memory goes away
        atomicAdd(&g_bulk_wait_timeouts, 1);
        for (int64_t k = 0; k < issued; ++k) {
            const int s = (int)(k % BULK_STAGES);
            if (k + BULK_STAGES < issued) continue;
            mbar_wait(bar(s), (uint32_t)((k / BULK_STAGES) & 1), BULK_WAIT_NS);
        }
    }
    asm volatile("cp.async.bulk.wait_group 0;" : : : "memory");
}

// One thread waits, with the bulk gather's bounded wait, on an mbarrier
// that nothing arrives on: the wait gives up after limit_ns and counts one
// timeout, as a stuck bulk copy would.
__global__ void wait_timeout_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" : : "r"(b) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" : : : "memory");
    if (!mbar_wait(b, 0, limit_ns)) atomicAdd(&g_bulk_wait_timeouts, 1);
}

}  // namespace zsk

using namespace zsk;

namespace {

// The bulk path needs every piece 16-byte aligned at both ends, and pieces
// long enough to be worth a TMA request each.
constexpr int64_t BULK_MIN_PS = 1024;

bool bulk_ok(const ZsGatherArgs &a, const uint16_t *shards, const uint16_t *flat_out) {
    if ((reinterpret_cast<uintptr_t>(flat_out) & 15) || (reinterpret_cast<uintptr_t>(shards) & 15))
        return false;
    if (a.S % 8 || a.out_lo % 8) return false;
    int64_t next = a.out_lo;
    for (int i = 0; i < a.n; ++i) {
        const ZsGatherEntry &e = a.e[i];
        if (e.ps < BULK_MIN_PS || e.ps % 8 || e.shard_off % 8 || e.out_off != next) return false;
        next += (int64_t)a.N * e.ps;
    }
    return next == a.out_hi;
}

}  // namespace

cudaError_t zsl_gather(const ZsGatherArgs &a, const uint16_t *shards, uint16_t *flat_out,
                       cudaStream_t s, int max_ctas, bool dependent) {
    if (a.n <= 0 || a.out_hi <= a.out_lo) return cudaSuccess;
    if (bulk_ok(a, shards, flat_out)) {
        // per device: its SM count, and the kernel's shared-memory opt-in
        // per device: the kernel's shared-memory opt-in, and the default
        // grid of 8 CTAs per SM: CTAs queue behind the resident ones, which
        // measured faster than one wave of resident CTAs
        // (atomic: host threads may launch gathers at once; both set it the same)
        static std::atomic<int> wave_of[64];
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
        int wave = wave_of[dev].load(std::memory_order_relaxed);
        if (wave <= 0) {
            int sms = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(gather_bulk_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         BULK_SMEM_ALLOC);
            if (e != cudaSuccess) return e;
            wave = 8 * (sms > 0 ? sms : 152);
            wave_of[dev].store(wave, std::memory_order_relaxed);
        }
        const int64_t chunks = (a.out_hi - a.out_lo + BULK_CHUNK_ELEMS - 1) / BULK_CHUNK_ELEMS;
        const int64_t cap = max_ctas > 0 ? max_ctas : wave;
        const int64_t blocks = chunks < cap ? chunks : cap;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)blocks);
        cfg.blockDim = dim3(32);
        cfg.dynamicSmemBytes = BULK_SMEM_ALLOC;
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = dependent ? 1 : 0;
        e = cudaLaunchKernelEx(&cfg, gather_bulk_kernel, a, shards, flat_out);
        return e != cudaSuccess ? e : cudaGetLastError();
    }
    const int a0 = (int)((reinterpret_cast<uintptr_t>(flat_out) >> 1) & 7);
    const int64_t groups = ((a0 + a.out_hi - 1) >> 3) - ((a0 + a.out_lo) >> 3) + 1;
    int64_t blocks = (groups + THREADS - 1) / THREADS;
    const int64_t cap = max_ctas > 0 ? max_ctas : 152 * 8;   // 8 CTAs of 256 fill an SM
    if (blocks > cap) blocks = cap;
    gather_kernel<<<(unsigned)blocks, THREADS, 0, s>>>(a, shards, flat_out, a0);
    return cudaGetLastError();
}

cudaError_t zsl_bulk_wait_timeouts(int *count, bool reset) {
    cudaError_t e = cudaMemcpyFromSymbol(count, g_bulk_wait_timeouts, sizeof(int));
    if (e == cudaSuccess && reset) {
        const int zero = 0;
        e = cudaMemcpyToSymbol(g_bulk_wait_timeouts, &zero, sizeof(int));
    }
    return e;
}

cudaError_t zsl_wait_timeout_test(int64_t limit_ns, cudaStream_t s) {
    wait_timeout_kernel<<<1, 32, 0, s>>>((uint64_t)limit_ns);
    return cudaGetLastError();
}
