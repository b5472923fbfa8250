// A5 all_gather_coalesced: repack shard space into the flat buffer of a
// gather group ([ZeRO-3 chapter] §5.2: shards sorted by ds_id, one flat
// buffer, per-parameter views).
//
// Output-centric: a thread owns 8 output slots aligned to 16 bytes in the
// output's address space.  When the 8 slots come from one rank's shard of
// one parameter they are one contiguous run of shard space: one 16-byte
// load (two and a lane shift when the phases differ) and one 16-byte store.
// Slots that straddle a shard boundary are assembled one by one.
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

}  // namespace zsk

using namespace zsk;

cudaError_t zsl_gather(const ZsGatherArgs &a, const uint16_t *shards, uint16_t *flat_out,
                       cudaStream_t s, int max_ctas) {
    if (a.n <= 0 || a.out_hi <= a.out_lo) return cudaSuccess;
    const int a0 = (int)((reinterpret_cast<uintptr_t>(flat_out) >> 1) & 7);
    const int64_t groups = ((a0 + a.out_hi - 1) >> 3) - ((a0 + a.out_lo) >> 3) + 1;
    int64_t blocks = (groups + THREADS - 1) / THREADS;
    const int64_t cap = max_ctas > 0 ? max_ctas : 152 * 8;
    if (blocks > cap) blocks = cap;
    gather_kernel<<<(unsigned)blocks, THREADS, 0, s>>>(a, shards, flat_out, a0);
    return cudaGetLastError();
}
