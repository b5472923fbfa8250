// Internal types of libzs shared by the host plan builder and the kernels.
#pragma once

#include <cstdint>
#include <vector>

#include "zs.h"

// Work unit of the element-wise kernels: a contiguous run of destination
// elements of one rank's shard of one parameter (or of one persistent
// parameter) inside one reduce bucket.  Every shard-space and persistent-space
// element belongs to exactly one tile, so the tiles partition the work of the
// reduce-scatter, the norm, the fused Adam pass and the partition copy.
struct ZsTile {
    int64_t dst;       // first element in shard space [N][S] (row-major) or persistent space
    int64_t src;       // element index of dst's data in the bucket's gradient buffer
    int64_t flat;      // element index in model flat space; -1: persistent tile
    int64_t win;       // element index in input space (full parameters)
    int32_t len;       // destination elements (includes padding and alignment columns)
    int32_t valid;     // leading elements that carry data; the rest are zero
    int32_t flat_len;  // leading elements that also go to model flat space
    int32_t bucket;    // reduce bucket of the tile
};
static_assert(sizeof(ZsTile) == 48, "tile layout");

constexpr int64_t ZS_TILE_ELEMS = 8192;     // destination elements per tile (before alignment)
constexpr int64_t ZS_LEVEL1_CHUNK = 4096;   // tile partial sums per first-level norm block

// Bytes of the device table: the tile records, then the reduce-scatter's
// launch order (int32 per tile), padded to 16 bytes.
inline int64_t zs_table_tile_bytes(int64_t ntiles) { return ntiles * (int64_t)sizeof(ZsTile); }
inline int64_t zs_table_bytes(int64_t ntiles) {
    return zs_table_tile_bytes(ntiles) + (ntiles * 4 + 15) / 16 * 16;
}

struct ZsParam {
    int64_t numel, ds_id, ps, pad;
    int64_t shard_off, persist_off, flat_off, input_off;
    int32_t persistent, position, sub_group, gather_bucket, first_rb, n_rb;
};

struct ZsEntry {
    int32_t param;
    int64_t e_lo, e_hi, buf_off;
};

struct ZsBucket {
    int32_t first_entry, n_entries;
    int64_t buf_elems, grad_elems, first_tile, n_tiles;
};

struct ZsGather {
    int32_t first, n;  // into zs_plan::gather_params
    int64_t flat_off, flat_elems;
};

struct ZsSubGroup {
    int32_t first, n;  // into zs_plan::order
    int64_t s_lo, s_hi, p_lo, p_hi;
};

struct zs_plan {
    zs_config cfg;
    std::vector<ZsParam> params;       // by caller index
    std::vector<int32_t> order;        // caller indices in ds_id order
    std::vector<ZsEntry> entries;
    std::vector<ZsBucket> buckets;
    std::vector<int32_t> gather_params;
    std::vector<ZsGather> gathers;
    std::vector<ZsSubGroup> sub_groups;
    std::vector<ZsTile> tiles;
    // launch order of the per-bucket reduce-scatter: launch position i
    // (numbered like the tiles) works on tile rs_order[i].  Within each
    // bucket the tiles go largest first, so that a launch does not end
    // waiting on one large tile that started late; no result depends on
    // this order.
    std::vector<int32_t> rs_order;
    int64_t S = 0, S_logical = 0, Pn_alloc = 0, Pn = 0, psi = 0, flat_elems = 0;
    int64_t padding = 0, max_buf = 0, max_gather = 0, n_level1 = 1;
    int32_t G = 1;                     // shard owners per group (N unless HSDP)
    const ZsTile *d_tiles = nullptr;   // caller memory given to zs_plan_upload
    const int32_t *d_rs_order = nullptr;   // rs_order, after the tiles in that memory
};

// Records a message for zs_last_error() and returns status.
zs_status zs_fail(zs_status status, const char *fmt, ...)
#if defined(__GNUC__)
    __attribute__((format(printf, 2, 3)))
#endif
    ;
void zs_clear_error();

// zs_all_gather_coalesced with its grid capped at max_ctas CTAs (0: no cap
// beyond the default); dependent: bulk-path launches are programmatic
// dependents of the previous kernel of the stream; fn names the caller in
// error messages.
zs_status zs_gather_impl(const zs_plan *P, int32_t n, const int32_t *params,
                         const void *param_shards, void *flat_out, int64_t flat_capacity,
                         int64_t *view_offsets, void *stream, int max_ctas, bool dependent,
                         const char *fn);
