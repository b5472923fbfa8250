/*
 * zs.h — C ABI of libzs: the ZeRO-3 per-step shard data path on one GPU.
 *
 * N data-parallel ranks are *virtual*: all of their buffers live in the HBM
 * of one GPU, and the collectives of the method (reduce-scatter of the
 * gradient buckets, the scalar all-reduce of the gradient norm, the
 * coalesced all-gather of the parameters) are kernels over those buffers.
 *
 * Sources (page title, then the section on it):
 *   [ZeRO-3 chapter] "03 · ZeRO-3：参数分片与 all-gather 调度"
 *   [Grok blog]      "DeepSpeed ZeRO Stage 3：参数分区，让大模型训练“零负担”"
 *   [Core flow]      "ZeRO-3 核心流程：把参数也切开的那一档"
 *
 * Conventions
 * -----------
 * - Every entry point returns a zs_status; ZS_OK is 0.  Argument errors are
 *   found on the host, return ZS_EINVAL and enqueue nothing.  A CUDA error
 *   returns ZS_ECUDA.  No call aborts or exits; zs_last_error() gives a
 *   message for the calling thread.
 * - Device buffers are owned by the caller; the library allocates no device
 *   memory (its only device memory is static: the scratch array of
 *   zs_grad_norm_noalloc and a counter of timed-out waits).  The plan is
 *   host memory owned by the library (zs_free_plan).
 * - Device work is enqueued on the caller's cudaStream_t (passed as void*,
 *   NULL = legacy default stream).  No call synchronises the host with the
 *   device; results such as the gradient norm stay in device memory.
 * - bf16 buffers hold IEEE bfloat16 bit patterns (2 bytes per element).
 * - Device buffers read or written with 16-byte vectors must be 16-byte
 *   aligned: every buffer except the flat output of the gathers, which needs
 *   only 2-byte alignment.  Misalignment is ZS_EINVAL.
 * - CUDA graphs: the device calls only enqueue work on the given stream
 *   (no host synchronisation, no allocation), so a sequence of them can be
 *   captured and replayed; scalars such as the Adam step count and the
 *   hyper-parameters are captured by value (re-capture, or update the
 *   kernel nodes, to advance them).
 * - Host threads: a plan is read-only once uploaded (zs_plan_upload), so
 *   calls on one plan may come from several threads; a scheduler (zs_sched)
 *   holds mutable state and must be used by one thread at a time.
 * - Distinct buffers of a call must not overlap (rank gradients, gradient
 *   shards, parameter shards, each state buffer, the persistent buffers, the
 *   flat output, scratch); a buffer the call updates in place (the fp32
 *   master and moments) is one buffer, read and written.  Overlapping
 *   buffers give undefined results and are not detected.
 *
 * Layouts (elements; "ds_id order" = parameters sorted by ds_id)
 * --------------------------------------------------------------
 * ps_p      = ceil(numel_p / N): rank r owns flat elements
 *             [r*ps_p, (r+1)*ps_p) of parameter p, zero beyond numel_p
 *             ([ZeRO-3 chapter] §3.1, item 1).
 * persistent: numel_p < param_persistence_threshold; never partitioned
 *             ([ZeRO-3 chapter] §5.3, last paragraph).
 * shard space      [N][S]: row r holds rank r's shards of all partitioned
 *             parameters; p at columns [S_p, S_p+ps_p), S_p = running sum
 *             of ps rounded up to a multiple of 8.  Gradient shards, 16-bit
 *             parameter shards and the fp32 master / exp_avg / exp_avg_sq
 *             shards all use it ([ZeRO-3 chapter] §6.1: one flat buffer of
 *             gradient partitions, fp32 partitions per rank).
 * persistent space [Pn]: persistent parameters whole, once, at P_p =
 *             running sum of numel rounded up to 8.
 * model flat space: partitioned parameters gathered, back to back in ds_id
 *             order, each its N shards in rank order (N*ps_p elements, the
 *             first numel_p of which are the parameter), at F_p = running
 *             sum of N*ps ([ZeRO-3 chapter] §5.2, all_gather_coalesced).
 * input space: all parameters whole, back to back in ds_id order at W_p =
 *             running sum of numel (the weights handed to zs_partition).
 * reduce bucket buffer: one per rank and bucket; the bucket's entries
 *             (a parameter, or a chunk [c*B,(c+1)*B) of a parameter larger
 *             than B = reduce_bucket_size) back to back, each starting at a
 *             multiple of 8; buf_elems (zs_bucket_info_t) elements, a multiple
 *             of 8.  Rank k's buffer holds rank k's gradient (bf16).
 */
#ifndef ZS_H
#define ZS_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t zs_status;
#define ZS_OK        0
#define ZS_EINVAL   (-1)   /* bad argument: nothing was enqueued            */
#define ZS_ENOMEM   (-2)   /* host allocation failed                        */
#define ZS_ECUDA    (-3)   /* a CUDA call failed (message names it)         */
#define ZS_ESTATE   (-4)   /* call out of order (e.g. plan not uploaded)    */
#define ZS_ETIMEOUT (-5)   /* a bounded device wait gave up (reported by
                              zs_device_wait_timeouts)                     */

/* Largest N the per-bucket reduce-scatter accepts (its rank pointers travel
 * as kernel arguments). */
#define ZS_MAX_RANKS 256

/* 16-bit storage of gradients and parameters (zs_config.dtype): IEEE
 * bfloat16, or IEEE binary16 for fp16 mixed precision with a loss scale
 * ([Core flow] §1 table stores parameters and gradients in fp16).  All
 * arithmetic is float32 either way; the dtype changes only the conversions
 * (round to nearest even; an fp16 overflow becomes inf). */
#define ZS_DTYPE_BF16 0
#define ZS_DTYPE_FP16 1

/* Bits of the device flag word written by zs_grad_norm / zs_shard_step. */
#define ZS_SKIP_NONFINITE 1   /* gradient norm not finite: update skipped */

typedef struct zs_plan zs_plan;   /* opaque, host memory */

/* Defaults: the DeepSpeed ZeRO-3 values quoted on the pages —
 * stage3_param_persistence_threshold 1e5, reduce_bucket_size 5e6,
 * stage3_prefetch_bucket_size 5e7 ([Core flow] §4 config block;
 * [ZeRO-3 chapter] §5.2, §5.3), sub_group_size 1e9 ([ZeRO-3 chapter] §6.1,
 * counted in per-rank shard elements). */
typedef struct {
    int32_t n_ranks;                      /* N >= 1                              */
    int32_t dtype;                        /* ZS_DTYPE_BF16 (default) or FP16     */
    int64_t param_persistence_threshold;  /* persistent iff numel < threshold    */
    int64_t reduce_bucket_size;           /* elements, >= 1                      */
    int64_t prefetch_bucket_size;         /* elements, >= 1 (gather buckets)     */
    int64_t sub_group_size;               /* per-rank elements, >= 1             */
    /* HSDP ([Core flow] §4: FSDP inside a group, DDP across groups): the N
     * ranks form N/G replica groups of G consecutive ranks; parameters are
     * partitioned over the G ranks of a group (every layout below then uses
     * G where it says N) and the groups hold identical replicas, stored
     * once.  The gradient mean sums each group's ranks in rank order, then
     * the group sums in group order, and divides by N.  0 or N: plain ZeRO-3
     * (bit-identical to it).  Must divide N. */
    int32_t shard_group_size;
    int32_t reserved;                     /* must be 0                           */
} zs_config;

typedef struct {
    float   lr, beta1, beta2, eps, weight_decay;
    int32_t adamw;            /* 1: decoupled decay (AdamW); 0: L2 into the gradient */
    int32_t bias_correction;  /* 1: divide the moments by 1-beta^t                   */
} zs_adam_hparams;

typedef struct {
    int32_t n_ranks, n_params;
    int32_t n_reduce_buckets, n_gather_buckets;
    int32_t n_sub_groups, dtype;
    int32_t shard_group_size, reserved;   /* G (N unless HSDP)                      */
    int64_t psi;                    /* sum of numel                                   */
    int64_t shard_elems;            /* S: length of one shard row (multiple of 8)     */
    int64_t shard_elems_logical;    /* sum of ps over partitioned parameters          */
    int64_t persist_elems;          /* length of persistent space (multiple of 8)     */
    int64_t persist_elems_logical;  /* sum of numel over persistent parameters        */
    int64_t flat_elems;             /* length of model flat space                     */
    int64_t padding_elems;          /* sum of N*ps - numel                            */
    int64_t max_bucket_buf_elems;   /* largest reduce bucket buffer                   */
    int64_t max_gather_elems;       /* largest gather bucket                          */
    int64_t bytes_per_rank;         /* 16*(shard_elems_logical + persist_elems_logical) */
    int64_t n_tiles;                /* work tiles of the kernels                      */
    int64_t device_table_bytes;     /* device memory zs_plan_upload needs             */
    int64_t norm_scratch_elems;     /* doubles of norm scratch the calls need         */
} zs_plan_info_t;

typedef struct {
    int64_t numel, ds_id;
    int64_t partition_size;   /* ps (0 for persistent)                  */
    int64_t padding;          /* N*ps - numel (0 for persistent)        */
    int64_t shard_offset;     /* S_p, or -1 for persistent              */
    int64_t persist_offset;   /* P_p, or -1 for partitioned             */
    int64_t flat_offset;      /* F_p, or -1 for persistent              */
    int64_t input_offset;     /* W_p                                    */
    int32_t persistent;
    int32_t position;         /* rank of the parameter in ds_id order   */
    int32_t sub_group;
    int32_t gather_bucket;    /* -1 for persistent                      */
    int32_t first_reduce_bucket;
    int32_t n_reduce_buckets; /* > 1 when the parameter is split in chunks */
} zs_param_info_t;

typedef struct {
    int32_t n_entries, reserved;
    int64_t buf_elems;        /* elements of each rank's buffer (multiple of 8) */
    int64_t grad_elems;       /* gradient elements the bucket carries           */
    int64_t first_tile, n_tiles;
} zs_bucket_info_t;

typedef struct {
    int32_t n_params, reserved;
    int64_t flat_offset;      /* of the bucket in model flat space */
    int64_t flat_elems;
} zs_gather_bucket_info_t;

typedef struct {
    int32_t n_params, reserved;
    int64_t shard_lo, shard_hi;       /* shard-space columns of the sub-group */
    int64_t persist_lo, persist_hi;   /* persistent-space range               */
} zs_sub_group_info_t;

/* Device pointers of the per-rank optimizer state and 16-bit buffers, all in
 * the layouts above ([ZeRO-3 chapter] §6.1: per-rank fp32 partitions, the
 * flat gradient-partition buffer; [Core flow] §1: 2 + 2 + 12 bytes per
 * element).  Shard arrays have N*S elements, persistent arrays Pn. */
typedef struct {
    void  *grad_shards;      /* bf16 [N][S]  reduced gradients            */
    void  *param_shards;     /* bf16 [N][S]  16-bit parameter shards      */
    float *master;           /* fp32 [N][S]                               */
    float *exp_avg;          /* fp32 [N][S]                               */
    float *exp_avg_sq;       /* fp32 [N][S]                               */
    void  *persist_grads;    /* bf16 [Pn]                                 */
    void  *persist_params;   /* bf16 [Pn]                                 */
    float *p_master;         /* fp32 [Pn]                                 */
    float *p_exp_avg;        /* fp32 [Pn]                                 */
    float *p_exp_avg_sq;     /* fp32 [Pn]                                 */
} zs_shard_state;

/* Message of the last failed call on this thread ("" if none). */
const char *zs_last_error(void);

/* Library version string. */
const char *zs_version(void);

/* Fill *cfg with the defaults above for n_ranks ranks. */
void zs_default_config(zs_config *cfg, int32_t n_ranks);

/* A1 — build the partition plan ([ZeRO-3 chapter] §3.1 partition range,
 * §5.3 persistence, §6.1 sub-groups, §6.2 reduce buckets, §5.2 gather
 * buckets).  numel[n_params] (>= 0), ds_id[n_params] unique or NULL for
 * index order.  Host only: no device call.  *out receives a plan owned by
 * the caller until zs_free_plan.  n_params == 0 gives an empty plan.
 * Errors: ZS_EINVAL (bad config, negative numel, duplicate ds_id),
 * ZS_ENOMEM. */
zs_status zs_build_partition(const zs_config *cfg, int32_t n_params, const int64_t *numel,
                             const int64_t *ds_id, zs_plan **out);

/* Release a plan (NULL is a no-op).  Device memory given to zs_plan_upload
 * stays the caller's. */
void zs_free_plan(zs_plan *plan);

/* Plan queries (host only).  Index arguments out of range: ZS_EINVAL. */
zs_status zs_plan_info(const zs_plan *plan, zs_plan_info_t *out);
zs_status zs_param_info(const zs_plan *plan, int32_t param, zs_param_info_t *out);
zs_status zs_param_at(const zs_plan *plan, int32_t position, int32_t *param);
zs_status zs_bucket_info(const zs_plan *plan, int32_t bucket, zs_bucket_info_t *out);
zs_status zs_bucket_entry(const zs_plan *plan, int32_t bucket, int32_t entry, int32_t *param,
                          int64_t *elem_lo, int64_t *elem_hi, int64_t *buf_offset);
zs_status zs_gather_bucket_info(const zs_plan *plan, int32_t gather_bucket,
                                zs_gather_bucket_info_t *out);
zs_status zs_gather_bucket_param(const zs_plan *plan, int32_t gather_bucket, int32_t i,
                                 int32_t *param);
zs_status zs_sub_group_info(const zs_plan *plan, int32_t sub_group, zs_sub_group_info_t *out);

/* Host copy of the plan's work table (the bytes zs_plan_upload sends to the
 * device), for inspection and tests.  The table is an array of n_tiles
 * records of 48 bytes: int64 dst, src, flat, win; int32 len, valid,
 * flat_len, bucket.  A tile is a run of `len` destination elements starting
 * at `dst` in shard space (row-major [N][S]) or, when flat < 0, in
 * persistent space; its first `valid` elements take their data from
 * element `src` on of the bucket `bucket`'s gradient buffers and from
 * element `win` on of input space; the rest are zero padding; its first
 * flat_len elements also go to model flat space from element `flat` on.
 * When bytes >= device_table_bytes the rest of the device table follows:
 * n_tiles int32, the launch order of zs_reduce_scatter (launch position
 * i, in tile numbering, works on tile order[i]; within each bucket a
 * permutation of the bucket's tiles, most valid elements first, then
 * longest, then table order, so that a bucket's launch does not end on a
 * large tile that started late).  Errors: ZS_EINVAL (bytes < 48 * n_tiles). */
zs_status zs_plan_table(const zs_plan *plan, void *host_out, int64_t bytes);

/* Copy the plan's work tables to device memory owned by the caller
 * (d_table: 16-byte aligned, >= device_table_bytes).  Enqueued on stream;
 * the plan keeps d_table and uses it in every later device call, so it must
 * stay allocated while the plan is used, and only this call may write it
 * (zs_reduce_scatter reads it before waiting for the previous kernel of
 * the stream).  Calling it again moves the plan to the new buffer.
 * Errors: ZS_EINVAL, ZS_ECUDA. */
zs_status zs_plan_upload(zs_plan *plan, void *d_table, int64_t bytes, void *stream);

/* A1 data movement — partition full fp32 parameters (input space,
 * input_elems = psi floats, 16-byte aligned) into every rank's fp32 master
 * shard and bf16 parameter shard, zero padding, and the persistent
 * parameters into persistent space; exp_avg and exp_avg_sq are zeroed
 * ([ZeRO-3 chapter] §3.1: _partition_param copies the rank's range into
 * ds_tensor; §6.1: _create_fp32_partitions).  grad buffers of st are not
 * touched (may be NULL).  Errors: ZS_EINVAL, ZS_ESTATE (not uploaded),
 * ZS_ECUDA. */
zs_status zs_partition(const zs_plan *plan, const float *full_params, const zs_shard_state *st,
                       void *stream);

/* A2 — reduce-scatter one bucket ([ZeRO-3 chapter] §6.2: a full IPG bucket
 * is all-reduced and each rank keeps its range, or reduce-scattered to the
 * owners; [Grok blog] §3: sum, average, scatter).  For every element
 * (r, S_p+j) of the bucket: s = 0; for k = 0..N-1 s += float(g_k[e]) in
 * that order (0 for e >= numel); grad_shards[r][S_p+j] = bf16_rne(s / N).
 * Persistent entries write persist_grads the same way on the full range.
 * rank_grads: HOST array of N device pointers (16-byte aligned, >=
 * buf_elems elements each; buffers that start on 128-byte boundaries, as
 * separate allocations do, are read a line at a time).  If norm_scratch is
 * not NULL (>= norm_scratch_elems doubles), the bucket's tiles also write
 * their sums of squared results there for zs_grad_norm.  The launch keeps
 * stream order: it waits for the previous kernel of the stream before
 * reading rank_grads or writing anything, so back-to-back calls each leave
 * the GPU partly idle while the previous bucket drains;
 * zs_reduce_scatter_range takes several ready buckets in one launch.
 * While it waits it may already have the start of its slice of every rank
 * buffer fetched into L2, which changes no value it reads.  Errors: ZS_EINVAL (bucket out of range,
 * N > ZS_MAX_RANKS, NULL or misaligned pointer), ZS_ESTATE, ZS_ECUDA. */
zs_status zs_reduce_scatter(const zs_plan *plan, int32_t bucket, const void *const *rank_grads,
                            void *grad_shards, void *persist_grads, double *norm_scratch,
                            void *stream);

/* A3 — global gradient norm and clip coefficient ([ZeRO-3 chapter] §6.3:
 * unscale_and_clip_grads(sub_group_id, global_norm); [Core flow] 坑 1: the
 * norm must cover all shards, each rank alone would clip differently).
 * norm = sqrt(sum of squares of every shard element and every persistent
 * element); coef = min(1, max_norm / (norm + 1e-6)) in fp32, 1 when
 * max_norm <= 0 or when the norm is not finite.  The sum of squares is
 * accumulated without rounding error up to about 2^-46 relative (squares
 * of 16-bit values are exact in fp32, each addition's error is carried in
 * a float32 pair, the per-tile sums and above are float64), then
 * norm = float32(sqrt(sum)) as with an exactly rounded sum, so the norm
 * and the coefficient have the bits of the exact definition except when
 * the root lies within that error of a float32 rounding boundary.
 * recompute = 0 uses the per-tile sums that zs_reduce_scatter left in
 * norm_scratch (every bucket must have been reduced with it since);
 * recompute = 1 first recomputes them from grad_shards / persist_grads,
 * with the same bits.  Writes device scalars d_norm,
 * d_clip_coef and the flag word d_flags (ZS_SKIP_NONFINITE).  Errors:
 * ZS_EINVAL, ZS_ESTATE, ZS_ECUDA. */
zs_status zs_grad_norm(const zs_plan *plan, const void *grad_shards, const void *persist_grads,
                       double *norm_scratch, int32_t recompute, float max_norm, float *d_norm,
                       float *d_clip_coef, int32_t *d_flags, void *stream);

/* Dynamic loss scale for fp16 gradients, kept in device memory so that no
 * host synchronisation is needed.  d_scale holds the scale S the caller
 * multiplied the loss by for this step; d_good_steps the number of steps
 * since the last overflow.  After the norm: on an overflow (non-finite
 * norm) S = max(S / scale_factor, min_scale) and the count restarts; after
 * scale_window consecutive good steps S = S * scale_factor (float32).  The
 * pages name the unscale step only ([ZeRO-3 chapter] §6.3,
 * unscale_and_clip_grads); this schedule is DeepSpeed's dynamic loss
 * scaler without hysteresis.  d_good_steps may be NULL when
 * scale_window <= 0: the scale is then static (read, never changed). */
typedef struct {
    float   *d_scale;        /* device, in/out                               */
    int32_t *d_good_steps;   /* device, in/out (NULL: static scale)          */
    float    scale_factor;   /* > 1, e.g. 2                                  */
    float    min_scale;      /* > 0, e.g. 1                                  */
    int32_t  scale_window;   /* e.g. 1000; <= 0: static scale                */
    int32_t  reserved;       /* must be 0                                    */
} zs_loss_scaler;

/* A3 with a loss scale — unscale_and_clip_grads ([ZeRO-3 chapter] §6.3):
 * the stored (reduced) gradients are the gradients of the loss times S.
 * norm = float32(sqrt(sum of squares)) / S, the norm of the true gradients,
 * written to d_norm; clip = min(1, max_norm / (norm + 1e-6)) (1 when
 * max_norm <= 0); d_clip_coef = clip / S, the factor zs_adam_step and
 * zs_adam_gather apply to the stored gradients; a non-finite norm (an
 * overflow) sets ZS_SKIP_NONFINITE and reports coef 1.  Then the scaler is
 * updated as described at zs_loss_scaler.  With S = 1 and a static scale
 * this is zs_grad_norm exactly.  Other arguments as zs_grad_norm.  Errors:
 * ZS_EINVAL (NULL scaler or d_scale, bad factor / min_scale, reserved != 0),
 * ZS_ESTATE, ZS_ECUDA. */
zs_status zs_unscale_and_clip(const zs_plan *plan, const void *grad_shards,
                              const void *persist_grads, double *norm_scratch, int32_t recompute,
                              float max_norm, const zs_loss_scaler *scaler, float *d_norm,
                              float *d_clip_coef, int32_t *d_flags, void *stream);

/* Size, in doubles, of the norm scratch array built into the library for
 * zs_grad_norm_noalloc (8 MiB of device memory per GPU that loads it). */
#define ZS_NOALLOC_NORM_MAX_SCRATCH (1LL << 20)

/* zs_grad_norm with recompute = 1, for callers that cannot allocate device
 * memory.  The pages have no counterpart: this exists for callers that are
 * handed only their inputs and outputs (a plugin inside a host framework
 * that owns every device allocation) or that must keep cudaMalloc, which
 * can synchronise the device, out of their step loop.  The scratch lives in
 * an array of ZS_NOALLOC_NORM_MAX_SCRATCH doubles inside the library;
 * nothing is allocated.  Same inputs and outputs as zs_grad_norm (the
 * reduced gradients, max_norm, device scalars d_norm, d_clip_coef,
 * d_flags); the result equals zs_grad_norm(..., recompute = 1, ...) bit for
 * bit.
 * - The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress, with that device current); make that first call
 *   before any stream capture.  The address is kept per device and per
 *   CUDA context: after the device's context is destroyed and created again
 *   (cudaDeviceReset), the next call looks it up again, so that call too
 *   should come before any capture.
 * - Every call on a device shares the one array and it keeps the last
 *   call's contents; each call writes every element it reads, so nothing
 *   needs clearing.  Calls that overlap on the GPU (other streams, other
 *   host threads) race on the array and give wrong norms.
 * - Errors: ZS_EINVAL when the plan needs more than
 *   ZS_NOALLOC_NORM_MAX_SCRATCH doubles (n_tiles + first-level blocks, i.e.
 *   about 8.6e9 elements) or on a bad pointer, ZS_ESTATE when the plan is
 *   not uploaded, ZS_ECUDA. */
zs_status zs_grad_norm_noalloc(const zs_plan *plan, const void *grad_shards,
                               const void *persist_grads, float max_norm, float *d_norm,
                               float *d_clip_coef, int32_t *d_flags, void *stream);

/* A4 — Adam(W) on one sub-group (-1: all) of every rank's fp32 shard and
 * of its persistent parameters, then the bf16 cast of the new master into
 * param_shards / persist_params ([ZeRO-3 chapter] §6.3: per sub-group
 * clip, optimizer step on the rank's fp32 partition, write back the 16-bit
 * shard; §6.1 sub_group_size).  In fp32, per element, in this order:
 *   g = float(grad) * coef
 *   AdamW: p = p - (lr*wd)*p        |  Adam-L2: g = g + wd*p
 *   m = b1*m + (1-b1)*g;  v = b2*v + (1-b2)*(g*g)
 *   p = p - lr * ((m/bc1) / (sqrt(v/bc2) + eps));  param = bf16_rne(p)
 * with 1-b, lr*wd, bc = 1-b^t computed in double on the host and rounded to
 * fp32 (bc = 1 without bias correction).  step t >= 1 is the caller's
 * counter.  d_clip_coef / d_flags are device scalars from zs_grad_norm;
 * when d_flags has ZS_SKIP_NONFINITE set nothing is written.  Errors:
 * ZS_EINVAL (sub_group out of range, step < 1, bad pointer), ZS_ECUDA. */
zs_status zs_adam_step(const zs_plan *plan, int32_t sub_group, const zs_adam_hparams *hp,
                       int64_t step, const float *d_clip_coef, const int32_t *d_flags,
                       const zs_shard_state *st, void *stream);

/* A5 — all_gather_coalesced ([ZeRO-3 chapter] §5.2: sort the group by
 * ds_id, pack one flat buffer, one collective, per-parameter views; §7:
 * a wrong order is silently wrong).  params[n]: parameter indices in any
 * order, no duplicates.  Partitioned parameters are laid out in ds_id
 * order, each as its N shards in rank order (N*ps elements, the first
 * numel of which are the parameter); flat_out (2-byte aligned) receives
 * them; view_offsets (HOST, n entries) receives each listed parameter's
 * offset in flat_out, -1 for a persistent parameter (already whole, not
 * gathered).  flat_capacity: elements available at flat_out.  The bytes
 * equal what each of the N ranks would receive.  Errors: ZS_EINVAL
 * (index out of range, duplicate, capacity too small), ZS_ESTATE,
 * ZS_ECUDA. */
zs_status zs_all_gather_coalesced(const zs_plan *plan, int32_t n, const int32_t *params,
                                  const void *param_shards, void *flat_out,
                                  int64_t flat_capacity, int64_t *view_offsets, void *stream);

/* Bounded waits that gave up, counted on the current device since the last
 * reset.  A gather whose runs are all 16-byte aligned (flat_out 16-byte
 * aligned, every partition_size a multiple of 8 and at least 1024) moves
 * its bytes with TMA bulk copies through shared memory, one mbarrier wait
 * per chunk; a wait that does not complete within a bound (about a second)
 * is abandoned, the gather's output is then incomplete, and this counter
 * goes up.  Synchronous (reads device memory).  reset != 0 sets it back to
 * 0.  Returns ZS_ETIMEOUT, with *count filled, when the count is not 0.
 * Has no counterpart in the pages: it is this library's report of its own
 * bounded waits.  Errors: ZS_EINVAL (NULL count), ZS_ECUDA. */
zs_status zs_device_wait_timeouts(int32_t *count, int32_t reset);

/* Test hook for the timeout path: enqueues one thread that waits, with the
 * bulk gather's bounded wait but a limit of limit_ns nanoseconds (0 <
 * limit_ns <= 2e9), on an mbarrier that nothing arrives on.  The wait gives
 * up, the count of zs_device_wait_timeouts goes up by one, and the CUDA
 * context stays usable: nothing faults, traps or spins without bound.  Has
 * no counterpart in the pages.  Errors: ZS_EINVAL (limit), ZS_ECUDA. */
zs_status zs_test_wait_timeout(int64_t limit_ns, void *stream);

/* A2 over the consecutive buckets [first_bucket, first_bucket + n_buckets)
 * in one launch, for buckets that become ready back to back ([ZeRO-3
 * chapter] §6.2: a full IPG bucket is reduced and scattered; when several
 * fill at once, as at the end of the backward pass, one launch takes them
 * all).  Same result as zs_reduce_scatter on each of those buckets in turn.
 * Separate zs_reduce_scatter calls keep stream order: each waits for the
 * kernel before it to finish, which leaves the GPU partly idle while the
 * previous bucket's last tiles drain; a range has no such gap inside it.
 * d_rank_grads: DEVICE array [n_buckets][N] of device pointers (rank k's
 * buffer of bucket first_bucket + i at [i*N + k]; 16-byte aligned; a NULL
 * or misaligned entry is not read and makes that tile's norm partial NaN).
 * norm_scratch (NULL, or >= norm_scratch_elems doubles) receives the
 * tiles' partial sums.  n_buckets = 0 enqueues nothing.  Errors: ZS_EINVAL
 * (range outside the plan, pointers), ZS_ESTATE, ZS_ECUDA. */
zs_status zs_reduce_scatter_range(const zs_plan *plan, int32_t first_bucket, int32_t n_buckets,
                                  const void *const *d_rank_grads, void *grad_shards,
                                  void *persist_grads, double *norm_scratch, void *stream);

/* A2 over every bucket in one launch — the first pass of zs_shard_step.
 * Same result as zs_reduce_scatter on each bucket in turn.  d_rank_grads
 * as in zs_shard_step; norm_scratch (>= norm_scratch_elems doubles) receives
 * every tile's partial sum.  Errors: ZS_EINVAL, ZS_ESTATE, ZS_ECUDA. */
zs_status zs_reduce_scatter_all(const zs_plan *plan, const void *const *d_rank_grads,
                                void *grad_shards, void *persist_grads, double *norm_scratch,
                                void *stream);

/* A4 + A5 in one launch — the second pass of zs_shard_step: Adam(W) and the
 * bf16 cast of every element (all sub-groups), and each new bf16 parameter
 * also written at its place in model flat space (flat_out, flat_elems,
 * 2-byte aligned), as zs_all_gather_coalesced of every gather bucket would.
 * Same arguments and skip rule as zs_adam_step.
 * ZeRO-1/2 residency ([Core flow] §4 table: stages 1 and 2 keep the full
 * parameters on every rank; [ZeRO-3 chapter] §1): st->param_shards may be
 * NULL, and then the new parameters are written only to flat_out, the full
 * replica (a rank's shard is a slice of it), saving the shard write;
 * zs_shard_step and zs_shard_step_scaled accept the same.  ZeRO-1's
 * gradient all-reduce is zs_reduce_scatter followed by
 * zs_all_gather_coalesced over grad_shards.  Errors: ZS_EINVAL, ZS_ESTATE,
 * ZS_ECUDA. */
zs_status zs_adam_gather(const zs_plan *plan, const zs_adam_hparams *hp, int64_t step,
                         const float *d_clip_coef, const int32_t *d_flags,
                         const zs_shard_state *st, void *flat_out, void *stream);

/* A6 — the fused step: reduce-scatter of every bucket with the norm partial
 * sums (one launch over all tiles), the norm / clip finish, then Adam(W),
 * the bf16 cast and the write of the gathered parameters into model flat
 * space (one launch over all tiles).  Results are bit-identical to
 * zs_reduce_scatter (every bucket, with norm_scratch) -> zs_grad_norm
 * (recompute 0) -> zs_adam_step(-1) -> zs_all_gather_coalesced of every
 * gather bucket into its place in model flat space.
 * d_rank_grads: DEVICE array [n_reduce_buckets][N] of device pointers
 * (rank k's buffer of bucket b at [b*N + k]; 16-byte aligned; a NULL or
 * misaligned entry is not read and makes the norm NaN, so the update is
 * skipped).  flat_out: model flat space (flat_elems, 2-byte aligned).
 * Errors: ZS_EINVAL, ZS_ESTATE, ZS_ECUDA. */
zs_status zs_shard_step(const zs_plan *plan, const void *const *d_rank_grads,
                        const zs_shard_state *st, double *norm_scratch,
                        const zs_adam_hparams *hp, int64_t step, float max_norm,
                        float *d_norm, float *d_clip_coef, int32_t *d_flags,
                        void *flat_out, void *stream);

/* A6 with a loss scale: zs_reduce_scatter_all -> zs_unscale_and_clip
 * (recompute 0) -> zs_adam_gather, for fp16 plans (any plan works).  Same
 * arguments as zs_shard_step plus the scaler.  Errors as zs_shard_step. */
zs_status zs_shard_step_scaled(const zs_plan *plan, const void *const *d_rank_grads,
                               const zs_shard_state *st, double *norm_scratch,
                               const zs_adam_hparams *hp, int64_t step, float max_norm,
                               const zs_loss_scaler *scaler, float *d_norm, float *d_clip_coef,
                               int32_t *d_flags, void *flat_out, void *stream);

/* ------------------------------------------------------------------------
 * Gather scheduler — the forward / backward fetch and release of gathered
 * parameters ([ZeRO-3 chapter] §5.1-5.3 PartitionedParameterCoordinator:
 * trace, fetch_sub_module, release_sub_module; §7: an order change
 * invalidates the trace).  A model is given as modules, each a list of
 * parameter indices.  Each pass calls, per module in execution order,
 * zs_sched_fetch (gathers what is missing, prefetches ahead along the
 * recorded trace, makes the compute stream wait), then the caller's compute
 * on the compute stream, then zs_sched_release.  zs_sched_end_pass releases
 * everything (the optimizer step repartitions all parameters, §6.3).
 * Rules:
 * - the first pass records the module order; later passes prefetch from it;
 *   a fetch that differs from the recorded order stops prefetching for the
 *   pass and the next pass records again;
 * - prefetch walks the trace's parameter uses after the current module,
 *   skipping available / in-flight / persistent parameters, while the
 *   elements added stay below min(prefetch_bucket_size,
 *   max_live_parameters - live elements), one coalesced gather per module
 *   reached (a compute then waits only for its own module's gather);
 * - release keeps a parameter whose next use in the trace is within
 *   max_reuse_distance elements of parameter uses;
 * - gathers go to the caller's arena (bf16/fp16, arena_elems elements):
 *   one contiguous block per gather, placed where the latest release of
 *   the free space it covers is oldest (never used first, then lowest
 *   offset), laid out as
 *   zs_all_gather_coalesced lays them; a gather reusing released space waits
 *   on the compute stream's release event.  Size the arena for the live
 *   budget (max_live_parameters, padded to G*ps per parameter) plus what the
 *   reuse distance keeps plus the largest module, with slack for first-fit
 *   fragmentation; a fetch that does not fit fails with ZS_ENOMEM.
 * Gathers are enqueued on the gather stream, which the compute stream waits
 * on through CUDA events; neither call blocks the host.  The first fetch of
 * a pass also makes the gather stream wait for everything enqueued on the
 * compute stream before it, so that gathers read shards rewritten between
 * passes (the optimizer step; [ZeRO-3 chapter] §6.3) on that stream.  A
 * scheduler uses one compute stream and one gather stream, fixed by its
 * first fetch; a call with other streams fails with ZS_EINVAL. */
typedef struct zs_sched zs_sched;   /* opaque, host memory + CUDA events */

typedef struct {
    int64_t prefetch_bucket_size;   /* elements, e.g. 5e7                     */
    int64_t max_live_parameters;    /* elements gathered at once, e.g. 1e9    */
    int64_t max_reuse_distance;     /* elements, e.g. 1e9                     */
    int64_t arena_elems;            /* capacity of the arena                  */
    int64_t gather_ctas;            /* CTAs per gather launch, 0..2^20: 0 lets
                                       a gather take the whole GPU (its CTAs
                                       queued behind one another then delay
                                       the compute stream's kernels); a cap
                                       (e.g. 152, one per SM) leaves room for
                                       them, as a collective's few channels
                                       would; the bulk-copy path still moves
                                       about 6 TB/s with one CTA per SM     */
    int64_t log_limit;              /* log records kept, the most recent ones:
                                       0 = 2^20, -1 = all (grows with every
                                       pass), n > 0 = n                     */
} zs_sched_config;

typedef struct {
    int64_t passes, gathers, params_gathered, elems_gathered, elems_prefetched;
    int64_t fetch_misses;           /* parameters gathered by the fetch itself */
    int64_t max_live_elems, max_arena_elems, invalidations;
} zs_sched_stats_t;

/* One record of the scheduler's log (for inspection and tests):
 * kind 1 gather: op, module position, param, offset, aux = release waited (-1)
 * kind 2 wait:   the compute of the module position waits for gather op
 *                (op -1: nothing to wait for)
 * kind 3 release: param released (-1: none) after the module position,
 *                aux = release index */
typedef struct {
    int32_t kind, module_pos, op, param;
    int64_t offset, aux;
} zs_sched_event;

/* Build a scheduler for the plan's parameters.  module_offsets[n_modules+1]
 * and module_params (CSR) list each module's parameter indices.  d_arena is
 * the device arena (16-byte aligned, arena_elems 2-byte elements), or NULL
 * for a plan-only scheduler that makes no CUDA call (its log and stats are
 * the same).  Errors: ZS_EINVAL (bad module list, parameter out of range,
 * arena smaller than the largest module), ZS_ECUDA, ZS_ENOMEM. */
zs_status zs_sched_create(const zs_plan *plan, int32_t n_modules, const int32_t *module_offsets,
                          const int32_t *module_params, const zs_sched_config *cfg,
                          void *d_arena, zs_sched **out);
void zs_sched_destroy(zs_sched *sched);

/* Fetch a module: param_shards is the plan's shard buffer [N][S].
 * Errors: ZS_EINVAL (module out of range), ZS_ENOMEM (the module's missing
 * parameters do not fit the arena), ZS_ECUDA. */
zs_status zs_sched_fetch(zs_sched *sched, int32_t module, const void *param_shards,
                         void *compute_stream, void *gather_stream);
/* Release after the module's compute (enqueued on compute_stream). */
zs_status zs_sched_release(zs_sched *sched, int32_t module, void *compute_stream);
/* End of a pass: release everything; completes or resets the trace. */
zs_status zs_sched_end_pass(zs_sched *sched, void *compute_stream);
/* Arena offset of the view of a gathered parameter (valid between the fetch
 * and the release of a module using it); -1 for a persistent parameter.
 * Errors: ZS_EINVAL (index), ZS_ESTATE (not gathered now). */
zs_status zs_sched_param_offset(const zs_sched *sched, int32_t param, int64_t *offset);
zs_status zs_sched_stats(const zs_sched *sched, zs_sched_stats_t *out);
/* Copy up to cap of the kept log records (oldest first); *n receives how
 * many are kept (at most log_limit). */
zs_status zs_sched_log(const zs_sched *sched, zs_sched_event *out, int64_t cap, int64_t *n);

#ifdef __cplusplus
}
#endif

#endif /* ZS_H */
