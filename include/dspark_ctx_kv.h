/*
 * dspark_ctx_kv.h -- C ABI of the GB300 (sm_103a) DSpark fused context-KV write.
 *
 * One call norms, ropes and stores the context K/V of every draft layer:
 * it reads K and V of each (token, layer, kv-head) row from the fused
 * projection output, applies the layer's Gemma RMSNorm to K (fp32, then
 * rounded to bf16), applies partial NeoX RoPE to the leading rotary_dim dims
 * of K at the token's position, and stores K|V into the layer's paged cache,
 * as raw bf16 or as OCP fp8 e4m3 of x / scale.  Tokens whose slot is < 0 are
 * padding: nothing is written for them and their positions are not used.
 *
 * Defining passages: vLLM DSpark context-KV writer page (module docstring:
 * layouts, norm, RoPE, fp8 rule, padding, cache/scale offset tables;
 * DSparkContextKVWriter._validate, _ensure_tables, __call__;
 * rotary_dims_supported) and the DSpark draft model page
 * (MiniMaxM3DSparkModel.precompute_and_store_context_kv, _shared_slot_mapping).
 *
 * Conventions for every function below:
 *  - Pointers documented as "device" must point to device memory of the
 *    current CUDA device; "host" pointers to host memory.
 *  - The caller owns every buffer.  dspark_ctx_kv_write allocates nothing,
 *    synchronises nothing and copies nothing, so it may be captured into a
 *    CUDA graph.
 *  - Functions return a dspark_status; none throws, aborts or exits.
 *    dspark_ctx_kv_last_error() describes the most recent failure of the
 *    calling thread.
 */
#ifndef DSPARK_CTX_KV_H
#define DSPARK_CTX_KV_H

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSPARK_HEAD_DIM 128
#define DSPARK_CACHE_ROW 256 /* K at [0, 128), V at [128, 256) */

/* Cache element type: raw bf16, or uint8 bytes holding OCP fp8 e4m3 codes. */
typedef enum { DSPARK_KV_BF16 = 0, DSPARK_KV_FP8_E4M3 = 1 } dspark_kv_dtype;

typedef enum {
    DSPARK_OK = 0,
    DSPARK_ERR_INVALID_ARG = 1,            /* null pointer, negative size, bad eps, mismatch */
    DSPARK_ERR_UNSUPPORTED_ROTARY_DIM = 2, /* rotary_dim not 16, 32 or 64 (head_dim 128) */
    DSPARK_ERR_BLOCK_SIZE = 3,             /* block_size not a positive power of two */
    DSPARK_ERR_ALIGNMENT = 4,              /* a buffer or layer offset misaligned */
    DSPARK_ERR_DTYPE = 5,                  /* unknown kv dtype, or cache dtype mismatch */
    DSPARK_ERR_CAPTURING = 6,              /* table rebuild requested while capturing */
    DSPARK_ERR_CUDA = 7,                   /* a CUDA runtime call failed */
} dspark_status;

/* Bits the kernel ORs into *error_flags (dspark_ctx_kv_write_ex).  A row
 * whose slot or position is out of range is skipped (nothing is written for
 * it) and reported; in-range rows are unaffected. */
#define DSPARK_FLAG_SLOT_RANGE 0x1u /* slot >= num_blocks * block_size */
#define DSPARK_FLAG_POS_RANGE 0x2u  /* position < 0 or >= max_pos (valid slot) */
#define DSPARK_FLAG_TIMEOUT 0x4u    /* an internal wait gave up and the kernel stopped early */
#define DSPARK_FLAG_COUNTER 0x8u    /* dspark_ctx_kv_write_sched: the work counter was not zero at launch */

/*
 * dspark_ctx_kv_write -- the fused write (writer page, module docstring and
 * DSparkContextKVWriter.__call__; one launch for all layers).
 *
 *  all_kv        device, bf16 [num_ctx, L, 2, nkv, 128] contiguous, 16-byte
 *                aligned: [t, l, 0, h, :] is K, [t, l, 1, h, :] is V.
 *  knorm_w       device, bf16 [L, 128] contiguous, 16-byte aligned: the
 *                per-layer Gemma K-norm weights w, applied as (1 + w).
 *  positions     device, int64 [num_ctx]: rotary position of each token
 *                (shared by all layers).
 *  slot_mapping  device, int64 [num_ctx], shared by all layers; < 0 marks
 *                padding.  Valid slots must be distinct and below
 *                num_blocks * block_size (duplicates race; out-of-range rows
 *                are skipped and flagged).
 *  num_ctx       number of tokens; 0 returns DSPARK_OK without a launch.
 *  cos_sin       device, bf16 [max_pos, rotary_dim] contiguous, 16-byte
 *                aligned: cos(pos * f_i) in [0, r/2), sin in [r/2, r).
 *  max_pos       rows of cos_sin (positions outside [0, max_pos) are
 *                skipped and flagged).
 *  layer0_cache  device, layer 0's cache [num_blocks, nkv, block_size, 256]
 *                of bf16 or uint8 (fp8), 16-byte aligned.  Layer l's cache
 *                starts cache_offsets[l] elements after it.
 *  num_blocks    blocks per layer cache.
 *  cache_offsets device, int64 [L]: element offset of each layer's cache from
 *                layer0_cache (multiples of 16 elements, may be negative;
 *                cache_offsets[0] is normally 0).  See the table builder.
 *  k_scales,     device, [L] arrays of device pointers to each layer's fp32
 *  v_scales      k / v scale (read when the kernel runs, so a graph replay
 *                sees current values).  Ignored (may be NULL) for bf16.
 *  L, nkv        draft layers and KV heads per layer (>= 1).
 *  block_size    tokens per cache block: a power of two.
 *  rotary_dim    16, 32 or 64.
 *  eps           the norm's epsilon (finite, >= 0).
 *  kv_dtype      a dspark_kv_dtype.
 *  stream        the CUDA stream the kernel is enqueued on.
 *
 * This entry point has no error word, so it cannot report what the kernel
 * flags: rows skipped as out of range, and a launch that gave up on one of
 * its bounded internal waits (DSPARK_FLAG_TIMEOUT) and left rows unwritten,
 * both pass silently.  dspark_ctx_kv_write_ex reports both.
 */
int dspark_ctx_kv_write(const void *all_kv, const void *knorm_w, const int64_t *positions,
                        const int64_t *slot_mapping, int64_t num_ctx, const void *cos_sin,
                        int64_t max_pos, void *layer0_cache, int64_t num_blocks,
                        const int64_t *cache_offsets, const float *const *k_scales,
                        const float *const *v_scales, int L, int nkv, int block_size,
                        int rotary_dim, float eps, int kv_dtype, cudaStream_t stream);

/* As dspark_ctx_kv_write, and the kernel ORs DSPARK_FLAG_* bits into
 * *error_flags (device, 4-byte aligned; NULL disables reporting).  The
 * caller clears the word; the call never does. */
int dspark_ctx_kv_write_ex(const void *all_kv, const void *knorm_w, const int64_t *positions,
                           const int64_t *slot_mapping, int64_t num_ctx, const void *cos_sin,
                           int64_t max_pos, void *layer0_cache, int64_t num_blocks,
                           const int64_t *cache_offsets, const float *const *k_scales,
                           const float *const *v_scales, int L, int nkv, int block_size,
                           int rotary_dim, float eps, int kv_dtype, unsigned int *error_flags,
                           cudaStream_t stream);

/*
 * dspark_ctx_kv_write_sched -- the write with a dynamic tail: as
 * dspark_ctx_kv_write_ex (one shared slot_mapping) or
 * dspark_ctx_kv_write_layer_slots (a device table of per-layer mappings) --
 * exactly one of the two non-NULL -- plus a work counter through which the
 * pipelined kernel hands the last tenth of a large call's units (a unit: a
 * token's rows of up to 8 layers) in runs of 4 to whichever CTA is free,
 * instead of a fixed CTA (a fixed split waits for its slowest CTA).  The
 * vLLM DSpark context-KV writer page has no counterpart: its kernel runs one
 * fixed grid.  Calls below 64 units per CTA (the grid is two CTAs per SM:
 * about 19.5k units on a 152-SM GPU), and layouts the pipelined kernel does
 * not take, keep the fixed split and leave the counter untouched.
 *
 *  work_counter  device, 2 x uint64, 8-byte aligned, owned by the caller:
 *                zero before its first use; every call leaves it zero
 *                again.  Calls that can run at the same time on the GPU
 *                (different streams without an order between them) need
 *                their own counters; NULL gives the fixed split.  A counter
 *                found far from zero raises DSPARK_FLAG_COUNTER and hands
 *                out nothing (rows of the tail stay unwritten; the call
 *                leaves it zero again); a small nonzero value skips that
 *                many runs unreported.
 */
int dspark_ctx_kv_write_sched(const void *all_kv, const void *knorm_w, const int64_t *positions,
                              const int64_t *slot_mapping, const int64_t *const *layer_slot_mappings,
                              int64_t num_ctx, const void *cos_sin, int64_t max_pos, void *layer0_cache,
                              int64_t num_blocks, const int64_t *cache_offsets, const float *const *k_scales,
                              const float *const *v_scales, int L, int nkv, int block_size, int rotary_dim,
                              float eps, int kv_dtype, unsigned int *error_flags, unsigned long long *work_counter,
                              cudaStream_t stream);

/*
 * dspark_ctx_kv_write_noalloc -- dspark_ctx_kv_write_sched with no memory
 * allocated by the caller or by the library: the per-layer tables are given
 * in HOST memory and the call keeps them, with the dynamic tail's work
 * counter, in one fixed device array of the library (16 + 32 *
 * DSPARK_NOALLOC_MAX_LAYERS bytes).  The DSpark pages have no counterpart
 * (their tables are framework tensors).
 *
 *  layer_slot_mappings_host  host array of L device pointers (per-layer
 *                   [num_ctx] int64 mappings), or NULL with slot_mapping
 *                   (exactly one of the two)
 *  cache_offsets_host  host int64[L], element offsets of each layer's cache
 *                   from layer0_cache (multiples of 16 elements)
 *  k_scales_host, v_scales_host  host arrays of L device float pointers
 *                   (fp8; NULL for bf16 caches)
 *  Other arguments as dspark_ctx_kv_write_sched.
 *
 * Each call copies its tables and the counter's zeros from host memory
 * into the array on `stream` (the host arrays may be reused as soon as the
 * call returns) and launches after that copy.  The first call on a device
 * also sets up: it looks up the array's device address once; make that call
 * before any stream capture.  There is one array per device, so calls whose
 * executions can overlap on the GPU (different streams with no order
 * between them, or threads issuing at the same time) race on it: order
 * them on one stream.  L above DSPARK_NOALLOC_MAX_LAYERS returns
 * DSPARK_ERR_INVALID_ARG before any CUDA call.
 */
#define DSPARK_NOALLOC_MAX_LAYERS 64
int dspark_ctx_kv_write_noalloc(const void *all_kv, const void *knorm_w, const int64_t *positions,
                                const int64_t *slot_mapping, const int64_t *const *layer_slot_mappings_host,
                                int64_t num_ctx, const void *cos_sin, int64_t max_pos, void *layer0_cache,
                                int64_t num_blocks, const int64_t *cache_offsets_host,
                                const float *const *k_scales_host, const float *const *v_scales_host, int L,
                                int nkv, int block_size, int rotary_dim, float eps, int kv_dtype,
                                unsigned int *error_flags, cudaStream_t stream);

/*
 * dspark_gemma_rms_norm -- the hidden-state Gemma RMSNorm of the context
 * states (DSpark draft model page: hidden_norm = _gemma_rms_norm(hidden_size,
 * eps), _normalize_context_states): for every row,
 * out = bf16(x * rsqrt(mean(x^2) + eps) * (1 + w)), evaluated in fp32.
 *
 *  x      device, bf16 [rows, hidden] contiguous, 16-byte aligned.
 *  w      device, bf16 [hidden], 16-byte aligned (applied as 1 + w).
 *  out    device, bf16 [rows, hidden], 16-byte aligned; may be x itself
 *         (in place), must not overlap it otherwise.
 *  hidden a positive multiple of 8, at most 8192.   eps: finite, >= 0.
 * rows == 0 returns DSPARK_OK without a launch.  One launch; allocates,
 * copies and synchronises nothing.
 */
int dspark_gemma_rms_norm(const void *x, const void *w, void *out, int64_t rows, int hidden, float eps,
                          cudaStream_t stream);

/*
 * dspark_ctx_kv_project -- the context-KV projection on the tensor cores
 * (DSpark draft model page, precompute_and_store_context_kv:
 * all_kv = _project_context_kv_token_major(context_states, ...)):
 * all_kv_out[t, n] = bf16(sum_k x[t, k] * w_kv[n, k]) with an fp32
 * accumulator, n = ((l * 2 + kv) * nkv + h) * 128 + d.
 *
 *  x           device, bf16 [num_ctx, hidden] contiguous, 16-byte aligned
 *              (the normed context states).
 *  w_kv        device, bf16 [L * 2 * nkv * 128, hidden] contiguous, 16-byte
 *              aligned: the K and V projection rows of every layer.
 *  all_kv_out  device, bf16 [num_ctx, L, 2, nkv, 128], 16-byte aligned.
 *  hidden      a positive multiple of 8; 1 <= L * nkv <= 65535;
 *              num_ctx <= 8,388,480 (0 returns DSPARK_OK without a launch).
 * One launch; allocates, copies and synchronises nothing (the tensor maps
 * travel as kernel parameters).
 */
int dspark_ctx_kv_project(const void *x, const void *w_kv, void *all_kv_out, int64_t num_ctx, int hidden, int L,
                          int nkv, cudaStream_t stream);

/*
 * dspark_ctx_kv_project_write -- the projection with the context-KV write in
 * its epilogue: the same result as dspark_ctx_kv_project followed by
 * dspark_ctx_kv_write_ex on its output, in one launch, without all_kv in
 * device memory.  x, w_kv, num_ctx and hidden as for dspark_ctx_kv_project;
 * every other argument as for dspark_ctx_kv_write_ex; L <= 32.
 */
int dspark_ctx_kv_project_write(const void *x, const void *w_kv, int64_t num_ctx, int hidden, const void *knorm_w,
                                const int64_t *positions, const int64_t *slot_mapping, const void *cos_sin,
                                int64_t max_pos, void *layer0_cache, int64_t num_blocks,
                                const int64_t *cache_offsets, const float *const *k_scales,
                                const float *const *v_scales, int L, int nkv, int block_size, int rotary_dim,
                                float eps, int kv_dtype, unsigned int *error_flags, cudaStream_t stream);

/*
 * dspark_qknorm_rope_kv_insert -- the draft tokens' fused QK-norm / RoPE,
 * also storing their K/V (DSpark draft model page,
 * dspark_qknorm_rope_kv_insert; norm, RoPE, cache layout and fp8 rule as in
 * the context-KV writer page).  One launch.
 *
 *  qkv           device, bf16 [num_tokens, (num_heads + 2 num_kv_heads) * 128]
 *                contiguous, 16-byte aligned: per token the query heads, then
 *                the key heads, then the value heads.  Updated in place: every
 *                query and key head of every token (padding included) becomes
 *                RoPE(GemmaRMSNorm(x)) in bf16; value heads are not changed.
 *  q_norm_w,     device, bf16 [128] each, 16-byte aligned: the Gemma weights
 *  k_norm_w      w of the query and key norms (applied as 1 + w to every head).
 *  cos_sin       device, bf16 [max_pos, rotary_dim], 16-byte aligned (cos | sin).
 *  positions     device, int64 [num_tokens].  A token whose position lies
 *                outside [0, max_pos) is left untouched (not inserted either)
 *                and DSPARK_FLAG_POS_RANGE is raised.
 *  num_heads, num_kv_heads   query heads and KV heads (>= 1); head_dim 128.
 *  rotary_dim    16, 32 or 64.   eps: finite, >= 0.
 *  slot_mapping  device, int64 [num_tokens], or NULL: no insert.  Tokens with
 *                slot >= 0 have each KV head's K'|V row stored at block
 *                slot / block_size, offset slot % block_size; valid slots
 *                must be distinct (duplicates race); a slot beyond the cache
 *                is not inserted and raises DSPARK_FLAG_SLOT_RANGE.
 *  kv_cache      device, [num_blocks, num_kv_heads, block_size, 256] of bf16
 *                (kv_dtype DSPARK_KV_BF16) or uint8 e4m3 codes
 *                (DSPARK_KV_FP8_E4M3), 16-byte aligned; NULL exactly when
 *                slot_mapping is NULL.
 *  k_scale,      device fp32 scalars read when the kernel runs: an fp8 cache
 *  v_scale       stores e4m3(x / scale) (IEEE fp32 division, RNE, saturating
 *                at +-448); NULL means 1.  Ignored for a bf16 cache.
 *  q_fp8_out     device, uint8 [num_tokens, num_heads * 128], 16-byte aligned,
 *                or NULL: receives e4m3(q' / q_fp8_scale) of every query head.
 *  q_fp8_scale   host fp32, positive and finite when q_fp8_out is given.
 *  error_flags   device word the kernel ORs DSPARK_FLAG_* bits into, or NULL.
 *  stream        the CUDA stream the kernel is enqueued on.
 * num_tokens == 0 returns DSPARK_OK without a launch.  Allocates, copies and
 * synchronises nothing.
 */
int dspark_qknorm_rope_kv_insert(void *qkv, const void *q_norm_w, const void *k_norm_w, const void *cos_sin,
                                 int64_t max_pos, const int64_t *positions, int64_t num_tokens, int num_heads,
                                 int num_kv_heads, int rotary_dim, float eps, const int64_t *slot_mapping,
                                 void *kv_cache, int64_t num_blocks, int block_size, int kv_dtype,
                                 const float *k_scale, const float *v_scale, void *q_fp8_out, float q_fp8_scale,
                                 unsigned int *error_flags, cudaStream_t stream);

/* As dspark_ctx_kv_write_ex, for a draft whose layers do not share one slot
 * mapping (DSpark draft model page, _shared_slot_mapping: drafts whose
 * layers span several KV-cache groups).  layer_slot_mappings: device, [L]
 * device pointers (8-byte aligned) to each layer's int64 [num_ctx] mapping,
 * e.g. dspark_ctx_kv_tables_layer_slots.  Layer l's rows of token t go to
 * layer l's slot of t (< 0: not written); valid slots must be distinct
 * within each layer.  Positions stay shared by all layers. */
int dspark_ctx_kv_write_layer_slots(const void *all_kv, const void *knorm_w, const int64_t *positions,
                                    const int64_t *const *layer_slot_mappings, int64_t num_ctx,
                                    const void *cos_sin, int64_t max_pos, void *layer0_cache, int64_t num_blocks,
                                    const int64_t *cache_offsets, const float *const *k_scales,
                                    const float *const *v_scales, int L, int nkv, int block_size, int rotary_dim,
                                    float eps, int kv_dtype, unsigned int *error_flags, cudaStream_t stream);

/*
 * dspark_ctx_kv_write_general -- the same write for the layouts the pages'
 * kernel refuses and hands to the unfused path (writer page,
 * DSparkContextKVWriter._validate and rotary_dims_supported accept only
 * head_dim 128, rotary_dim 16 / 32 / 64 and power-of-two block sizes):
 *
 *  head_dim      D = 64, 128 or 256.  all_kv is bf16 [num_ctx, L, 2, nkv, D],
 *                knorm_w bf16 [L, D], every layer's cache
 *                [num_blocks, nkv, block_size, 2D] (K at [0, D), V at [D, 2D)).
 *  rotary_dim    any even value in [2, D]: NeoX pairs (i, i + r/2), cos_sin
 *                bf16 [max_pos, rotary_dim] (cos | sin).
 *  block_size    any value >= 1: block slot / block_size, offset
 *                slot % block_size.
 *  slot_mapping, exactly one of the two is given: a mapping shared by every
 *  layer_slot_mappings  layer (device int64 [num_ctx]) or a device table of
 *                L device pointers to per-layer mappings (8-byte aligned).
 * Every other argument, the alignment rules (16-byte buffers, 16-element
 * layer offsets), the error flags and the statuses are those of
 * dspark_ctx_kv_write_ex / dspark_ctx_kv_write_layer_slots; an unsupported
 * head_dim is DSPARK_ERR_INVALID_ARG, an odd or out-of-range rotary_dim
 * DSPARK_ERR_UNSUPPORTED_ROTARY_DIM, block_size < 1 DSPARK_ERR_BLOCK_SIZE.
 * A call in the pages' layout takes the same kernels as dspark_ctx_kv_write_ex.
 * One launch; allocates, copies and synchronises nothing.
 */
int dspark_ctx_kv_write_general(const void *all_kv, const void *knorm_w, const int64_t *positions,
                                const int64_t *slot_mapping, const int64_t *const *layer_slot_mappings,
                                int64_t num_ctx, const void *cos_sin, int64_t max_pos, void *layer0_cache,
                                int64_t num_blocks, const int64_t *cache_offsets, const float *const *k_scales,
                                const float *const *v_scales, int L, int nkv, int head_dim, int block_size,
                                int rotary_dim, float eps, int kv_dtype, unsigned int *error_flags,
                                cudaStream_t stream);

/* 1 when dspark_ctx_kv_write_general handles this layout (head_dim 64, 128
 * or 256; rotary_dim even in [2, head_dim]; block_size >= 1), else 0. */
int dspark_ctx_kv_general_supported(int head_dim, int rotary_dim, int block_size);

/* 1 when the kernel handles this head (writer page, rotary_dims_supported:
 * head_dim 128 and rotary_dim 16, 32 or 64), else 0. */
int dspark_ctx_kv_rotary_dims_supported(int rotary_dim, int head_dim);

/*
 * Per-layer cache description for the layout check (writer page,
 * DSparkContextKVWriter._validate).  All fields describe the caller's
 * tensors; nothing is dereferenced.
 */
typedef struct {
    const void *data;      /* device address of the layer's cache */
    int64_t shape[4];      /* [num_blocks, nkv, block_size, 256] expected */
    int64_t stride[4];     /* in elements */
    int32_t ndim;
    int32_t elem_size;     /* bytes per element */
    int32_t cache_dtype;   /* dspark_kv_dtype of the cache tensor's element type
                              (bf16 -> DSPARK_KV_BF16, uint8 -> DSPARK_KV_FP8_E4M3,
                              anything else -> -1) */
    int32_t kv_dtype;      /* the layer's configured kv dtype (dspark_kv_dtype, -1 unknown) */
    const void *k_scale;   /* device address of the fp32 k scale */
    const void *v_scale;
    int32_t scales_ok;     /* 1 when both scales are fp32 tensors on the GPU */
} dspark_cache_desc;

/* DSPARK_OK when the layers form a layout the write supports: at least one
 * layer; 4-D contiguous caches with last dim 256; power-of-two block size;
 * fp8 caches are uint8 and bf16 caches are bf16; fp32 device scales; all
 * layers share shape, stride and dtype; every cache starts a multiple of 16
 * elements from layer 0's.  Otherwise the status of the first violation. */
int dspark_ctx_kv_validate_layers(int L, const dspark_cache_desc *layers);

/* As dspark_ctx_kv_validate_layers for dspark_ctx_kv_write_general: the
 * last dim may be 128, 256 or 512 (head_dim 64, 128, 256) and the block size
 * any value >= 1; every other rule is the same. */
int dspark_ctx_kv_validate_layers_general(int L, const dspark_cache_desc *layers);

/*
 * Offset/pointer tables (writer page, DSparkContextKVWriter._ensure_tables):
 * cache_offsets[L] (int64 element offsets from layer 0's cache) and the k /
 * v scale pointer tables, in device memory owned by the object.  The tables
 * are rebuilt only when the key (every layer's cache and scale address and
 * the element size) changes, so launches captured in a CUDA graph keep
 * addressing the same memory.
 */
typedef struct dspark_ctx_kv_tables dspark_ctx_kv_tables;

/* Allocates the object and its device tables (cudaMalloc on the current
 * device: call outside stream capture). */
int dspark_ctx_kv_tables_create(int L, dspark_ctx_kv_tables **out);

/* layer_caches, k_scale_ptrs, v_scale_ptrs: host arrays [L] of device
 * addresses.  Same key as the last successful update: DSPARK_OK, nothing
 * enqueued.  New key: validates alignment (16 elements) and enqueues the
 * host-to-device copy of the new tables on `stream`, unless `stream` is
 * capturing, which returns DSPARK_ERR_CAPTURING and keeps the old tables.
 * The tables must not be updated while launches that read them are still
 * running on another stream. */
int dspark_ctx_kv_tables_update(dspark_ctx_kv_tables *tables, void *const *layer_caches,
                                size_t elem_size, const float *const *k_scale_ptrs,
                                const float *const *v_scale_ptrs, cudaStream_t stream);

/* Per-layer slot mappings: layer_slot_ptrs is a host array [L] of device
 * addresses of int64 [num_ctx] mappings.  Same addresses as the last call:
 * DSPARK_OK, nothing enqueued; new ones: the device pointer table is copied
 * on `stream`, unless it is capturing (DSPARK_ERR_CAPTURING, table kept). */
int dspark_ctx_kv_tables_update_slots(dspark_ctx_kv_tables *tables, const int64_t *const *layer_slot_ptrs,
                                      cudaStream_t stream);
const int64_t *const *dspark_ctx_kv_tables_layer_slots(const dspark_ctx_kv_tables *tables);
const int64_t *dspark_ctx_kv_tables_cache_offsets(const dspark_ctx_kv_tables *tables);
const float *const *dspark_ctx_kv_tables_k_scales(const dspark_ctx_kv_tables *tables);
const float *const *dspark_ctx_kv_tables_v_scales(const dspark_ctx_kv_tables *tables);
/* Number of times the tables were (re)built: 0 before the first update. */
int64_t dspark_ctx_kv_tables_builds(const dspark_ctx_kv_tables *tables);
void dspark_ctx_kv_tables_destroy(dspark_ctx_kv_tables *tables);

/* Text of the calling thread's most recent error ("" if none). */
const char *dspark_ctx_kv_last_error(void);
/* Name of a dspark_status value. */
const char *dspark_ctx_kv_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* DSPARK_CTX_KV_H */
