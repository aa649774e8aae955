// C-ABI host layer of the DSpark fused context-KV write: argument checks,
// the layout check, the capture-safe offset/pointer tables and the launch.
//
// Defining passages: vLLM DSpark context-KV writer page --
// DSparkContextKVWriter._validate (layout rules), .supported, _ensure_tables
// (per-layer cache element offsets and scale addresses, rebuilt only when the
// data_ptrs change so CUDA-graph replays keep addressing the same memory),
// __call__ (num_ctx == 0 launches nothing), rotary_dims_supported (head_dim
// 128, rotary_dim 16/32/64); DSpark draft model page --
// dspark_qknorm_rope_kv_insert (the draft tokens' fused QK-norm/RoPE and K/V
// insert, its insert skipped without a slot mapping); precompute_and_store_
// context_kv (the context states' projection into all_kv, on its own or with
// the write fused into it).
#include "../../include/dspark_ctx_kv.h"

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "ctx_kv_internal.h"

namespace {

thread_local char g_last_error[512] = "";

int fail(int status, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return status;
}

int ok()
{
    g_last_error[0] = '\0';
    return DSPARK_OK;
}

// Which kernel serves a call: for small calls (at most kWarpPathMaxTokens
// tokens: draft steps) in the pages' layouts with 4 or 8 KV heads and a
// shared slot mapping, the warp-private pipelines (every warp starts on its
// own 4 KB unit at once: shorter chains than the shared stages give when a
// CTA gets one or two tokens); otherwise the pipelined one where a token's
// rows fit a stage, else the generic one for the pages' layouts; the general
// kernel for every other layout.  DSPARK_CTX_KV_KERNEL=warp picks the
// warp-private pipelines wherever they apply, =tma the pipelined kernel,
// =generic the generic kernel for the pages' layouts and =general the
// general kernel for every layout, for the calls made while it is set (all
// compute the same result; the tests run each).
constexpr int64_t kWarpPathMaxTokens = 1024;
bool force_kernel(const char *name)
{
    const char *e = std::getenv("DSPARK_CTX_KV_KERNEL");
    return e && std::strcmp(e, name) == 0;
}

// DSPARK_TEST_HOLD_NS=<ns> (tests of the timeout path only): the pipelined
// kernel's producer first waits that long on a device word that nothing
// sets, then stops as on any expired wait and reports DSPARK_FLAG_TIMEOUT.
uint64_t test_hold_ns()
{
    const char *e = std::getenv("DSPARK_TEST_HOLD_NS");
    if (!e)
        return 0;
    const long long v = std::atoll(e);
    return v > 0 ? (uint64_t)std::min(v, 1000000000LL) : 0;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool pow2(int64_t v) { return v > 0 && (v & (v - 1)) == 0; }

int log2_exact(int64_t v)
{
    int n = 0;
    while ((int64_t(1) << n) < v)
        n++;
    return n;
}

// Which layouts a call accepts: the pages' (head_dim 128, rotary_dim 16 /
// 32 / 64, power-of-two block sizes) or the general write's.
enum class Rules { pages, general };

// The write with a shared or a per-layer slot mapping (exactly one is given).
int write_common(const void *all_kv, const void *knorm_w, const int64_t *positions, const int64_t *slot_mapping,
                 const int64_t *const *layer_slots, int64_t num_ctx, const void *cos_sin, int64_t max_pos,
                 void *layer0_cache, int64_t num_blocks, const int64_t *cache_offsets, const float *const *k_scales,
                 const float *const *v_scales, int L, int nkv, int head_dim, int block_size, int rotary_dim,
                 float eps, int kv_dtype, unsigned int *error_flags, cudaStream_t stream, Rules rules,
                 unsigned long long *work_counter = nullptr);

}  // namespace

int dspark::api_fail(int status, const char *message) { return fail(status, "%s", message); }

extern "C" {

const char *dspark_ctx_kv_last_error(void) { return g_last_error; }

const char *dspark_ctx_kv_status_string(int status)
{
    switch (status) {
    case DSPARK_OK: return "DSPARK_OK";
    case DSPARK_ERR_INVALID_ARG: return "DSPARK_ERR_INVALID_ARG";
    case DSPARK_ERR_UNSUPPORTED_ROTARY_DIM: return "DSPARK_ERR_UNSUPPORTED_ROTARY_DIM";
    case DSPARK_ERR_BLOCK_SIZE: return "DSPARK_ERR_BLOCK_SIZE";
    case DSPARK_ERR_ALIGNMENT: return "DSPARK_ERR_ALIGNMENT";
    case DSPARK_ERR_DTYPE: return "DSPARK_ERR_DTYPE";
    case DSPARK_ERR_CAPTURING: return "DSPARK_ERR_CAPTURING";
    case DSPARK_ERR_CUDA: return "DSPARK_ERR_CUDA";
    default: return "DSPARK_ERR_UNKNOWN";
    }
}

int dspark_ctx_kv_rotary_dims_supported(int rotary_dim, int head_dim)
{
    return head_dim == DSPARK_HEAD_DIM && (rotary_dim == 16 || rotary_dim == 32 || rotary_dim == 64);
}

int dspark_ctx_kv_write_ex(const void *all_kv, const void *knorm_w, const int64_t *positions,
                           const int64_t *slot_mapping, int64_t num_ctx, const void *cos_sin,
                           int64_t max_pos, void *layer0_cache, int64_t num_blocks,
                           const int64_t *cache_offsets, const float *const *k_scales,
                           const float *const *v_scales, int L, int nkv, int block_size,
                           int rotary_dim, float eps, int kv_dtype, unsigned int *error_flags,
                           cudaStream_t stream)
{
    if (num_ctx > 0 && !slot_mapping)
        return fail(DSPARK_ERR_INVALID_ARG, "null slot_mapping");
    return write_common(all_kv, knorm_w, positions, slot_mapping, nullptr, num_ctx, cos_sin, max_pos, layer0_cache,
                        num_blocks, cache_offsets, k_scales, v_scales, L, nkv, DSPARK_HEAD_DIM, block_size,
                        rotary_dim, eps, kv_dtype, error_flags, stream, Rules::pages);
}

int dspark_ctx_kv_write_layer_slots(const void *all_kv, const void *knorm_w, const int64_t *positions,
                                    const int64_t *const *layer_slot_mappings, int64_t num_ctx,
                                    const void *cos_sin, int64_t max_pos, void *layer0_cache, int64_t num_blocks,
                                    const int64_t *cache_offsets, const float *const *k_scales,
                                    const float *const *v_scales, int L, int nkv, int block_size, int rotary_dim,
                                    float eps, int kv_dtype, unsigned int *error_flags, cudaStream_t stream)
{
    if (num_ctx > 0 && (!layer_slot_mappings || !aligned(layer_slot_mappings, 8)))
        return fail(DSPARK_ERR_INVALID_ARG, "layer_slot_mappings must be an 8-byte aligned device pointer table");
    return write_common(all_kv, knorm_w, positions, nullptr, layer_slot_mappings, num_ctx, cos_sin, max_pos,
                        layer0_cache, num_blocks, cache_offsets, k_scales, v_scales, L, nkv, DSPARK_HEAD_DIM,
                        block_size, rotary_dim, eps, kv_dtype, error_flags, stream, Rules::pages);
}

int dspark_ctx_kv_write_sched(const void *all_kv, const void *knorm_w, const int64_t *positions,
                              const int64_t *slot_mapping, const int64_t *const *layer_slot_mappings,
                              int64_t num_ctx, const void *cos_sin, int64_t max_pos, void *layer0_cache,
                              int64_t num_blocks, const int64_t *cache_offsets, const float *const *k_scales,
                              const float *const *v_scales, int L, int nkv, int block_size, int rotary_dim,
                              float eps, int kv_dtype, unsigned int *error_flags, unsigned long long *work_counter,
                              cudaStream_t stream)
{
    if (num_ctx > 0 && (slot_mapping == nullptr) == (layer_slot_mappings == nullptr))
        return fail(DSPARK_ERR_INVALID_ARG, "give exactly one of slot_mapping and layer_slot_mappings");
    if (num_ctx > 0 && layer_slot_mappings && !aligned(layer_slot_mappings, 8))
        return fail(DSPARK_ERR_ALIGNMENT, "layer_slot_mappings must be 8-byte aligned");
    return write_common(all_kv, knorm_w, positions, slot_mapping, layer_slot_mappings, num_ctx, cos_sin, max_pos,
                        layer0_cache, num_blocks, cache_offsets, k_scales, v_scales, L, nkv, DSPARK_HEAD_DIM,
                        block_size, rotary_dim, eps, kv_dtype, error_flags, stream, Rules::pages, work_counter);
}

int dspark_ctx_kv_general_supported(int head_dim, int rotary_dim, int block_size)
{
    return (head_dim == 64 || head_dim == 128 || head_dim == 256) && rotary_dim >= 2 && rotary_dim <= head_dim &&
           rotary_dim % 2 == 0 && block_size >= 1;
}

int dspark_ctx_kv_write_general(const void *all_kv, const void *knorm_w, const int64_t *positions,
                                const int64_t *slot_mapping, const int64_t *const *layer_slot_mappings,
                                int64_t num_ctx, const void *cos_sin, int64_t max_pos, void *layer0_cache,
                                int64_t num_blocks, const int64_t *cache_offsets, const float *const *k_scales,
                                const float *const *v_scales, int L, int nkv, int head_dim, int block_size,
                                int rotary_dim, float eps, int kv_dtype, unsigned int *error_flags,
                                cudaStream_t stream)
{
    if (num_ctx > 0 && (slot_mapping == nullptr) == (layer_slot_mappings == nullptr))
        return fail(DSPARK_ERR_INVALID_ARG, "give exactly one of slot_mapping and layer_slot_mappings");
    if (num_ctx > 0 && layer_slot_mappings && !aligned(layer_slot_mappings, 8))
        return fail(DSPARK_ERR_ALIGNMENT, "layer_slot_mappings must be 8-byte aligned");
    return write_common(all_kv, knorm_w, positions, slot_mapping, layer_slot_mappings, num_ctx, cos_sin, max_pos,
                        layer0_cache, num_blocks, cache_offsets, k_scales, v_scales, L, nkv, head_dim, block_size,
                        rotary_dim, eps, kv_dtype, error_flags, stream, Rules::general);
}

}  // extern "C"

namespace {

// Granlund-Montgomery magic of an invariant divisor d >= 3 that is not a
// power of two, for dividends 0 <= n < 2^63: with l = ceil(log2 d),
// m = ceil(2^(63 + l) / d) < 2^64 and floor(n / d) = umulhi(n, m) >> (l - 1).
void block_divisor(int64_t d, uint64_t *magic, int *shift)
{
    const int l = log2_exact(d);
    const unsigned __int128 num = (unsigned __int128)1 << (63 + l);
    *magic = (uint64_t)((num + (unsigned __int128)(d - 1)) / (unsigned __int128)d);
    *shift = l - 1;
}

int write_common(const void *all_kv, const void *knorm_w, const int64_t *positions, const int64_t *slot_mapping,
                 const int64_t *const *layer_slots, int64_t num_ctx, const void *cos_sin, int64_t max_pos,
                 void *layer0_cache, int64_t num_blocks, const int64_t *cache_offsets, const float *const *k_scales,
                 const float *const *v_scales, int L, int nkv, int head_dim, int block_size, int rotary_dim,
                 float eps, int kv_dtype, unsigned int *error_flags, cudaStream_t stream, Rules rules,
                 unsigned long long *work_counter)
{
    // Scalar checks first: they need no device and no pointer.
    if (num_ctx < 0)
        return fail(DSPARK_ERR_INVALID_ARG, "num_ctx %lld < 0", (long long)num_ctx);
    if (L <= 0 || nkv <= 0)
        return fail(DSPARK_ERR_INVALID_ARG, "L=%d nkv=%d must be >= 1", L, nkv);
    if (num_blocks <= 0 || max_pos <= 0)
        return fail(DSPARK_ERR_INVALID_ARG, "num_blocks=%lld max_pos=%lld must be >= 1",
                    (long long)num_blocks, (long long)max_pos);
    if (rules == Rules::pages) {
        if (!dspark_ctx_kv_rotary_dims_supported(rotary_dim, DSPARK_HEAD_DIM))
            return fail(DSPARK_ERR_UNSUPPORTED_ROTARY_DIM, "rotary_dim %d not in {16, 32, 64}", rotary_dim);
        if (!pow2(block_size))
            return fail(DSPARK_ERR_BLOCK_SIZE, "block size %d is not a power of two", block_size);
    } else {
        if (head_dim != 64 && head_dim != 128 && head_dim != 256)
            return fail(DSPARK_ERR_INVALID_ARG, "head_dim %d not 64, 128 or 256", head_dim);
        if (rotary_dim < 2 || rotary_dim > head_dim || rotary_dim % 2 != 0)
            return fail(DSPARK_ERR_UNSUPPORTED_ROTARY_DIM, "rotary_dim %d not even in [2, %d]", rotary_dim,
                        head_dim);
        if (block_size < 1)
            return fail(DSPARK_ERR_BLOCK_SIZE, "block size %d < 1", block_size);
    }
    if (kv_dtype != DSPARK_KV_BF16 && kv_dtype != DSPARK_KV_FP8_E4M3)
        return fail(DSPARK_ERR_DTYPE, "kv dtype %d unknown", kv_dtype);
    if (!(eps >= 0.0f) || std::isinf(eps))
        return fail(DSPARK_ERR_INVALID_ARG, "eps must be finite and >= 0");
    const int64_t row_elems = 2 * (int64_t)head_dim;
    const int64_t capacity = num_blocks * (int64_t)block_size;
    if (capacity / block_size != num_blocks || num_blocks > (INT64_MAX / nkv) / block_size / row_elems)
        return fail(DSPARK_ERR_INVALID_ARG, "cache of %lld blocks too large", (long long)num_blocks);
    if (num_ctx > (INT64_MAX / L) / nkv / row_elems)
        return fail(DSPARK_ERR_INVALID_ARG, "num_ctx %lld too large", (long long)num_ctx);
    if (num_ctx == 0)
        return ok();  // nothing to store, and no launch

    if (!all_kv || !knorm_w || !positions || !cos_sin || !layer0_cache || !cache_offsets)
        return fail(DSPARK_ERR_INVALID_ARG, "null buffer pointer");
    if (kv_dtype == DSPARK_KV_FP8_E4M3 && (!k_scales || !v_scales))
        return fail(DSPARK_ERR_INVALID_ARG, "fp8 cache needs k_scales and v_scales");
    if (!aligned(all_kv, 16) || !aligned(knorm_w, 16) || !aligned(cos_sin, 16) || !aligned(layer0_cache, 16))
        return fail(DSPARK_ERR_ALIGNMENT, "all_kv, knorm_w, cos_sin and layer0_cache must be 16-byte aligned");
    if (!aligned(positions, 8) || (slot_mapping && !aligned(slot_mapping, 8)) || !aligned(cache_offsets, 8) ||
        (k_scales && !aligned(k_scales, 8)) || (v_scales && !aligned(v_scales, 8)))
        return fail(DSPARK_ERR_ALIGNMENT, "int64 and pointer tables must be 8-byte aligned");
    if (error_flags && !aligned(error_flags, 4))
        return fail(DSPARK_ERR_ALIGNMENT, "error_flags must be 4-byte aligned");
    if (work_counter && !aligned(work_counter, 8))
        return fail(DSPARK_ERR_ALIGNMENT, "work_counter must be 8-byte aligned");

    dspark::CtxKvParams p{};
    p.work_counter = work_counter;
    p.all_kv = static_cast<const uint16_t *>(all_kv);
    p.knorm_w = static_cast<const uint16_t *>(knorm_w);
    p.positions = positions;
    p.slot_mapping = slot_mapping;
    p.layer_slots = layer_slots;
    p.cos_sin = static_cast<const uint16_t *>(cos_sin);
    p.cache0 = static_cast<unsigned char *>(layer0_cache);
    p.cache_offsets = cache_offsets;
    p.k_scales = k_scales;
    p.v_scales = v_scales;
    p.error_flags = error_flags;
    p.num_ctx = num_ctx;
    p.max_pos = max_pos;
    p.capacity = capacity;
    p.num_layers = L;
    p.num_kv_heads = nkv;
    p.block_size_log2 = pow2(block_size) ? log2_exact(block_size) : -1;
    p.eps = eps;
    p.rotary_dim = rotary_dim;
    p.block_size = block_size;
    if (!pow2(block_size))
        block_divisor(block_size, &p.bs_magic, &p.bs_magic_shift);
    p.test_hold_ns = test_hold_ns();
    const bool fp8 = kv_dtype == DSPARK_KV_FP8_E4M3;
    // the pipelined kernel where its stage holds a token's rows; else the
    // generic kernel (the pages' layouts) or the general one (any other)
    const bool pages_layout = head_dim == DSPARK_HEAD_DIM && pow2(block_size) &&
                              dspark_ctx_kv_rotary_dims_supported(rotary_dim, DSPARK_HEAD_DIM);
    cudaError_t e;
    if (force_kernel("general"))
        e = dspark::launch_ctx_kv_general(p, head_dim, fp8, stream);
    else if (pages_layout && force_kernel("generic"))
        e = dspark::launch_ctx_kv_write(p, rotary_dim, fp8, stream);
    else if (pages_layout && dspark::warp_path_supported(p) &&
             (force_kernel("warp") || (num_ctx <= kWarpPathMaxTokens && !force_kernel("tma"))))
        e = dspark::launch_ctx_kv_write_warp(p, fp8, stream);
    else if (dspark::tma_path_supported(p, head_dim))
        e = dspark::launch_ctx_kv_write_tma(p, head_dim, fp8, stream);
    else if (pages_layout)
        e = dspark::launch_ctx_kv_write(p, rotary_dim, fp8, stream);
    else
        e = dspark::launch_ctx_kv_general(p, head_dim, fp8, stream);
    if (e != cudaSuccess)
        return fail(DSPARK_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    return ok();
}

}  // namespace

extern "C" {

int dspark_ctx_kv_write(const void *all_kv, const void *knorm_w, const int64_t *positions,
                        const int64_t *slot_mapping, int64_t num_ctx, const void *cos_sin,
                        int64_t max_pos, void *layer0_cache, int64_t num_blocks,
                        const int64_t *cache_offsets, const float *const *k_scales,
                        const float *const *v_scales, int L, int nkv, int block_size,
                        int rotary_dim, float eps, int kv_dtype, cudaStream_t stream)
{
    return dspark_ctx_kv_write_ex(all_kv, knorm_w, positions, slot_mapping, num_ctx, cos_sin, max_pos,
                                  layer0_cache, num_blocks, cache_offsets, k_scales, v_scales, L, nkv,
                                  block_size, rotary_dim, eps, kv_dtype, nullptr, stream);
}

int dspark_qknorm_rope_kv_insert(void *qkv, const void *q_norm_w, const void *k_norm_w, const void *cos_sin,
                                 int64_t max_pos, const int64_t *positions, int64_t num_tokens, int num_heads,
                                 int num_kv_heads, int rotary_dim, float eps, const int64_t *slot_mapping,
                                 void *kv_cache, int64_t num_blocks, int block_size, int kv_dtype,
                                 const float *k_scale, const float *v_scale, void *q_fp8_out, float q_fp8_scale,
                                 unsigned int *error_flags, cudaStream_t stream)
{
    if (num_tokens < 0)
        return fail(DSPARK_ERR_INVALID_ARG, "num_tokens %lld < 0", (long long)num_tokens);
    if (num_heads <= 0 || num_kv_heads <= 0)
        return fail(DSPARK_ERR_INVALID_ARG, "num_heads=%d num_kv_heads=%d must be >= 1", num_heads, num_kv_heads);
    if (max_pos <= 0)
        return fail(DSPARK_ERR_INVALID_ARG, "max_pos %lld must be >= 1", (long long)max_pos);
    if (!dspark_ctx_kv_rotary_dims_supported(rotary_dim, DSPARK_HEAD_DIM))
        return fail(DSPARK_ERR_UNSUPPORTED_ROTARY_DIM, "rotary_dim %d not in {16, 32, 64}", rotary_dim);
    if (!(eps >= 0.0f) || std::isinf(eps))
        return fail(DSPARK_ERR_INVALID_ARG, "eps must be finite and >= 0");
    const int64_t width = (int64_t)num_heads + 2 * (int64_t)num_kv_heads;
    if (width > (int64_t)1 << 24 || num_tokens > (INT64_MAX / width) / (2 * DSPARK_HEAD_DIM))
        return fail(DSPARK_ERR_INVALID_ARG, "num_tokens %lld too large", (long long)num_tokens);
    const bool insert = slot_mapping != nullptr && kv_cache != nullptr;
    if ((slot_mapping != nullptr) != (kv_cache != nullptr))
        return fail(DSPARK_ERR_INVALID_ARG, "slot_mapping and kv_cache go together (both or neither)");
    int64_t capacity = 0;
    int bsl = 0;
    if (insert) {
        if (!pow2(block_size))
            return fail(DSPARK_ERR_BLOCK_SIZE, "block size %d is not a power of two", block_size);
        if (kv_dtype != DSPARK_KV_BF16 && kv_dtype != DSPARK_KV_FP8_E4M3)
            return fail(DSPARK_ERR_DTYPE, "kv dtype %d unknown", kv_dtype);
        if (num_blocks <= 0 || num_blocks > (INT64_MAX / num_kv_heads) / block_size / DSPARK_CACHE_ROW)
            return fail(DSPARK_ERR_INVALID_ARG, "cache of %lld blocks invalid", (long long)num_blocks);
        capacity = num_blocks * (int64_t)block_size;
        bsl = log2_exact(block_size);
        if (!aligned(kv_cache, 16))
            return fail(DSPARK_ERR_ALIGNMENT, "kv_cache must be 16-byte aligned");
        if (!aligned(slot_mapping, 8) || (k_scale && !aligned(k_scale, 4)) || (v_scale && !aligned(v_scale, 4)))
            return fail(DSPARK_ERR_ALIGNMENT, "slot_mapping must be 8-byte and scales 4-byte aligned");
    }
    if (q_fp8_out && (!(q_fp8_scale > 0.0f) || std::isinf(q_fp8_scale)))
        return fail(DSPARK_ERR_INVALID_ARG, "q_fp8_scale must be positive and finite");
    if (num_tokens == 0)
        return ok();  // nothing to rotate or insert, and no launch
    if (!qkv || !q_norm_w || !k_norm_w || !cos_sin || !positions)
        return fail(DSPARK_ERR_INVALID_ARG, "null buffer pointer");
    if (!aligned(qkv, 16) || !aligned(q_norm_w, 16) || !aligned(k_norm_w, 16) || !aligned(cos_sin, 16) ||
        (q_fp8_out && !aligned(q_fp8_out, 16)))
        return fail(DSPARK_ERR_ALIGNMENT, "qkv, the norm weights, cos_sin and q_fp8_out must be 16-byte aligned");
    if (!aligned(positions, 8))
        return fail(DSPARK_ERR_ALIGNMENT, "positions must be 8-byte aligned");
    if (error_flags && !aligned(error_flags, 4))
        return fail(DSPARK_ERR_ALIGNMENT, "error_flags must be 4-byte aligned");

    dspark::QkInsertParams p{};
    p.qkv = static_cast<uint16_t *>(qkv);
    p.q_norm_w = static_cast<const uint16_t *>(q_norm_w);
    p.k_norm_w = static_cast<const uint16_t *>(k_norm_w);
    p.cos_sin = static_cast<const uint16_t *>(cos_sin);
    p.positions = positions;
    p.slot_mapping = insert ? slot_mapping : nullptr;
    p.cache = insert ? static_cast<unsigned char *>(kv_cache) : nullptr;
    p.k_scale = k_scale;
    p.v_scale = v_scale;
    p.q_fp8 = static_cast<unsigned char *>(q_fp8_out);
    p.error_flags = error_flags;
    p.num_tokens = num_tokens;
    p.max_pos = max_pos;
    p.capacity = capacity;
    p.num_heads = num_heads;
    p.num_kv_heads = num_kv_heads;
    p.block_size_log2 = bsl;
    p.eps = eps;
    p.q_scale = q_fp8_out ? q_fp8_scale : 1.0f;
    const bool fp8 = insert && kv_dtype == DSPARK_KV_FP8_E4M3;
    cudaError_t e = dspark::launch_qk_insert(p, rotary_dim, fp8, stream);
    if (e != cudaSuccess)
        return fail(DSPARK_ERR_CUDA, "launch failed: %s", cudaGetErrorString(e));
    return ok();
}

namespace {

// Shape rules of the tensor-core projection: TMA needs 16-byte aligned bases
// and rows (hidden a multiple of 8 bf16); the grid holds L * nkv column tiles
// by ceil(T / 128) row tiles.
int check_projection(const void *x, const void *w_kv, int64_t num_ctx, int hidden, int L, int nkv)
{
    if (num_ctx < 0)
        return fail(DSPARK_ERR_INVALID_ARG, "num_ctx %lld < 0", (long long)num_ctx);
    if (L <= 0 || nkv <= 0 || (int64_t)L * nkv > 65535)
        return fail(DSPARK_ERR_INVALID_ARG, "L=%d nkv=%d: need 1 <= L * nkv <= 65535", L, nkv);
    if (hidden <= 0 || hidden % 8 != 0)
        return fail(DSPARK_ERR_ALIGNMENT, "hidden %d must be a positive multiple of 8", hidden);
    if (num_ctx > (int64_t)65535 * 128)
        return fail(DSPARK_ERR_INVALID_ARG, "num_ctx %lld above %d", (long long)num_ctx, 65535 * 128);
    if (num_ctx > 0 && (!x || !w_kv))
        return fail(DSPARK_ERR_INVALID_ARG, "null x or w_kv");
    if (num_ctx > 0 && (!aligned(x, 16) || !aligned(w_kv, 16)))
        return fail(DSPARK_ERR_ALIGNMENT, "x and w_kv must be 16-byte aligned");
    return DSPARK_OK;
}

}  // namespace

int dspark_ctx_kv_project(const void *x, const void *w_kv, void *all_kv_out, int64_t num_ctx, int hidden, int L,
                          int nkv, cudaStream_t stream)
{
    int st = check_projection(x, w_kv, num_ctx, hidden, L, nkv);
    if (st != DSPARK_OK)
        return st;
    if (num_ctx == 0)
        return ok();
    if (!all_kv_out || !aligned(all_kv_out, 16))
        return fail(DSPARK_ERR_ALIGNMENT, "all_kv_out must be a 16-byte aligned device buffer");
    dspark::ProjArgs a{};
    a.x = static_cast<const uint16_t *>(x);
    a.w_kv = static_cast<const uint16_t *>(w_kv);
    a.all_kv_out = static_cast<uint16_t *>(all_kv_out);
    a.T = num_ctx;
    a.hidden = hidden;
    a.L = L;
    a.nkv = nkv;
    cudaError_t e = dspark::launch_proj(a, stream);
    if (e != cudaSuccess)
        return fail(DSPARK_ERR_CUDA, "projection launch failed: %s", cudaGetErrorString(e));
    return ok();
}

int dspark_ctx_kv_project_write(const void *x, const void *w_kv, int64_t num_ctx, int hidden, const void *knorm_w,
                                const int64_t *positions, const int64_t *slot_mapping, const void *cos_sin,
                                int64_t max_pos, void *layer0_cache, int64_t num_blocks,
                                const int64_t *cache_offsets, const float *const *k_scales,
                                const float *const *v_scales, int L, int nkv, int block_size, int rotary_dim,
                                float eps, int kv_dtype, unsigned int *error_flags, cudaStream_t stream)
{
    int st = check_projection(x, w_kv, num_ctx, hidden, L, nkv);
    if (st != DSPARK_OK)
        return st;
    if (num_blocks <= 0 || max_pos <= 0)
        return fail(DSPARK_ERR_INVALID_ARG, "num_blocks=%lld max_pos=%lld must be >= 1", (long long)num_blocks,
                    (long long)max_pos);
    if (!dspark_ctx_kv_rotary_dims_supported(rotary_dim, DSPARK_HEAD_DIM))
        return fail(DSPARK_ERR_UNSUPPORTED_ROTARY_DIM, "rotary_dim %d not in {16, 32, 64}", rotary_dim);
    if (!pow2(block_size))
        return fail(DSPARK_ERR_BLOCK_SIZE, "block size %d is not a power of two", block_size);
    if (kv_dtype != DSPARK_KV_BF16 && kv_dtype != DSPARK_KV_FP8_E4M3)
        return fail(DSPARK_ERR_DTYPE, "kv dtype %d unknown", kv_dtype);
    if (!(eps >= 0.0f) || std::isinf(eps))
        return fail(DSPARK_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (L > 32)
        return fail(DSPARK_ERR_INVALID_ARG, "the fused projection write handles at most 32 layers (L=%d)", L);
    const int64_t capacity = num_blocks * (int64_t)block_size;
    if (capacity / block_size != num_blocks || num_blocks > (INT64_MAX / nkv) / block_size / DSPARK_CACHE_ROW)
        return fail(DSPARK_ERR_INVALID_ARG, "cache of %lld blocks too large", (long long)num_blocks);
    if (num_ctx == 0)
        return ok();
    if (!knorm_w || !positions || !slot_mapping || !cos_sin || !layer0_cache || !cache_offsets)
        return fail(DSPARK_ERR_INVALID_ARG, "null buffer pointer");
    if (kv_dtype == DSPARK_KV_FP8_E4M3 && (!k_scales || !v_scales))
        return fail(DSPARK_ERR_INVALID_ARG, "fp8 cache needs k_scales and v_scales");
    if (!aligned(knorm_w, 16) || !aligned(cos_sin, 16) || !aligned(layer0_cache, 16))
        return fail(DSPARK_ERR_ALIGNMENT, "knorm_w, cos_sin and layer0_cache must be 16-byte aligned");
    if (!aligned(positions, 8) || (slot_mapping && !aligned(slot_mapping, 8)) || !aligned(cache_offsets, 8) ||
        (k_scales && !aligned(k_scales, 8)) || (v_scales && !aligned(v_scales, 8)))
        return fail(DSPARK_ERR_ALIGNMENT, "int64 and pointer tables must be 8-byte aligned");
    if (error_flags && !aligned(error_flags, 4))
        return fail(DSPARK_ERR_ALIGNMENT, "error_flags must be 4-byte aligned");
    dspark::ProjArgs a{};
    a.x = static_cast<const uint16_t *>(x);
    a.w_kv = static_cast<const uint16_t *>(w_kv);
    a.knorm_w = static_cast<const uint16_t *>(knorm_w);
    a.positions = positions;
    a.slot_mapping = slot_mapping;
    a.cos_sin = static_cast<const uint16_t *>(cos_sin);
    a.cache0 = static_cast<unsigned char *>(layer0_cache);
    a.cache_offsets = cache_offsets;
    a.k_scales = k_scales;
    a.v_scales = v_scales;
    a.error_flags = error_flags;
    a.T = num_ctx;
    a.max_pos = max_pos;
    a.capacity = capacity;
    a.hidden = hidden;
    a.L = L;
    a.nkv = nkv;
    a.block_size_log2 = log2_exact(block_size);
    a.rotary_dim = rotary_dim;
    a.fp8 = kv_dtype == DSPARK_KV_FP8_E4M3;
    a.eps = eps;
    cudaError_t e = dspark::launch_proj(a, stream);
    if (e != cudaSuccess)
        return fail(DSPARK_ERR_CUDA, "projection launch failed: %s", cudaGetErrorString(e));
    return ok();
}

int dspark_gemma_rms_norm(const void *x, const void *w, void *out, int64_t rows, int hidden, float eps,
                          cudaStream_t stream)
{
    if (rows < 0)
        return fail(DSPARK_ERR_INVALID_ARG, "rows %lld < 0", (long long)rows);
    if (hidden <= 0 || hidden % 8 != 0 || hidden > 8192)
        return fail(DSPARK_ERR_INVALID_ARG, "hidden %d must be a positive multiple of 8, at most 8192", hidden);
    if (!(eps >= 0.0f) || std::isinf(eps))
        return fail(DSPARK_ERR_INVALID_ARG, "eps must be finite and >= 0");
    if (rows > INT64_MAX / hidden / 2)
        return fail(DSPARK_ERR_INVALID_ARG, "rows %lld too large", (long long)rows);
    if (rows == 0)
        return ok();
    if (!x || !w || !out)
        return fail(DSPARK_ERR_INVALID_ARG, "null buffer pointer");
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(out, 16))
        return fail(DSPARK_ERR_ALIGNMENT, "x, w and out must be 16-byte aligned");
    const uintptr_t xb = reinterpret_cast<uintptr_t>(x), ob = reinterpret_cast<uintptr_t>(out);
    const uintptr_t span = (uintptr_t)rows * (uintptr_t)hidden * 2;
    if (xb != ob && xb < ob + span && ob < xb + span)
        return fail(DSPARK_ERR_INVALID_ARG, "out overlaps x without being x");
    cudaError_t e = dspark::launch_gemma_norm(static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(w),
                                              static_cast<uint16_t *>(out), rows, hidden, eps, stream);
    if (e != cudaSuccess)
        return fail(DSPARK_ERR_CUDA, "norm launch failed: %s", cudaGetErrorString(e));
    return ok();
}

}  // extern "C"

namespace {

int validate_layers(int L, const dspark_cache_desc *layers, Rules rules)
{
    if (L <= 0 || !layers)
        return fail(DSPARK_ERR_INVALID_ARG, "no layers");
    const dspark_cache_desc &ref = layers[0];
    for (int l = 0; l < L; l++) {
        const dspark_cache_desc &a = layers[l];
        if (a.kv_dtype != DSPARK_KV_BF16 && a.kv_dtype != DSPARK_KV_FP8_E4M3)
            return fail(DSPARK_ERR_DTYPE, "layer %d: kv_cache_dtype unsupported", l);
        if (!a.data)
            return fail(DSPARK_ERR_INVALID_ARG, "layer %d: KV cache not bound", l);
        const bool row_ok = rules == Rules::pages ? a.shape[3] == DSPARK_CACHE_ROW
                                                  : (a.shape[3] == 128 || a.shape[3] == 256 || a.shape[3] == 512);
        if (a.ndim != 4 || !row_ok)
            return fail(DSPARK_ERR_INVALID_ARG, "layer %d: unexpected cache shape", l);
        for (int d = 0; d < 4; d++)
            if (a.shape[d] <= 0)
                return fail(DSPARK_ERR_INVALID_ARG, "layer %d: KV cache not bound (empty)", l);
        if (rules == Rules::pages && !pow2(a.shape[2]))
            return fail(DSPARK_ERR_BLOCK_SIZE, "layer %d: block size %lld is not a power of two", l,
                        (long long)a.shape[2]);
        int64_t expect = 1;
        for (int d = 3; d >= 0; d--) {
            if (a.shape[d] != 1 && a.stride[d] != expect)
                return fail(DSPARK_ERR_INVALID_ARG, "layer %d: cache is not contiguous", l);
            expect *= a.shape[d];
        }
        if (a.kv_dtype == DSPARK_KV_FP8_E4M3) {
            if (a.cache_dtype != DSPARK_KV_FP8_E4M3 || a.elem_size != 1)
                return fail(DSPARK_ERR_DTYPE, "layer %d: fp8 cache is not uint8", l);
        } else if (a.cache_dtype != DSPARK_KV_BF16 || a.elem_size != 2) {
            return fail(DSPARK_ERR_DTYPE, "layer %d: cache is not bf16", l);
        }
        if (!a.scales_ok || !a.k_scale || !a.v_scale)
            return fail(DSPARK_ERR_INVALID_ARG, "layer %d: k/v scale is not a CUDA fp32 tensor", l);
        bool same = a.ndim == ref.ndim && a.elem_size == ref.elem_size &&
                    a.cache_dtype == ref.cache_dtype && a.kv_dtype == ref.kv_dtype;
        for (int d = 0; d < 4; d++)
            same = same && a.shape[d] == ref.shape[d] && a.stride[d] == ref.stride[d];
        if (!same)
            return fail(DSPARK_ERR_INVALID_ARG, "layers do not share cache shape/stride/dtype");
        const int64_t delta = (int64_t)(reinterpret_cast<uintptr_t>(a.data) - reinterpret_cast<uintptr_t>(ref.data));
        if (delta % (16 * (int64_t)a.elem_size) != 0)
            return fail(DSPARK_ERR_ALIGNMENT, "layer caches are not 16-element aligned to each other");
    }
    return ok();
}

}  // namespace

extern "C" {

int dspark_ctx_kv_validate_layers(int L, const dspark_cache_desc *layers)
{
    return validate_layers(L, layers, Rules::pages);
}

int dspark_ctx_kv_validate_layers_general(int L, const dspark_cache_desc *layers)
{
    return validate_layers(L, layers, Rules::general);
}

}  // extern "C"

// --------------------------------------------------------------------------
// Offset / pointer tables.

struct dspark_ctx_kv_tables {
    int L = 0;
    int device = -1;
    int64_t *d_offsets = nullptr;         // [L]
    const float **d_scales = nullptr;     // [2L]: k then v
    const int64_t **d_slots = nullptr;    // [L]: per-layer slot mappings
    std::vector<uintptr_t> key;           // caches, k scales, v scales, elem size
    std::vector<uintptr_t> slot_key;      // per-layer slot mapping addresses
    int64_t builds = 0;
};

extern "C" {

int dspark_ctx_kv_tables_create(int L, dspark_ctx_kv_tables **out)
{
    if (!out || L <= 0)
        return fail(DSPARK_ERR_INVALID_ARG, "tables_create: L=%d", L);
    *out = nullptr;
    auto *t = new (std::nothrow) dspark_ctx_kv_tables();
    if (!t)
        return fail(DSPARK_ERR_INVALID_ARG, "tables_create: out of host memory");
    t->L = L;
    cudaError_t e = cudaGetDevice(&t->device);
    if (e == cudaSuccess)
        e = cudaMalloc(reinterpret_cast<void **>(&t->d_offsets), sizeof(int64_t) * L);
    if (e == cudaSuccess)
        e = cudaMalloc(reinterpret_cast<void **>(&t->d_scales), sizeof(float *) * 2 * L);
    if (e == cudaSuccess)
        e = cudaMalloc(reinterpret_cast<void **>(&t->d_slots), sizeof(int64_t *) * L);
    if (e != cudaSuccess) {
        cudaFree(t->d_offsets);
        cudaFree(t->d_scales);
        delete t;
        return fail(DSPARK_ERR_CUDA, "tables_create: %s", cudaGetErrorString(e));
    }
    *out = t;
    return ok();
}

int dspark_ctx_kv_tables_update(dspark_ctx_kv_tables *t, void *const *layer_caches, size_t elem_size,
                                const float *const *k_scale_ptrs, const float *const *v_scale_ptrs,
                                cudaStream_t stream)
{
    if (!t || !layer_caches)
        return fail(DSPARK_ERR_INVALID_ARG, "tables_update: null argument");
    if (elem_size != 1 && elem_size != 2)
        return fail(DSPARK_ERR_DTYPE, "tables_update: element size %zu", elem_size);
    const int L = t->L;
    std::vector<uintptr_t> key(3 * L + 1);
    for (int l = 0; l < L; l++) {
        key[l] = reinterpret_cast<uintptr_t>(layer_caches[l]);
        key[L + l] = k_scale_ptrs ? reinterpret_cast<uintptr_t>(k_scale_ptrs[l]) : 0;
        key[2 * L + l] = v_scale_ptrs ? reinterpret_cast<uintptr_t>(v_scale_ptrs[l]) : 0;
    }
    key[3 * L] = elem_size;
    if (key == t->key)
        return ok();  // same memory as the tables already describe
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess)
        return fail(DSPARK_ERR_CUDA, "tables_update: %s", cudaGetErrorString(e));
    if (cap != cudaStreamCaptureStatusNone)
        return fail(DSPARK_ERR_CAPTURING, "tables_update: the caches moved while the stream is capturing");
    std::vector<int64_t> offs(L);
    std::vector<const float *> scales(2 * L);
    const uintptr_t base = key[0];
    for (int l = 0; l < L; l++) {
        if (!key[l])
            return fail(DSPARK_ERR_INVALID_ARG, "tables_update: layer %d cache is null", l);
        const int64_t delta = (int64_t)(key[l] - base);
        if (delta % (int64_t)(16 * elem_size) != 0)
            return fail(DSPARK_ERR_ALIGNMENT, "layer caches are not 16-element aligned to each other");
        offs[l] = delta / (int64_t)elem_size;
        scales[l] = k_scale_ptrs ? k_scale_ptrs[l] : nullptr;
        scales[L + l] = v_scale_ptrs ? v_scale_ptrs[l] : nullptr;
    }
    // Pageable host source: the call returns once the bytes are staged, so
    // the vectors may go out of scope; the copies are ordered on `stream`.
    e = cudaMemcpyAsync(t->d_offsets, offs.data(), sizeof(int64_t) * L, cudaMemcpyHostToDevice, stream);
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(t->d_scales, scales.data(), sizeof(float *) * 2 * L, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess)
        return fail(DSPARK_ERR_CUDA, "tables_update: %s", cudaGetErrorString(e));
    t->key.swap(key);
    t->builds++;
    return ok();
}

int dspark_ctx_kv_tables_update_slots(dspark_ctx_kv_tables *t, const int64_t *const *layer_slot_ptrs,
                                      cudaStream_t stream)
{
    if (!t || !layer_slot_ptrs)
        return fail(DSPARK_ERR_INVALID_ARG, "tables_update_slots: null argument");
    const int L = t->L;
    std::vector<uintptr_t> key(L);
    for (int l = 0; l < L; l++) {
        key[l] = reinterpret_cast<uintptr_t>(layer_slot_ptrs[l]);
        if (!key[l] || key[l] % 8)
            return fail(DSPARK_ERR_INVALID_ARG, "tables_update_slots: layer %d mapping null or misaligned", l);
    }
    if (key == t->slot_key)
        return ok();  // the same mappings as the table already holds
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cap);
    if (e != cudaSuccess)
        return fail(DSPARK_ERR_CUDA, "tables_update_slots: %s", cudaGetErrorString(e));
    if (cap != cudaStreamCaptureStatusNone)
        return fail(DSPARK_ERR_CAPTURING, "tables_update_slots: the slot mappings moved while the stream is capturing");
    e = cudaMemcpyAsync(t->d_slots, layer_slot_ptrs, sizeof(int64_t *) * L, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess)
        return fail(DSPARK_ERR_CUDA, "tables_update_slots: %s", cudaGetErrorString(e));
    t->slot_key.swap(key);
    t->builds++;
    return ok();
}

const int64_t *const *dspark_ctx_kv_tables_layer_slots(const dspark_ctx_kv_tables *t)
{
    return t ? t->d_slots : nullptr;
}

const int64_t *dspark_ctx_kv_tables_cache_offsets(const dspark_ctx_kv_tables *t)
{
    return t ? t->d_offsets : nullptr;
}

const float *const *dspark_ctx_kv_tables_k_scales(const dspark_ctx_kv_tables *t)
{
    return t ? t->d_scales : nullptr;
}

const float *const *dspark_ctx_kv_tables_v_scales(const dspark_ctx_kv_tables *t)
{
    return t ? t->d_scales + t->L : nullptr;
}

int64_t dspark_ctx_kv_tables_builds(const dspark_ctx_kv_tables *t) { return t ? t->builds : 0; }

void dspark_ctx_kv_tables_destroy(dspark_ctx_kv_tables *t)
{
    if (!t)
        return;
    int prev = -1;
    bool switched = cudaGetDevice(&prev) == cudaSuccess && prev != t->device && t->device >= 0 &&
                    cudaSetDevice(t->device) == cudaSuccess;
    cudaFree(t->d_offsets);
    cudaFree(t->d_scales);
    cudaFree(t->d_slots);
    if (switched)
        cudaSetDevice(prev);
    delete t;
}

}  // extern "C"
