// The context-KV write with no allocation: the per-layer tables the kernels
// read (cache offsets, scale pointers, per-layer slot-mapping pointers) and
// the work counter of the dynamic tail live in one file-scope device array
// of fixed size instead of in memory that the caller or the tables object
// allocates.  Each call copies its tables, with the counter's zeros, from
// host memory into that array on the call's stream, then runs
// dspark_ctx_kv_write_sched on it.  The vLLM DSpark context-KV writer page
// has no counterpart (its tables are framework tensors).

#include <cinttypes>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "ctx_kv_internal.h"
#include "dspark_ctx_kv.h"

namespace {

constexpr int kMaxLayers = DSPARK_NOALLOC_MAX_LAYERS;
// words: [0, 2) work counter {claimed, finished}; then offsets, k_scales,
// v_scales and layer slot-mapping pointers, kMaxLayers words each
constexpr int kCounter = 0, kOffsets = 2, kKScales = kOffsets + kMaxLayers, kVScales = kKScales + kMaxLayers,
              kSlots = kVScales + kMaxLayers, kWords = kSlots + kMaxLayers;
static_assert(kWords * 8 == 16 + 32 * kMaxLayers, "scratch layout");

static __device__ __align__(256) unsigned long long g_noalloc_scratch[kWords];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
unsigned long long *g_scratch[kMaxDevices];  // device address of the array, per device (null: not set up)

// The array's device address on the current device, found once per device.
cudaError_t scratch_address(unsigned long long **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch[dev]) {
        void *a = nullptr;
        e = cudaGetSymbolAddress(&a, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        g_scratch[dev] = static_cast<unsigned long long *>(a);
    }
    *out = g_scratch[dev];
    return cudaSuccess;
}

uint64_t word(const void *p)
{
    uint64_t w = 0;
    static_assert(sizeof(p) == sizeof(w), "64-bit pointers");
    std::memcpy(&w, &p, sizeof w);
    return w;
}

}  // namespace

extern "C" int dspark_ctx_kv_write_noalloc(const void *all_kv, const void *knorm_w, const int64_t *positions,
                                           const int64_t *slot_mapping,
                                           const int64_t *const *layer_slot_mappings_host, int64_t num_ctx,
                                           const void *cos_sin, int64_t max_pos, void *layer0_cache,
                                           int64_t num_blocks, const int64_t *cache_offsets_host,
                                           const float *const *k_scales_host, const float *const *v_scales_host,
                                           int L, int nkv, int block_size, int rotary_dim, float eps, int kv_dtype,
                                           unsigned int *error_flags, cudaStream_t stream)
{
    char msg[160];
    if (L < 1 || L > kMaxLayers) {
        std::snprintf(msg, sizeof msg, "L=%d: the no-allocation write takes 1 to %d layers", L, kMaxLayers);
        return dspark::api_fail(DSPARK_ERR_INVALID_ARG, msg);
    }
    if (num_ctx <= 0)  // the scalar checks, and nothing to store
        return dspark_ctx_kv_write_sched(all_kv, knorm_w, positions, slot_mapping, nullptr, num_ctx, cos_sin,
                                         max_pos, layer0_cache, num_blocks, nullptr, nullptr, nullptr, L, nkv,
                                         block_size, rotary_dim, eps, kv_dtype, error_flags, nullptr, stream);
    if ((slot_mapping == nullptr) == (layer_slot_mappings_host == nullptr))
        return dspark::api_fail(DSPARK_ERR_INVALID_ARG, "give exactly one of slot_mapping and layer_slot_mappings");
    if (!cache_offsets_host)
        return dspark::api_fail(DSPARK_ERR_INVALID_ARG, "null cache_offsets");
    const bool fp8 = kv_dtype == DSPARK_KV_FP8_E4M3;
    if (fp8 && (!k_scales_host || !v_scales_host))
        return dspark::api_fail(DSPARK_ERR_INVALID_ARG, "fp8 cache needs k_scales and v_scales");

    // the call's tables, host side: zeros for the counter and unused words
    uint64_t h[kWords] = {};
    for (int l = 0; l < L; l++) {
        const int64_t off = cache_offsets_host[l];
        if (off % 16 != 0) {
            std::snprintf(msg, sizeof msg, "cache_offsets[%d] = %" PRId64 " is not a multiple of 16 elements", l,
                          off);
            return dspark::api_fail(DSPARK_ERR_ALIGNMENT, msg);
        }
        std::memcpy(&h[kOffsets + l], &off, sizeof off);
        if (k_scales_host)
            h[kKScales + l] = word(k_scales_host[l]);
        if (v_scales_host)
            h[kVScales + l] = word(v_scales_host[l]);
        if (layer_slot_mappings_host) {
            if (!layer_slot_mappings_host[l])
                return dspark::api_fail(DSPARK_ERR_INVALID_ARG, "null per-layer slot mapping");
            h[kSlots + l] = word(layer_slot_mappings_host[l]);
        }
    }
    unsigned long long *d = nullptr;
    cudaError_t e = scratch_address(&d);
    if (e != cudaSuccess) {
        std::snprintf(msg, sizeof msg, "no-allocation scratch: %s", cudaGetErrorString(e));
        return dspark::api_fail(DSPARK_ERR_CUDA, msg);
    }
    // stream-ordered after every earlier call on `stream` and before this
    // launch; the host copy is staged before the call returns
    e = cudaMemcpyAsync(d, h, sizeof h, cudaMemcpyHostToDevice, stream);
    if (e != cudaSuccess) {
        std::snprintf(msg, sizeof msg, "no-allocation scratch copy: %s", cudaGetErrorString(e));
        return dspark::api_fail(DSPARK_ERR_CUDA, msg);
    }
    const float *const *ks = k_scales_host ? reinterpret_cast<const float *const *>(d + kKScales) : nullptr;
    const float *const *vs = v_scales_host ? reinterpret_cast<const float *const *>(d + kVScales) : nullptr;
    const int64_t *const *ls =
        layer_slot_mappings_host ? reinterpret_cast<const int64_t *const *>(d + kSlots) : nullptr;
    return dspark_ctx_kv_write_sched(all_kv, knorm_w, positions, slot_mapping, ls, num_ctx, cos_sin, max_pos,
                                     layer0_cache, num_blocks, reinterpret_cast<const int64_t *>(d + kOffsets), ks,
                                     vs, L, nkv, block_size, rotary_dim, eps, kv_dtype, error_flags, d + kCounter,
                                     stream);
}
