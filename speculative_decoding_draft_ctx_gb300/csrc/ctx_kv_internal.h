// Internal interface between the C-ABI host layer (ctx_kv_api.cpp) and the
// sm_103a kernels (ctx_kv_kernel.cu).  Not part of the public ABI.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

namespace dspark {

constexpr int kHeadDim = 128;
constexpr int kRowElems = 256;

// Everything one launch reads; all pointers are device pointers and have
// been validated (non-null, aligned) by the host layer.
struct CtxKvParams {
    const uint16_t *all_kv;      // bf16 bits [T, L, 2, H, 128]
    const uint16_t *knorm_w;     // bf16 bits [L, 128]
    const int64_t *positions;    // [T]
    const int64_t *slot_mapping; // [T]
    const uint16_t *cos_sin;     // bf16 bits [max_pos, rotary_dim]
    unsigned char *cache0;       // layer 0 cache base
    const int64_t *cache_offsets;     // [L] element offsets
    const float *const *k_scales;     // [L] (fp8 only)
    const float *const *v_scales;     // [L] (fp8 only)
    unsigned int *error_flags;        // may be null
    int64_t num_ctx;
    int64_t max_pos;
    int64_t capacity;            // num_blocks * block_size
    int32_t num_layers;
    int32_t num_kv_heads;
    int32_t head_chunks;         // ceil(num_kv_heads / heads per unit)
    int32_t block_size_log2;
    float eps;
};

// Generic kernel (any layer count and head count): enqueues the write on
// `stream`.  Returns cudaSuccess or the launch error.
cudaError_t launch_ctx_kv_write(const CtxKvParams &p, int rotary_dim, bool fp8, cudaStream_t stream);

// Pipelined bulk-copy kernel: handles up to 32 layers and up to 64 KV heads
// (one layer's K|V rows of a token fit a 32 KB stage).
bool tma_path_supported(const CtxKvParams &p);
cudaError_t launch_ctx_kv_write_tma(const CtxKvParams &p, int rotary_dim, bool fp8, cudaStream_t stream);

}  // namespace dspark
