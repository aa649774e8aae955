// Internal interface between the C-ABI host layer (ctx_kv_api.cpp) and the
// sm_103a kernels (ctx_kv_kernel.cu).  Not part of the public ABI.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include <cuda_runtime_api.h>

#ifdef __CUDACC__
#include <cstdlib>
#include <cstring>
#include <utility>

#include <cuda_runtime.h>
#endif

namespace dspark {

#ifdef __CUDACC__
// Launches `kernel` with programmatic stream serialization allowed, so that
// it may start while the previous kernel of the stream drains (the kernel
// itself executes griddepcontrol.wait before touching global memory).
// DSPARK_PDL=0 launches it the plain way.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), int blocks, int threads, size_t smem, cudaStream_t stream,
                       Args &&...args)
{
    const char *env = std::getenv("DSPARK_PDL");
    const bool pdl = !(env && std::strcmp(env, "0") == 0);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3((unsigned)threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// The kernel side of launch_pdl, before any global load or store (L2
// prefetch hints may precede it: they hand no data to the program): wait for
// the stream's previous kernel to finish and its writes to be visible, then
// let the next kernel be scheduled as this grid's CTAs exit (it is scheduled
// only once every CTA of this grid has issued this or exited, so it never
// takes a slot one of ours still waits for).
__device__ __forceinline__ void pdl_enter()
{
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
#endif

// Records `message` as the calling thread's last error (what
// dspark_ctx_kv_last_error returns) and returns `status`: for entry points
// defined outside the host layer.
int api_fail(int status, const char *message);

constexpr int kHeadDim = 128;
constexpr int kRowElems = 256;

// Everything one launch reads; all pointers are device pointers and have
// been validated (non-null, aligned) by the host layer.
struct CtxKvParams {
    const uint16_t *all_kv;      // bf16 bits [T, L, 2, H, 128]
    const uint16_t *knorm_w;     // bf16 bits [L, 128]
    const int64_t *positions;    // [T]
    const int64_t *slot_mapping; // [T], shared by every layer (unused when layer_slots is set)
    const int64_t *const *layer_slots; // [L] device pointers to per-layer [T] slot mappings, or null
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
    int32_t block_size_log2;     // -1 (general kernel only): not a power of two
    float eps;
    // general kernel only (launch_ctx_kv_general)
    int32_t rotary_dim;          // even, 2..head_dim
    int32_t block_size;
    int32_t bs_magic_shift;      // block = umulhi(slot, bs_magic) >> bs_magic_shift
    uint64_t bs_magic;           //   when block_size_log2 < 0
    // test hook of the pipelined and warp-private kernels (0: off): the
    // producer (every warp) first waits this many ns on a device word that
    // nothing sets, then gives up as on any expired wait
    // (DSPARK_FLAG_TIMEOUT, nothing written)
    uint64_t test_hold_ns;
    // pipelined kernel: a device pair {claimed, finished} (zero between
    // launches) for handing out the tail of the units dynamically, or null
    unsigned long long *work_counter;
};

// Generic kernel (any layer count and head count): enqueues the write on
// `stream`.  Returns cudaSuccess or the launch error.
cudaError_t launch_ctx_kv_write(const CtxKvParams &p, int rotary_dim, bool fp8, cudaStream_t stream);

// The write for head dims 64, 128 and 256, any even rotary_dim up to the
// head dim and any block size (ctx_kv_general.cu): all_kv [T, L, 2, H, D],
// knorm_w [L, D], cache rows of 2D elements.
cudaError_t launch_ctx_kv_general(const CtxKvParams &p, int head_dim, bool fp8, cudaStream_t stream);

// Pipelined bulk-copy kernel: head dims 64, 128 and 256, any even rotary dim
// up to the head dim (p.rotary_dim), any block size; up to 32 layers, and one
// layer's K|V rows of a token must fit a 32 KB stage (nkv * 4 * head_dim
// bytes); a shared or a per-layer slot mapping.
bool tma_path_supported(const CtxKvParams &p, int head_dim);
cudaError_t launch_ctx_kv_write_tma(const CtxKvParams &p, int head_dim, bool fp8, cudaStream_t stream);

// Warp-private pipelines (ctx_kv_warp.cu): head dim 128, rotary dim 16 / 32 /
// 64, power-of-two block sizes, 4 or 8 KV heads, any layer count, a shared
// slot mapping.
bool warp_path_supported(const CtxKvParams &p);
cudaError_t launch_ctx_kv_write_warp(const CtxKvParams &p, bool fp8, cudaStream_t stream);

// Draft-token fused QK-norm / RoPE / KV insert (qk_insert_kernel.cu).
struct QkInsertParams {
    uint16_t *qkv;               // bf16 bits [T, (Hq + 2 Hkv) * 128], updated in place
    const uint16_t *q_norm_w;    // bf16 bits [128]
    const uint16_t *k_norm_w;    // bf16 bits [128]
    const uint16_t *cos_sin;     // bf16 bits [max_pos, rotary_dim]
    const int64_t *positions;    // [T]
    const int64_t *slot_mapping; // [T] or null (no insert)
    unsigned char *cache;        // [num_blocks, Hkv, block_size, 256] or null (no insert)
    const float *k_scale;        // fp8 cache: device fp32 scalars (null = 1)
    const float *v_scale;
    unsigned char *q_fp8;        // [T, Hq * 128] e4m3 codes, or null
    unsigned int *error_flags;   // may be null
    int64_t num_tokens;
    int64_t max_pos;
    int64_t capacity;            // num_blocks * block_size
    int32_t num_heads;
    int32_t num_kv_heads;
    int32_t block_size_log2;
    float eps;
    float q_scale;
};

cudaError_t launch_qk_insert(const QkInsertParams &p, int rotary_dim, bool fp8_cache, cudaStream_t stream);

// Fused context-KV projection (proj_gemm.cu): all_kv = bf16(x w^T) on the
// tensor cores, stored to all_kv_out, or (all_kv_out null) written straight
// into the caches by the context-KV write in the GEMM's epilogue.
struct ProjArgs {
    const uint16_t *x;           // bf16 [T, hidden]
    const uint16_t *w_kv;        // bf16 [L * 2 * nkv * 128, hidden]
    uint16_t *all_kv_out;        // bf16 [T, L * 2 * nkv * 128], or null: write
    const uint16_t *knorm_w;     // write: bf16 [L, 128]
    const int64_t *positions;
    const int64_t *slot_mapping;
    const uint16_t *cos_sin;
    unsigned char *cache0;
    const int64_t *cache_offsets;
    const float *const *k_scales;
    const float *const *v_scales;
    unsigned int *error_flags;
    int64_t T;
    int64_t max_pos;
    int64_t capacity;
    int32_t hidden;
    int32_t L;
    int32_t nkv;
    int32_t block_size_log2;
    int32_t rotary_dim;
    bool fp8;
    float eps;
};

cudaError_t launch_proj(const ProjArgs &a, cudaStream_t stream);

// Hidden-state Gemma RMSNorm (hidden_norm.cu): rows of hidden bf16 values,
// hidden a multiple of 8 and at most 8192; out may equal x.
cudaError_t launch_gemma_norm(const uint16_t *x, const uint16_t *w, uint16_t *out, int64_t rows, int hidden,
                              float eps, cudaStream_t stream);

}  // namespace dspark
