// sm_103a kernel of the DSpark fused context-KV write.
//
// Defining passage: vLLM DSpark context-KV writer page, module docstring (one
// launch for all draft layers: Gemma RMSNorm of K in fp32 materialised to
// bf16, partial NeoX RoPE at the token's position, store of K|V into each
// layer's [num_blocks, nkv, block_size, 256] cache as bf16 or fp8 e4m3 of
// x / scale, slots < 0 not written).
//
// Work decomposition.  A unit is (token t, layer l, a chunk of up to four KV
// heads).  One warp processes one unit at a time, grid-striding over units in
// token-major order so that consecutive warps stream consecutive all_kv
// bytes.  Within the warp, lanes 0..15 hold K and lanes 16..31 hold V of the
// same head, 8 bf16 (16 bytes) each: one 16-byte load per lane fetches a whole
// 512-byte K|V row (four full 128-byte lines), and one 16-byte (bf16) or
// 8-byte (fp8) store per lane writes the row's contiguous 512 / 256 bytes of
// cache.  The four heads of a unit are loaded before any is used, so each
// lane keeps 64 bytes in flight.  Nothing here is a contraction: the kernel is
// bound by HBM bandwidth, and the tensor cores have no role.
//
// Per row:
//   sum of squares over K: 8 FMAs per lane, then a 4-step xor shuffle within
//     the 16 K lanes (the V lanes run the same instructions on V and discard
//     them, which keeps the warp converged at no extra issue cost);
//   y = bf16((k * rsqrt(ss/128 + eps)) * (1 + w)) in fp32;
//   RoPE: the rotated partner of dim d (d < r) is d +- r/2, which lives
//     r/16 lanes away, so one xor shuffle of the packed bf16 pairs brings it
//     in; out = y*c -+ y_partner*s with one fused multiply-add (the product
//     y_partner*s of two bf16 values is exact in fp32);
//   fp8: x / scale as an IEEE fp32 division, then a saturating RNE pack to
//     e4m3 pairs (cvt.rn.satfinite.e4m3x2.f32 via cuda_fp8.h).
// With per-layer slot mappings the slot of (t, l) comes from layer l's
// mapping (a device pointer table).  Rows whose slot or position is out of
// range are skipped and reported
// through the optional error word; no access leaves the caller's buffers.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ctx_kv_internal.h"

namespace dspark {
namespace {

constexpr int kThreads = 256;
constexpr int kHeadsPerUnit = 4;
constexpr unsigned kFlagSlot = 0x1u;
constexpr unsigned kFlagPos = 0x2u;

__device__ __forceinline__ uint4 ld_stream_v4(const void *p)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ void st_stream_v4(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_stream_v2(void *p, uint2 v)
{
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// bf16 element 2j of a packed word is its low half, 2j+1 its high half.
__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8])
{
    f[0] = bf_lo(v.x), f[1] = bf_hi(v.x), f[2] = bf_lo(v.y), f[3] = bf_hi(v.y);
    f[4] = bf_lo(v.z), f[5] = bf_hi(v.z), f[6] = bf_lo(v.w), f[7] = bf_hi(v.w);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d)
{
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

__device__ __forceinline__ uint2 quantise8(const float (&f)[8], float scale)
{
    float q[8];
#pragma unroll
    for (int j = 0; j < 8; j++)
        q[j] = __fdiv_rn(f[j], scale);
    return make_uint2(pack_e4m3x4(q[0], q[1], q[2], q[3]), pack_e4m3x4(q[4], q[5], q[6], q[7]));
}

__device__ __forceinline__ float load_scale(const float *const *table, int l)
{
    const float *p = reinterpret_cast<const float *>(
        __ldg(reinterpret_cast<const unsigned long long *>(table) + l));
    return __ldg(p);
}

template <int ROT, bool FP8>
__global__ void __launch_bounds__(kThreads) ctx_kv_write_kernel(const CtxKvParams p)
{
    pdl_enter();
    constexpr int kRotLanes = ROT / 8;  // K lanes holding rotary dims
    constexpr int kPartner = ROT / 16;  // lane distance of a rotated pair
    const int lane = threadIdx.x & 31;
    const int kv = lane >> 4;  // 0: K lane, 1: V lane
    const int q = lane & 15;   // 8-element chunk of the 128-dim head
    const bool rot_lane = kv == 0 && q < kRotLanes;
    const float sgn = (q & kPartner) ? 1.0f : -1.0f;  // upper half adds, lower subtracts

    const int L = p.num_layers, H = p.num_kv_heads, HC = p.head_chunks;
    const int64_t per_tok = (int64_t)L * HC;
    const int64_t units = p.num_ctx * per_tok;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t bs_mask = (int64_t(1) << p.block_size_log2) - 1;
    unsigned flags = 0;

    for (int64_t u = warp; u < units; u += nwarps) {
        const int64_t t = u / per_tok;
        const int rem = (int)(u - t * per_tok);
        const int l = rem / HC;
        const int h0 = (rem - l * HC) * kHeadsPerUnit;
        const int nh = min(kHeadsPerUnit, H - h0);
        const int64_t slot =
            p.layer_slots ? __ldg(reinterpret_cast<const int64_t *>(__ldg(
                                reinterpret_cast<const unsigned long long *>(p.layer_slots) + l)) + t)
                          : __ldg(p.slot_mapping + t);
        if (slot < 0)
            continue;  // padding: neither read nor written
        const int64_t pos = __ldg(p.positions + t);
        if (slot >= p.capacity) {
            flags |= kFlagSlot;
            continue;
        }
        if (pos < 0 || pos >= p.max_pos) {
            flags |= kFlagPos;
            continue;
        }

        const uint16_t *src = p.all_kv + ((((t * L + l) * 2 + kv) * H + h0) * kHeadDim + q * 8);
        uint4 x[kHeadsPerUnit];
#pragma unroll
        for (int i = 0; i < kHeadsPerUnit; i++)
            if (i < nh)
                x[i] = ld_stream_v4(src + i * kHeadDim);

        const uint4 wr = __ldg(reinterpret_cast<const uint4 *>(p.knorm_w + l * kHeadDim + q * 8));
        uint4 cr = make_uint4(0, 0, 0, 0), sr = cr;
        if (rot_lane) {
            const uint16_t *cs = p.cos_sin + pos * ROT + (q & (kPartner - 1)) * 8;
            cr = __ldg(reinterpret_cast<const uint4 *>(cs));
            sr = __ldg(reinterpret_cast<const uint4 *>(cs + ROT / 2));
        }
        const int64_t layer_off = __ldg(p.cache_offsets + l);
        float ksc = 1.0f, vsc = 1.0f;
        if (FP8) {
            ksc = load_scale(p.k_scales, l);
            vsc = load_scale(p.v_scales, l);
        }

        float w1[8], c[8], s[8];
        unpack8(wr, w1);
#pragma unroll
        for (int j = 0; j < 8; j++)
            w1[j] = 1.0f + w1[j];
        unpack8(cr, c);
        unpack8(sr, s);

        const int64_t row0 = ((slot >> p.block_size_log2) * H + h0) * ((int64_t)bs_mask + 1) + (slot & bs_mask);
        const int64_t head_stride = bs_mask + 1;  // rows between consecutive heads

#pragma unroll
        for (int i = 0; i < kHeadsPerUnit; i++) {
            if (i >= nh)
                break;
            float f[8];
            unpack8(x[i], f);
            float ss = 0.0f;
#pragma unroll
            for (int j = 0; j < 8; j++)
                ss = fmaf(f[j], f[j], ss);
            ss += __shfl_xor_sync(0xffffffffu, ss, 8);
            ss += __shfl_xor_sync(0xffffffffu, ss, 4);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            const float inv = rsqrtf(fmaf(ss, 1.0f / kHeadDim, p.eps));

            uint32_t y[4];
#pragma unroll
            for (int j = 0; j < 4; j++)
                y[j] = pack_bf16x2((f[2 * j] * inv) * w1[2 * j], (f[2 * j + 1] * inv) * w1[2 * j + 1]);
            uint32_t yp[4];
#pragma unroll
            for (int j = 0; j < 4; j++)
                yp[j] = __shfl_xor_sync(0xffffffffu, y[j], kPartner);

            uint32_t ko[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const float a0 = fmaf(bf_lo(y[j]), c[2 * j], sgn * (bf_lo(yp[j]) * s[2 * j]));
                const float a1 = fmaf(bf_hi(y[j]), c[2 * j + 1], sgn * (bf_hi(yp[j]) * s[2 * j + 1]));
                ko[j] = rot_lane ? pack_bf16x2(a0, a1) : y[j];
            }

            const int64_t elem = layer_off + (row0 + i * head_stride) * kRowElems;
            if (!FP8) {
                const uint4 out = kv == 0 ? make_uint4(ko[0], ko[1], ko[2], ko[3]) : x[i];
                st_stream_v4(p.cache0 + elem * 2 + lane * 16, out);
            } else {
                float o[8];
                if (kv == 0) {
                    unpack8(make_uint4(ko[0], ko[1], ko[2], ko[3]), o);
                } else {
#pragma unroll
                    for (int j = 0; j < 8; j++)
                        o[j] = f[j];
                }
                st_stream_v2(p.cache0 + elem + lane * 8, quantise8(o, kv == 0 ? ksc : vsc));
            }
        }
    }
    if (flags && lane == 0 && p.error_flags)
        atomicOr(p.error_flags, flags);
}

template <int ROT, bool FP8>
cudaError_t launch_variant(const CtxKvParams &p, cudaStream_t stream)
{
    // Resident blocks per SM and SM count, per device (queried once).
    static std::mutex mu;
    static int cached_blocks[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    int max_blocks;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (dev < 0 || dev >= 64)
            return cudaErrorInvalidDevice;
        if (cached_blocks[dev] == 0) {
            int sms = 0, per_sm = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess)
                return e;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ctx_kv_write_kernel<ROT, FP8>,
                                                              kThreads, 0);
            if (e != cudaSuccess)
                return e;
            cached_blocks[dev] = sms * (per_sm > 0 ? per_sm : 1);
        }
        max_blocks = cached_blocks[dev];
    }
    const int64_t units = p.num_ctx * (int64_t)p.num_layers * p.head_chunks;
    const int64_t warps_per_block = kThreads / 32;
    const int64_t need = (units + warps_per_block - 1) / warps_per_block;
    const int blocks = (int)(need < max_blocks ? need : max_blocks);
    return launch_pdl(ctx_kv_write_kernel<ROT, FP8>, blocks, kThreads, 0, stream, p);
}

}  // namespace

cudaError_t launch_ctx_kv_write(const CtxKvParams &p, int rotary_dim, bool fp8, cudaStream_t stream)
{
    CtxKvParams q = p;
    q.head_chunks = (p.num_kv_heads + kHeadsPerUnit - 1) / kHeadsPerUnit;
    switch (rotary_dim) {
    case 16:
        return fp8 ? launch_variant<16, true>(q, stream) : launch_variant<16, false>(q, stream);
    case 32:
        return fp8 ? launch_variant<32, true>(q, stream) : launch_variant<32, false>(q, stream);
    case 64:
        return fp8 ? launch_variant<64, true>(q, stream) : launch_variant<64, false>(q, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace dspark
