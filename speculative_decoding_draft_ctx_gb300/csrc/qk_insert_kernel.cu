// sm_103a kernel of the DSpark draft-token fused QK-norm / RoPE / KV insert.
//
// Defining passage: DSpark draft model page, dspark_qknorm_rope_kv_insert
// (the fused QK-norm/RoPE on qkv, also storing the draft tokens' k/v; its
// arguments qkv, q_norm_weight, k_norm_weight, cos_sin_cache, positions,
// num_heads, num_kv_heads, rotary_dim, eps, slot_mapping, kv_cache,
// block_size, kv_cache_dtype, q_fp8_out, q_fp8_scale), with the norm, RoPE,
// cache layout and fp8 rule of the context-KV writer page.
//
// Work decomposition.  qkv is [T, W * 128] bf16 with W = Hq + 2 Hkv heads per
// token (queries, keys, values).  A CTA takes one token at a time (grid
// stride over tokens, so no index division); its warps split the token's
// heads in groups of four, 8 lanes per head: lane q of a head holds dims
// [8q, 8q + 8) and [64 + 8q, 64 + 8q + 8), two 16-byte words, so one load
// instruction of a warp reads four whole 128-byte halves of heads.  A warp
// issues the loads of up to kBatch of its groups before it computes.  A
// query or key head is normed (sum of squares on paired fp32 FMAs, then 3
// xor shuffles inside the head's 8 lanes), rotated (RoPE acts on dims < 64;
// the partner of dim d < r/2 is d + r/2, r/16 lanes away; fma.rn.f32.bf16 on
// the bf16 halves: the partner product is exact, one rounding) and written
// back in place; a query head also goes to the fp8 query output when one is
// given; a key head and the value head of the same index fill the two halves
// of the token's cache row when the token has a slot.  Value heads are read
// only by calls that insert.  The first loads of a token are issued with its
// position and slot loads, so their latencies overlap; the cos|sin words,
// which need the position, follow.  The (1 + w) values of both norms stay in
// shared memory; the cos|sin words are loaded once per token.
// fp8 codes come from the exact fp32 quotient x / scale (ctx_kv_device.cuh).
// Warps are independent: nothing waits on anything.
//
// Tokens whose position is outside the cos|sin table are left untouched and
// reported; tokens whose slot is beyond the cache are rotated but not
// inserted, and reported.  No access leaves the caller's buffers.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ctx_kv_device.cuh"
#include "ctx_kv_internal.h"
#include "ctx_kv_pipe.cuh"

namespace dspark {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kBatch = 3;  // head groups per warp whose loads are issued together (a 64 + 2 x 8 head
                           // token: 20 groups, one round of loads for 8 warps)
constexpr unsigned kFlagSlot = 0x1u;
constexpr unsigned kFlagPos = 0x2u;

__device__ __forceinline__ uint4 ld16(const void *p) { return *reinterpret_cast<const uint4 *>(p); }
__device__ __forceinline__ void st16(void *p, uint4 v) { *reinterpret_cast<uint4 *>(p) = v; }
__device__ __forceinline__ void st8(void *p, uint2 v) { *reinterpret_cast<uint2 *>(p) = v; }

// RoPE on a bf16 pair: for each half, y * c + yp * sn with a single rounding
// (the product of two bf16 values is exact in fp32, formed as an FMA with -0
// so that a zero product keeps its sign), the operands read as bf16 halves.
__device__ __forceinline__ uint64_t rope_bf2(uint32_t y, uint32_t c, uint32_t yp, uint32_t sn)
{
    float lo, hi;
    asm("{\n\t.reg .b16 y0, y1, c0, c1, p0, p1, s0, s1;\n\t.reg .f32 t0, t1;\n\t"
        "mov.b32 {y0, y1}, %2;\n\tmov.b32 {c0, c1}, %3;\n\t"
        "mov.b32 {p0, p1}, %4;\n\tmov.b32 {s0, s1}, %5;\n\t"
        "fma.rn.f32.bf16 t0, p0, s0, 0f80000000;\n\t"
        "fma.rn.f32.bf16 t1, p1, s1, 0f80000000;\n\t"
        "fma.rn.f32.bf16 %0, y0, c0, t0;\n\t"
        "fma.rn.f32.bf16 %1, y1, c1, t1;\n\t}"
        : "=f"(lo), "=f"(hi)
        : "r"(y), "r"(c), "r"(yp), "r"(sn));
    return pr(lo, hi);
}

// (1 + w) table in shared memory: float4 slot (norm, half jj of an 8-dim
// chunk, chunk c of the 16): lane q reads chunks c = q (dims 8q..) and
// c = 8 + q (dims 64 + 8q..), so the 8 lanes of a head read 128 contiguous
// bytes per load (conflict-free).
__device__ __forceinline__ int w1_slot(int norm, int jj, int c) { return norm * 32 + jj * 16 + c; }

template <int ROT, bool FP8>
__global__ void __launch_bounds__(kThreads, 3) qk_insert_kernel(const QkInsertParams p)
{
    if (threadIdx.x == 0 && blockIdx.x < p.num_tokens) {
        // While the previous kernel drains: this CTA's first token -- its
        // qkv row, position and slot -- into L2 (hints only; every load below
        // still follows griddepcontrol.wait).
        const int64_t t = blockIdx.x, W = p.num_heads + 2 * p.num_kv_heads;
        pipe::prefetch_l2_bulk(p.qkv + t * W * kHeadDim, (uint32_t)(W * kHeadDim * 2));
        pipe::prefetch_l2(p.positions + t);
        if (p.slot_mapping)
            pipe::prefetch_l2(p.slot_mapping + t);
    }
    pdl_enter();
    constexpr int kPartner = ROT / 16;  // lane distance of a rotated pair
    constexpr int kRotLanes = ROT / 8;  // lanes whose first word holds rotary dims
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int q = lane & 7;    // the lane's slice of its head
    const int sub = lane >> 3; // the lane's head within a group of four
    const unsigned smask = 0xffu << (8 * sub);
    const bool rot_lane = q < kRotLanes;
    const int Hq = p.num_heads, Hkv = p.num_kv_heads, W = Hq + 2 * Hkv;
    const int groups = (W + 3) >> 2;
    const int bsl = p.block_size_log2;
    const int64_t head_stride = (int64_t)kRowElems << bsl;  // cache elements between kv heads of one slot

    // The first token's position, slot and first head groups are loaded
    // before anything else, so that their latency overlaps the weight
    // table's set-up; value heads are read whenever an insert is asked for,
    // and dropped for padded tokens.
    uint16_t *trow = p.qkv + (int64_t)blockIdx.x * W * kHeadDim;
    uint4 xa[kBatch], xb[kBatch];
    int hd[kBatch];
    bool live[kBatch];
    auto load_batch = [&](int g0) {
#pragma unroll
        for (int i = 0; i < kBatch; i++) {
            const int g = g0 + i * kWarps;
            const int hh = 4 * g + sub;
            hd[i] = hh;
            live[i] = g < groups && hh < W && (hh < Hq + Hkv || p.slot_mapping != nullptr);
            if (live[i]) {
                const uint16_t *src = trow + hh * kHeadDim;
                xa[i] = ld16(src + 8 * q);
                xb[i] = ld16(src + 64 + 8 * q);
            }
        }
    };
    int64_t pos_first = 0, slot_first = -1;
    if (blockIdx.x < p.num_tokens) {
        pos_first = __ldg(p.positions + blockIdx.x);
        slot_first = p.slot_mapping ? __ldg(p.slot_mapping + blockIdx.x) : -1;
        if (warp < groups)
            load_batch(warp);
    }

    __shared__ float4 w1[64];  // (1 + w) of the query norm (slots 0..31) and the key norm (32..63)
    {
        const int i = threadIdx.x;  // kThreads == 2 * 128: one weight element per thread
        const int norm = i >> 7, d = i & 127, c = d >> 3, e = d & 7;
        const uint16_t wb = __ldg((norm ? p.k_norm_w : p.q_norm_w) + d);
        reinterpret_cast<float *>(w1)[w1_slot(norm, e >> 2, c) * 4 + (e & 3)] = 1.0f + __uint_as_float((uint32_t)wb << 16);
    }
    __syncthreads();
    Fp8Scale kq, vq, qq;
    if (FP8) {
        kq = fp8_scale(p.k_scale ? __ldg(p.k_scale) : 1.0f);
        vq = fp8_scale(p.v_scale ? __ldg(p.v_scale) : 1.0f);
    }
    if (p.q_fp8)
        qq = fp8_scale(p.q_scale);
    unsigned flags = 0;

    for (int64_t t = blockIdx.x; t < p.num_tokens; t += gridDim.x) {
        int g0 = warp;
        int64_t pos = pos_first, slot = slot_first;
        if (t != blockIdx.x) {
            trow = p.qkv + t * W * kHeadDim;
            pos = __ldg(p.positions + t);
            slot = p.slot_mapping ? __ldg(p.slot_mapping + t) : -1;
            if (g0 < groups)
                load_batch(g0);
        }
        if (pos < 0 || pos >= p.max_pos) {
            flags |= kFlagPos;  // untouched, and not inserted either
            continue;
        }
        if (slot >= p.capacity) {
            flags |= kFlagSlot;
            slot = -1;
        }
        // cos and sign * sin (bf16 pairs) of this token for the lane's first word
        uint32_t cw[4] = {0, 0, 0, 0}, sw[4] = {0, 0, 0, 0};
        if (rot_lane) {
            const uint16_t *cs = p.cos_sin + pos * ROT + 8 * (q & (kPartner - 1));
            const uint4 c4 = __ldg(reinterpret_cast<const uint4 *>(cs));
            const uint4 s4 = __ldg(reinterpret_cast<const uint4 *>(cs + ROT / 2));
            const uint32_t flip = (q & kPartner) ? 0u : 0x80008000u;  // the lower half subtracts
            cw[0] = c4.x, cw[1] = c4.y, cw[2] = c4.z, cw[3] = c4.w;
            sw[0] = s4.x ^ flip, sw[1] = s4.y ^ flip, sw[2] = s4.z ^ flip, sw[3] = s4.w ^ flip;
        }
        // row of (slot, kv head 0) in the cache, in elements
        const int64_t row0 =
            slot >= 0 ? ((((slot >> bsl) * Hkv) << bsl) + (slot & ((int64_t(1) << bsl) - 1))) * kRowElems : 0;

        for (; g0 < groups; g0 += kWarps * kBatch) {
            if (g0 != warp)
                load_batch(g0);
#pragma unroll
            for (int i = 0; i < kBatch; i++) {
                if (!live[i])
                    continue;
                const int hh = hd[i];
                if (hh >= Hq + Hkv) {
                    if (slot < 0)
                        continue;  // a padded token's value head: read, not inserted
                    // value head: inserted as it is (or encoded) into the V half of the row
                    unsigned char *d = p.cache + (row0 + (hh - Hq - Hkv) * head_stride + kHeadDim) * (FP8 ? 1 : 2);
                    if (FP8) {
                        st8(d + 8 * q, quantise8(xa[i], vq));
                        st8(d + 64 + 8 * q, quantise8(xb[i], vq));
                    } else {
                        st16(d + 16 * q, xa[i]);
                        st16(d + 128 + 16 * q, xb[i]);
                    }
                    continue;
                }
                const bool is_q = hh < Hq;
                const uint32_t kw[8] = {xa[i].x, xa[i].y, xa[i].z, xa[i].w, xb[i].x, xb[i].y, xb[i].z, xb[i].w};
                uint64_t x2[8];
#pragma unroll
                for (int k = 0; k < 8; k++)
                    x2[k] = bf2_to_f2(kw[k]);
                uint64_t a0 = mul2(x2[0], x2[0]), a1 = mul2(x2[1], x2[1]);
#pragma unroll
                for (int k = 2; k < 8; k += 2) {
                    a0 = fma2(x2[k], x2[k], a0);
                    a1 = fma2(x2[k + 1], x2[k + 1], a1);
                }
                float slo, shi;
                unpr(add2(a0, a1), slo, shi);
                float ss = slo + shi;
                ss += __shfl_xor_sync(smask, ss, 4);
                ss += __shfl_xor_sync(smask, ss, 2);
                ss += __shfl_xor_sync(smask, ss, 1);
                float inv;  // ss/128 + eps >= eps > 0 (hardware reciprocal square root)
                asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(fmaf(ss, 1.0f / kHeadDim, p.eps)));
                const uint64_t inv2 = pr(inv, inv);
                const int nm = is_q ? 0 : 1;
                const float4 wa0 = w1[w1_slot(nm, 0, q)], wa1 = w1[w1_slot(nm, 1, q)];
                const float4 wb0 = w1[w1_slot(nm, 0, 8 + q)], wb1 = w1[w1_slot(nm, 1, 8 + q)];
                const uint64_t w2[8] = {pr(wa0.x, wa0.y), pr(wa0.z, wa0.w), pr(wa1.x, wa1.y), pr(wa1.z, wa1.w),
                                        pr(wb0.x, wb0.y), pr(wb0.z, wb0.w), pr(wb1.x, wb1.y), pr(wb1.z, wb1.w)};
                uint32_t y[8];
#pragma unroll
                for (int k = 0; k < 8; k++)
                    y[k] = f2_to_bf2(mul2(mul2(x2[k], inv2), w2[k]));
                // RoPE on the first word (dims 8q .. 8q+7); the partner is kPartner lanes away
#pragma unroll
                for (int k = 0; k < 4; k++) {
                    const uint32_t yp = __shfl_xor_sync(smask, y[k], kPartner);
                    const uint32_t rv = f2_to_bf2(rope_bf2(y[k], cw[k], yp, sw[k]));
                    y[k] = rot_lane ? rv : y[k];
                }
                const uint4 oa = make_uint4(y[0], y[1], y[2], y[3]), ob = make_uint4(y[4], y[5], y[6], y[7]);
                uint16_t *dst = trow + hh * kHeadDim;
                st16(dst + 8 * q, oa);
                st16(dst + 64 + 8 * q, ob);
                if (is_q) {
                    if (p.q_fp8) {
                        unsigned char *d = p.q_fp8 + (t * Hq + hh) * kHeadDim;
                        st8(d + 8 * q, quantise8(oa, qq));
                        st8(d + 64 + 8 * q, quantise8(ob, qq));
                    }
                } else if (slot >= 0) {
                    unsigned char *d = p.cache + (row0 + (hh - Hq) * head_stride) * (FP8 ? 1 : 2);
                    if (FP8) {
                        st8(d + 8 * q, quantise8(oa, kq));
                        st8(d + 64 + 8 * q, quantise8(ob, kq));
                    } else {
                        st16(d + 16 * q, oa);
                        st16(d + 128 + 16 * q, ob);
                    }
                }
            }
        }
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (flags && lane == 0 && p.error_flags)
        atomicOr(p.error_flags, flags);
}

template <int ROT, bool FP8>
cudaError_t launch_variant(const QkInsertParams &p, cudaStream_t stream)
{
    // at most one CTA per token, at most the CTAs resident at once
    static std::mutex mu;
    static int cached_blocks[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    int max_blocks;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (cached_blocks[dev] == 0) {
            int sms = 0, per_sm = 0;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess)
                return e;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, qk_insert_kernel<ROT, FP8>, kThreads, 0);
            if (e != cudaSuccess)
                return e;
            cached_blocks[dev] = sms * (per_sm > 0 ? per_sm : 1);
        }
        max_blocks = cached_blocks[dev];
    }
    const int blocks = (int)(p.num_tokens < max_blocks ? p.num_tokens : max_blocks);
    return launch_pdl(qk_insert_kernel<ROT, FP8>, blocks, kThreads, 0, stream, p);
}

}  // namespace

cudaError_t launch_qk_insert(const QkInsertParams &p, int rotary_dim, bool fp8_cache, cudaStream_t stream)
{
    switch (rotary_dim) {
    case 16:
        return fp8_cache ? launch_variant<16, true>(p, stream) : launch_variant<16, false>(p, stream);
    case 32:
        return fp8_cache ? launch_variant<32, true>(p, stream) : launch_variant<32, false>(p, stream);
    case 64:
        return fp8_cache ? launch_variant<64, true>(p, stream) : launch_variant<64, false>(p, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace dspark
