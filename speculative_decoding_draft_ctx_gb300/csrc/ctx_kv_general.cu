// sm_103a kernel of the DSpark context-KV write for the layouts the pages'
// kernel refuses: head dims 64 and 256 besides 128, any even rotary_dim up to
// the head dim, and block sizes that are not powers of two.
//
// Defining passage: vLLM DSpark context-KV writer page, module docstring (the
// write: Gemma RMSNorm of K in fp32 materialised to bf16, partial NeoX RoPE at
// the token's position, K|V stored into each layer's paged cache as bf16 or as
// fp8 e4m3 of x / scale, slots < 0 not written) and
// DSparkContextKVWriter._validate / rotary_dims_supported (what that kernel
// accepts: head_dim 128, rotary_dim 16/32/64, power-of-two block sizes).
// The arithmetic is the same; only the layout is wider.
//
// Work decomposition (as in the generic head-dim-128 kernel): a unit is
// (token, layer, up to HPU KV heads) and one warp processes one unit at a
// time, grid-striding in token-major order.  Lanes 0..15 hold K and lanes
// 16..31 V of the same head, E = D / 16 bf16 each, so one load per lane and
// head fetches the whole 4D-byte K|V row and one store per lane writes its
// contiguous 4D (bf16) or 2D (fp8) cache bytes.  All HPU heads of a unit are
// loaded before the first is used.
//
// RoPE for any even r.  The partner of dim d < r is d + r/2 or d - r/2; when
// r/2 is not a multiple of E a lane's partners straddle two other lanes, so
// the normed K row goes through a per-warp shared buffer (two of them,
// alternating between heads, so one __syncwarp per head orders the writes of
// a head before its reads and the reads of head i before the rewrite at
// i + 2).  The token's cos|sin row is staged once per unit in the same way.
// out = y c -+ y_p s is one fused multiply-add around the exact product y_p s
// (two bf16 values: 16 significant bits), then one rounding to bf16.
//
// Block decode: power-of-two block sizes shift and mask; other sizes divide
// by the invariant block size with a multiply-high (Granlund and Montgomery,
// "Division by invariant integers using multiplication", 1994, Thm 4.2):
// for 0 <= n < 2^63 and 2^(l-1) < d < 2^l, m = ceil(2^(63+l) / d) < 2^64
// gives floor(n / d) = umulhi(n, m) >> (l - 1).  The host computes m and l.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ctx_kv_device.cuh"
#include "ctx_kv_internal.h"

namespace dspark {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFlagSlot = 0x1u;
constexpr unsigned kFlagPos = 0x2u;

// W consecutive 32-bit words (2W bf16) of one lane.
template <int W>
struct Words {
    uint32_t w[W];
};

// Streaming loads and stores of 2, 4 or 8 words (8, 16 or 32 bytes, aligned
// to the access size up to 16 bytes).
template <int W>
__device__ __forceinline__ Words<W> ld_stream(const void *p)
{
    Words<W> r;
    const char *c = static_cast<const char *>(p);
    if constexpr (W == 2) {
        asm("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];" : "=r"(r.w[0]), "=r"(r.w[1]) : "l"(c));
    } else {
#pragma unroll
        for (int k = 0; k < W / 4; k++)
            asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                : "=r"(r.w[4 * k]), "=r"(r.w[4 * k + 1]), "=r"(r.w[4 * k + 2]), "=r"(r.w[4 * k + 3])
                : "l"(c + 16 * k));
    }
    return r;
}

template <int W>
__device__ __forceinline__ Words<W> ld_cached(const void *p)
{
    Words<W> r;
    const char *c = static_cast<const char *>(p);
    if constexpr (W == 1) {
        r.w[0] = __ldg(reinterpret_cast<const unsigned int *>(c));
    } else if constexpr (W == 2) {
        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(c));
        r.w[0] = v.x, r.w[1] = v.y;
    } else {
#pragma unroll
        for (int k = 0; k < W / 4; k++) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(c + 16 * k));
            r.w[4 * k] = v.x, r.w[4 * k + 1] = v.y, r.w[4 * k + 2] = v.z, r.w[4 * k + 3] = v.w;
        }
    }
    return r;
}

template <int W>
__device__ __forceinline__ void st_stream(void *p, const Words<W> &v)
{
    char *c = static_cast<char *>(p);
    if constexpr (W == 1) {
        asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(c), "r"(v.w[0]) : "memory");
    } else if constexpr (W == 2) {
        asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(c), "r"(v.w[0]), "r"(v.w[1]) : "memory");
    } else {
#pragma unroll
        for (int k = 0; k < W / 4; k++)
            asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(c + 16 * k), "r"(v.w[4 * k]),
                         "r"(v.w[4 * k + 1]), "r"(v.w[4 * k + 2]), "r"(v.w[4 * k + 3])
                         : "memory");
    }
}

__device__ __forceinline__ float bf_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ float bf_at(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

// e4m3 codes of x / s for the 2W bf16 values of v: W / 2 words of 4 codes
// (exact quotient, see ctx_kv_device.cuh).
template <int W>
__device__ __forceinline__ Words<W / 2> quantise(const Words<W> &v, const Fp8Scale &q)
{
    Words<W / 2> out;
#pragma unroll
    for (int k = 0; k < W / 2; k++) {
        uint64_t pq[2];
#pragma unroll
        for (int j = 0; j < 2; j++)
            pq[j] = quotient2(bf2_to_f2(clamp_bf2(v.w[2 * k + j], q.bound)), q.s2, q.n2);
        out.w[k] = e4m3x4(pq[0], pq[1]);
    }
    return out;
}

__device__ __forceinline__ float load_scale(const float *const *table, int l)
{
    const float *p = reinterpret_cast<const float *>(
        __ldg(reinterpret_cast<const unsigned long long *>(table) + l));
    return __ldg(p);
}

template <int D>
__host__ __device__ constexpr int heads_per_unit()
{
    return D == 64 ? 8 : 4;
}

// Resident blocks per SM the register budget is set for: every warp keeps
// HPU heads (HPU * 4D bytes) in flight.
template <int D>
__host__ __device__ constexpr int min_blocks()
{
    return D == 256 ? 2 : 3;
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kThreads, min_blocks<D>()) ctx_kv_general_kernel(const CtxKvParams p)
{
    pdl_enter();
    constexpr int E = D / 16;  // bf16 per lane
    constexpr int W = E / 2;   // 32-bit words per lane
    constexpr int HPU = heads_per_unit<D>();
    // per warp: the normed K row of the current head (two alternating
    // buffers) and the unit's cos|sin row (r <= D values)
    __shared__ __align__(16) uint16_t s_y[kWarps][2][D];
    __shared__ __align__(16) uint16_t s_cs[kWarps][D];

    const int lane = threadIdx.x & 31;
    const int wib = threadIdx.x >> 5;
    const int kv = lane >> 4;  // 0: K lane, 1: V lane
    const int d0 = (lane & 15) * E;
    const int r = p.rotary_dim, half = r >> 1;
    const bool rot_lane = kv == 0 && d0 < r;

    const int L = p.num_layers, H = p.num_kv_heads, HC = p.head_chunks;
    const int64_t per_tok = (int64_t)L * HC;
    const int64_t units = p.num_ctx * per_tok;
    const int64_t warp = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int64_t nwarps = ((int64_t)gridDim.x * blockDim.x) >> 5;
    const int64_t bs = p.block_size;
    unsigned flags = 0;

    for (int64_t u = warp; u < units; u += nwarps) {
        const int64_t t = u / per_tok;
        const int rem = (int)(u - t * per_tok);
        const int l = rem / HC;
        const int h0 = (rem - l * HC) * HPU;
        const int nh = min(HPU, H - h0);
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

        const uint16_t *src = p.all_kv + ((((t * L + l) * 2 + kv) * H + h0) * D + d0);
        Words<W> x[HPU];
#pragma unroll
        for (int i = 0; i < HPU; i++)
            if (i < nh)
                x[i] = ld_stream<W>(src + i * D);

        const Words<W> wr = ld_cached<W>(p.knorm_w + (int64_t)l * D + d0);
        float w1[E];
#pragma unroll
        for (int j = 0; j < W; j++) {
            w1[2 * j] = 1.0f + bf_lo(wr.w[j]);
            w1[2 * j + 1] = 1.0f + bf_hi(wr.w[j]);
        }
        const int64_t layer_off = __ldg(p.cache_offsets + l);
        Fp8Scale ksc{}, vsc{};
        if constexpr (FP8) {
            ksc = fp8_scale(load_scale(p.k_scales, l));
            vsc = fp8_scale(load_scale(p.v_scales, l));
        }

        // the previous unit's reads of s_cs and s_y are done before any lane
        // rewrites them; the staged cos|sin row is visible after the first
        // head's __syncwarp below
        __syncwarp();
        {
            const uint32_t *cs = reinterpret_cast<const uint32_t *>(p.cos_sin + pos * r);
            uint32_t *dst = reinterpret_cast<uint32_t *>(s_cs[wib]);
            for (int k = lane; k < half; k += 32)
                dst[k] = __ldg(cs + k);
        }

        int64_t blk, off;
        if (p.block_size_log2 >= 0) {
            blk = slot >> p.block_size_log2;
            off = slot & (bs - 1);
        } else {
            blk = (int64_t)(__umul64hi((unsigned long long)slot, p.bs_magic) >> p.bs_magic_shift);
            off = slot - blk * bs;
        }
        const int64_t row0 = (blk * H + h0) * bs + off;

#pragma unroll
        for (int i = 0; i < HPU; i++) {
            if (i >= nh)
                break;
            float f[E];
#pragma unroll
            for (int j = 0; j < W; j++) {
                f[2 * j] = bf_lo(x[i].w[j]);
                f[2 * j + 1] = bf_hi(x[i].w[j]);
            }
            float ss = 0.0f;
#pragma unroll
            for (int j = 0; j < E; j++)
                ss = fmaf(f[j], f[j], ss);
            ss += __shfl_xor_sync(0xffffffffu, ss, 8);
            ss += __shfl_xor_sync(0xffffffffu, ss, 4);
            ss += __shfl_xor_sync(0xffffffffu, ss, 2);
            ss += __shfl_xor_sync(0xffffffffu, ss, 1);
            const float inv = rsqrtf(fmaf(ss, 1.0f / D, p.eps));

            Words<W> y;
#pragma unroll
            for (int j = 0; j < W; j++)
                y.w[j] = pack_bf16x2((f[2 * j] * inv) * w1[2 * j], (f[2 * j + 1] * inv) * w1[2 * j + 1]);
            uint16_t *yb = s_y[wib][i & 1];
            if (kv == 0) {
                uint32_t *yw = reinterpret_cast<uint32_t *>(yb + d0);
#pragma unroll
                for (int j = 0; j < W; j++)
                    yw[j] = y.w[j];
            }
            __syncwarp();

            Words<W> out;
            if (kv == 0) {
                if (rot_lane) {
                    float o[E];
#pragma unroll
                    for (int j = 0; j < E; j++) {
                        const int d = d0 + j;
                        const float yd = (j & 1) ? bf_hi(y.w[j >> 1]) : bf_lo(y.w[j >> 1]);
                        if (d < r) {
                            const bool lower = d < half;
                            const int fi = lower ? d : d - half;
                            const float c = bf_at(s_cs[wib][fi]);
                            const float s = bf_at(s_cs[wib][half + fi]);
                            const float yp = bf_at(yb[lower ? d + half : d - half]);
                            o[j] = fmaf(yd, c, lower ? -(yp * s) : yp * s);
                        } else {
                            o[j] = yd;
                        }
                    }
#pragma unroll
                    for (int j = 0; j < W; j++) {
                        // dims >= r keep y exactly: a bf16 value converts to itself
                        out.w[j] = pack_bf16x2(o[2 * j], o[2 * j + 1]);
                    }
                } else {
                    out = y;
                }
            } else {
                out = x[i];
            }

            const int64_t elem = layer_off + (row0 + (int64_t)i * bs) * (2 * D);
            if constexpr (!FP8) {
                st_stream<W>(p.cache0 + (elem + lane * E) * 2, out);
            } else {
                st_stream<W / 2>(p.cache0 + elem + lane * E, quantise<W>(out, kv == 0 ? ksc : vsc));
            }
        }
    }
    if (flags && lane == 0 && p.error_flags)
        atomicOr(p.error_flags, flags);
}

template <int D, bool FP8>
cudaError_t launch_variant(const CtxKvParams &p, cudaStream_t stream)
{
    // Resident blocks per SM times the SM count, per device (queried once).
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
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, ctx_kv_general_kernel<D, FP8>, kThreads, 0);
            if (e != cudaSuccess)
                return e;
            cached_blocks[dev] = sms * (per_sm > 0 ? per_sm : 1);
        }
        max_blocks = cached_blocks[dev];
    }
    CtxKvParams q = p;
    q.head_chunks = (p.num_kv_heads + heads_per_unit<D>() - 1) / heads_per_unit<D>();
    const int64_t units = q.num_ctx * (int64_t)q.num_layers * q.head_chunks;
    const int64_t need = (units + kWarps - 1) / kWarps;
    const int blocks = (int)(need < max_blocks ? need : max_blocks);
    return launch_pdl(ctx_kv_general_kernel<D, FP8>, blocks, kThreads, 0, stream, q);
}

}  // namespace

cudaError_t launch_ctx_kv_general(const CtxKvParams &p, int head_dim, bool fp8, cudaStream_t stream)
{
    switch (head_dim) {
    case 64:
        return fp8 ? launch_variant<64, true>(p, stream) : launch_variant<64, false>(p, stream);
    case 128:
        return fp8 ? launch_variant<128, true>(p, stream) : launch_variant<128, false>(p, stream);
    case 256:
        return fp8 ? launch_variant<256, true>(p, stream) : launch_variant<256, false>(p, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace dspark
