// sm_103a kernel of the hidden-state Gemma RMSNorm of the context states.
//
// Defining passage: DSpark draft model page -- MiniMaxM3DSparkModel.__init__
// (hidden_norm = _gemma_rms_norm(hidden_size, eps)), _normalize_context_states
// (the context states through hidden_norm), _gemma_rms_norm (the target's
// Gemma RMSNorm: y = x * rsqrt(mean(x^2) + eps) * (1 + w), an fp32 1 + w
// weight; the unfused path ran "about ten kernels").  Here: one launch.
//
// One warp per row, grid-striding over rows: lane j holds the 16-byte chunks
// j, j + 32, ... of the row (kChunks per lane, 8 bf16 each; rows up to 4096
// wide), all loaded before any is used, so a warp keeps a whole row in
// flight; wider rows (up to 8192) are read twice, the second time from L2.
// Sum of squares on mixed bf16 FMAs (fma.rn.f32.bf16 on the register halves,
// four chains), a 5-step xor shuffle, the hardware reciprocal square root;
// y = bf16((x * inv) * (1 + w)) in fp32 with (1 + w) read through L1
// (every row uses the same weight).  Rows wider than 1024 (up to 4096) are shared by
// four warps instead (finer work units: no ragged last wave of whole
// rows).  A row is read before it is written, so
// the output may be the input (in place).  Bound: HBM, 2 * hidden * 2 bytes
// per row.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ctx_kv_device.cuh"
#include "ctx_kv_internal.h"
#include "ctx_kv_pipe.cuh"

namespace dspark {
namespace {

constexpr int kThreadsN = 256;
constexpr int kWarpsN = kThreadsN / 32;

// The weight chunk and the output store of a chunk are issued in program
// order (volatile asm), so the compiler does not hoist every weight load of
// the row ahead of the stores and run out of registers.
__device__ __forceinline__ uint4 ld_weight(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ void st_out(void *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

// acc + lo^2 + hi^2 of a bf16 pair, read as register halves (a bf16 square
// is exact in fp32, so each step rounds once); no unpacked copy of the row
// stays alive for the second phase.
__device__ __forceinline__ float sumsq_bf2(uint32_t w, float acc)
{
    float r;
    asm("{\n\t.reg .b16 l, h;\n\t.reg .f32 t;\n\tmov.b32 {l, h}, %1;\n\t"
        "fma.rn.f32.bf16 t, l, l, %2;\n\tfma.rn.f32.bf16 %0, h, h, t;\n\t}"
        : "=f"(r)
        : "r"(w), "f"(acc));
    return r;
}

__device__ __forceinline__ uint4 ld_stream(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// While the previous kernel drains: row r of x into L2 (a hint only; the
// loads still follow griddepcontrol.wait).  Rows are a multiple of 16 bytes
// and x is 16-byte aligned.
__device__ __forceinline__ void prefetch_row(const uint16_t *x, int64_t r, int64_t rows, int hidden)
{
    if (r < rows && (threadIdx.x & 31) == 0)
        pipe::prefetch_l2_bulk(x + r * hidden, (uint32_t)hidden * 2u);
}

// Widths up to 32 * 8 * kChunks elements; rows wider than 4096 take the
// two-pass variant (kChunks 0): the sum of squares first, then the row is
// read again (an L2 hit) to be normed, so no lane holds more than it must.
template <int kChunks>
__global__ void __launch_bounds__(kThreadsN, kChunks <= 4 ? 4 : (kChunks <= 8 ? 3 : 2))
    gemma_norm_kernel(const uint16_t *x, const uint16_t *w, uint16_t *out, int64_t rows, int hidden, float eps)
{
    prefetch_row(x, (int64_t)blockIdx.x * kWarpsN + (threadIdx.x >> 5), rows, hidden);
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int chunks = hidden >> 3;
    const float inv_n = 1.0f / (float)hidden;
    const int64_t nw = (int64_t)gridDim.x * kWarpsN;
    for (int64_t r = (int64_t)blockIdx.x * kWarpsN + (threadIdx.x >> 5); r < rows; r += nw) {
        const uint16_t *xr = x + r * hidden;
        uint4 v[kChunks];
#pragma unroll
        for (int i = 0; i < kChunks; i++) {
            const int c = lane + 32 * i;
            v[i] = c < chunks ? ld_stream(xr + 8 * c) : make_uint4(0, 0, 0, 0);
        }
        float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
#pragma unroll
        for (int i = 0; i < kChunks; i++) {
            s0 = sumsq_bf2(v[i].x, s0);
            s1 = sumsq_bf2(v[i].y, s1);
            s2 = sumsq_bf2(v[i].z, s2);
            s3 = sumsq_bf2(v[i].w, s3);
        }
        float ss = (s0 + s1) + (s2 + s3);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, o);
        float inv;  // ss/n + eps >= eps > 0 (hardware reciprocal square root)
        asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(fmaf(ss, inv_n, eps)));
        const uint64_t inv2 = pr(inv, inv), one = pr(1.0f, 1.0f);
        uint16_t *orow = out + r * hidden;
#pragma unroll
        for (int i = 0; i < kChunks; i++) {
            const int c = lane + 32 * i;
            if (c >= chunks)
                break;
            const uint4 wv = ld_weight(w + 8 * c);
            const uint32_t xs[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
            uint32_t y[4];
#pragma unroll
            for (int k = 0; k < 4; k++)
                y[k] = f2_to_bf2(mul2(mul2(bf2_to_f2(xs[k]), inv2), add2(bf2_to_f2(ws[k]), one)));
            st_out(orow + 8 * c, y[0], y[1], y[2], y[3]);
        }
    }
}

// Four warps per row (rows wider than 1024, up to 4096), so that the work is cut into
// units four times finer than whole rows; the four partial sums of squares
// meet in shared memory.
__global__ void __launch_bounds__(kThreadsN) gemma_norm_split_kernel(const uint16_t *x, const uint16_t *w,
                                                                     uint16_t *out, int64_t rows, int hidden,
                                                                     float eps)
{
    constexpr int kRowsPerCta = kWarpsN / 4, kChunksS = 4;  // 128 threads x 4 chunks = 4096 elements
    if (((threadIdx.x >> 5) & 3) == 0)
        prefetch_row(x, (int64_t)blockIdx.x * kRowsPerCta + (threadIdx.x >> 7), rows, hidden);
    pdl_enter();
    __shared__ float part[kWarpsN];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int slot = warp >> 2;                  // row within the CTA (warp & 3: the warp within its row)
    const int tr = threadIdx.x & 127;            // thread within its row
    const int chunks = hidden >> 3;
    const float inv_n = 1.0f / (float)hidden;
    for (int64_t r0 = (int64_t)blockIdx.x * kRowsPerCta; r0 < rows; r0 += (int64_t)gridDim.x * kRowsPerCta) {
        const int64_t r = r0 + slot;
        const bool live = r < rows;
        const uint16_t *xr = x + (live ? r : 0) * hidden;
        uint4 v[kChunksS];
#pragma unroll
        for (int i = 0; i < kChunksS; i++) {
            const int c = tr + 128 * i;
            v[i] = (live && c < chunks) ? ld_stream(xr + 8 * c) : make_uint4(0, 0, 0, 0);
        }
        float s0 = 0.0f, s1 = 0.0f, s2 = 0.0f, s3 = 0.0f;
#pragma unroll
        for (int i = 0; i < kChunksS; i++) {
            s0 = sumsq_bf2(v[i].x, s0);
            s1 = sumsq_bf2(v[i].y, s1);
            s2 = sumsq_bf2(v[i].z, s2);
            s3 = sumsq_bf2(v[i].w, s3);
        }
        float ss = (s0 + s1) + (s2 + s3);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, o);
        if (lane == 0)
            part[warp] = ss;
        __syncthreads();
        ss = (part[4 * slot] + part[4 * slot + 1]) + (part[4 * slot + 2] + part[4 * slot + 3]);
        __syncthreads();  // part[] is reused by the next rows
        if (!live)
            continue;
        float inv;  // ss/n + eps >= eps > 0 (hardware reciprocal square root)
        asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(fmaf(ss, inv_n, eps)));
        const uint64_t inv2 = pr(inv, inv), one = pr(1.0f, 1.0f);
        uint16_t *orow = out + r * hidden;
#pragma unroll
        for (int i = 0; i < kChunksS; i++) {
            const int c = tr + 128 * i;
            if (c >= chunks)
                break;
            const uint4 wv = ld_weight(w + 8 * c);
            const uint32_t xs[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
            const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
            uint32_t y[4];
#pragma unroll
            for (int k = 0; k < 4; k++)
                y[k] = f2_to_bf2(mul2(mul2(bf2_to_f2(xs[k]), inv2), add2(bf2_to_f2(ws[k]), one)));
            st_out(orow + 8 * c, y[0], y[1], y[2], y[3]);
        }
    }
}

__global__ void __launch_bounds__(kThreadsN, 4)
    gemma_norm_two_pass_kernel(const uint16_t *x, const uint16_t *w, uint16_t *out, int64_t rows, int hidden,
                               float eps)
{
    prefetch_row(x, (int64_t)blockIdx.x * kWarpsN + (threadIdx.x >> 5), rows, hidden);
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int chunks = hidden >> 3;
    const float inv_n = 1.0f / (float)hidden;
    const int64_t nw = (int64_t)gridDim.x * kWarpsN;
    for (int64_t r = (int64_t)blockIdx.x * kWarpsN + (threadIdx.x >> 5); r < rows; r += nw) {
        const uint16_t *xr = x + r * hidden;
        uint64_t a0 = pr(0.0f, 0.0f), a1 = a0;
#pragma unroll 4
        for (int c = lane; c < chunks; c += 32) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr + 8 * c));
            const uint64_t p0 = bf2_to_f2(v.x), p1 = bf2_to_f2(v.y), p2 = bf2_to_f2(v.z), p3 = bf2_to_f2(v.w);
            a0 = fma2(p0, p0, a0);
            a1 = fma2(p1, p1, a1);
            a0 = fma2(p2, p2, a0);
            a1 = fma2(p3, p3, a1);
        }
        float lo, hi;
        unpr(add2(a0, a1), lo, hi);
        float ss = lo + hi;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
            ss += __shfl_xor_sync(0xffffffffu, ss, o);
        float inv;  // ss/n + eps >= eps > 0 (hardware reciprocal square root)
        asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(fmaf(ss, inv_n, eps)));
        const uint64_t inv2 = pr(inv, inv), one = pr(1.0f, 1.0f);
        uint16_t *orow = out + r * hidden;
#pragma unroll 4
        for (int c = lane; c < chunks; c += 32) {
            const uint4 v = __ldg(reinterpret_cast<const uint4 *>(xr + 8 * c));
            const uint4 wv = __ldg(reinterpret_cast<const uint4 *>(w + 8 * c));
            const uint32_t xs[4] = {v.x, v.y, v.z, v.w};
            const uint32_t ws[4] = {wv.x, wv.y, wv.z, wv.w};
            uint32_t y[4];
#pragma unroll
            for (int k = 0; k < 4; k++)
                y[k] = f2_to_bf2(mul2(mul2(bf2_to_f2(xs[k]), inv2), add2(bf2_to_f2(ws[k]), one)));
            *reinterpret_cast<uint4 *>(orow + 8 * c) = make_uint4(y[0], y[1], y[2], y[3]);
        }
    }
}

// kChunks: 16-byte chunks per lane of the one-warp-per-row kernel; 0: the
// two-pass kernel; -1: the four-warps-per-row kernel.
template <int kChunks>
cudaError_t launch_norm_variant(const uint16_t *x, const uint16_t *w, uint16_t *out, int64_t rows, int hidden,
                                float eps, cudaStream_t stream)
{
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
            if constexpr (kChunks > 0)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemma_norm_kernel<kChunks>, kThreadsN, 0);
            else if constexpr (kChunks == 0)
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemma_norm_two_pass_kernel, kThreadsN, 0);
            else
                e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, gemma_norm_split_kernel, kThreadsN, 0);
            if (e != cudaSuccess)
                return e;
            cached_blocks[dev] = sms * (per_sm > 0 ? per_sm : 1);
        }
        max_blocks = cached_blocks[dev];
    }
    const int rows_per_cta = kChunks < 0 ? kWarpsN / 4 : kWarpsN;
    const int64_t need = (rows + rows_per_cta - 1) / rows_per_cta;
    const int blocks = (int)(need < max_blocks ? need : max_blocks);
    if constexpr (kChunks > 0)
        return launch_pdl(gemma_norm_kernel<kChunks>, blocks, kThreadsN, 0, stream, x, w, out, rows, hidden, eps);
    else if constexpr (kChunks == 0)
        return launch_pdl(gemma_norm_two_pass_kernel, blocks, kThreadsN, 0, stream, x, w, out, rows, hidden, eps);
    else
        return launch_pdl(gemma_norm_split_kernel, blocks, kThreadsN, 0, stream, x, w, out, rows, hidden, eps);
}

}  // namespace

cudaError_t launch_gemma_norm(const uint16_t *x, const uint16_t *w, uint16_t *out, int64_t rows, int hidden,
                              float eps, cudaStream_t stream)
{
    const int per_lane = (hidden / 8 + 31) / 32;  // 16-byte chunks per lane
    // rows wider than 1024 and at most 4096: each row over four warps (faster than
    // a warp per row at every row count: 512, 8192 and 65536 rows)
    static int sms = 0;
    if (sms == 0) {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) == cudaSuccess && cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) ==
                                                      cudaSuccess)
            sms = v;
    }
    if (hidden <= 4096 && per_lane > 4 && sms > 0)
        return launch_norm_variant<-1>(x, w, out, rows, hidden, eps, stream);
    if (per_lane <= 4)
        return launch_norm_variant<4>(x, w, out, rows, hidden, eps, stream);
    if (per_lane <= 8)
        return launch_norm_variant<8>(x, w, out, rows, hidden, eps, stream);
    if (per_lane <= 16)
        return launch_norm_variant<16>(x, w, out, rows, hidden, eps, stream);
    if (per_lane <= 32)
        return launch_norm_variant<0>(x, w, out, rows, hidden, eps, stream);  // two passes
    return cudaErrorInvalidValue;
}

}  // namespace dspark
