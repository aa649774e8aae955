// Inline-PTX helpers of the bulk-copy pipelines (ctx_kv_tma.cu,
// ctx_kv_owned.cu): mbarrier waits bounded by the global timer, bulk
// asynchronous copies global -> shared with L2 cache hints, streaming
// stores, and the bf16 RoPE pair FMA.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ctx_kv_device.cuh"

namespace dspark {
namespace pipe {

constexpr unsigned long long kTimeoutNs = 4000000000ull;  // 4 s


__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// One poll of a barrier phase.  A waiting warp is suspended by the hardware
// (up to kSuspendNs) until the phase completes, so waiting warps do not take
// issue slots from the warps that compute.
constexpr uint32_t kSuspendNs = 200000;

// Raises the transaction count the current phase of `bar` waits for,
// without arriving.
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity), "n"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with the given parity to complete.  Gives up
// (and raises the CTA's abort word) after kTimeoutNs, or as soon as another
// warp of the CTA has given up.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort)
{
    if (mbar_try_wait(bar, parity))
        return true;
    const unsigned long long t0 = globaltimer();
    while (true) {
        if (mbar_try_wait(bar, parity))
            return true;
        if (*abort)
            return false;
        if (globaltimer() - t0 > kTimeoutNs) {
            *abort = 1;
            return false;
        }
    }
}

// Bulk copy global -> shared, completing on `bar`; `policy` is an L2 cache
// policy (evict-first for data read exactly once).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar,
                                         uint64_t policy)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Hints that bring global memory into L2 and hand no data to the program.
// L2 is the point of coherence of every SM's global accesses, so they may be
// issued before griddepcontrol.wait even on bytes the previous kernel is
// still writing: the copies made after the wait read the lines as that
// kernel leaves them.  Bulk form: 16-byte aligned address, size a multiple
// of 16.
__device__ __forceinline__ void prefetch_l2_bulk(const void *src, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void *p)
{
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ uint64_t evict_first_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ uint64_t evict_last_policy()
{
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// A plain load (not asm) so the compiler may schedule the loads of a group
// together; the mbarrier waits carry "memory" clobbers, so none moves above
// the wait that makes its stage valid.
__device__ __forceinline__ uint4 lds128(const void *p) { return *reinterpret_cast<const uint4 *>(p); }

__device__ __forceinline__ void st_stream_v4(void *p, uint4 v)
{
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

__device__ __forceinline__ void st_stream_v1(void *p, uint32_t v)
{
    asm volatile("st.global.cs.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_stream_v2(void *p, uint2 v)
{
    asm volatile("st.global.cs.v2.u32 [%0], {%1, %2};" ::"l"(p), "r"(v.x), "r"(v.y) : "memory");
}

// RoPE on a bf16 pair: for each half, y * c + yp * sn with a single rounding
// (the product yp * sn of two bf16 values is exact in fp32, formed as an FMA
// with -0 so that a zero product keeps its sign).  The operands stay bf16:
// the mixed-precision fma.rn.f32.bf16 reads register halves directly.
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

}  // namespace pipe
}  // namespace dspark
