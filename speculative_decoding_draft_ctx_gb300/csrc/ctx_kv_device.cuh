// Device helpers shared by the sm_103a kernels of this library: bf16 and
// paired-fp32 arithmetic and the fp8 e4m3 encoding of x / scale.
//
// The fp8 store holds e4m3(x / scale) with the division in fp32 (vLLM DSpark
// context-KV writer page, module docstring: "fp8 e4m3 of x / scale").  The
// quotient is formed exactly, without a division instruction.  x is first
// clamped in magnitude to a bf16 bound just above 512 s and negated, in one
// instruction (min.xorsign.abs against the negated bound): x' = -sign(x)
// min(|x|, B), so x' n cannot overflow and every clamped quotient still
// saturates.  With the negated correctly rounded reciprocal n = -RN(1/s),
// Markstein's FMA correction  p0 = x' n,  e = p0 s + x' (exact),
// p = p0 + e n  gives p = RN(-x' / s) = RN(x_c / s) whenever |x| and |x / s|
// are at least 2^-90 (below, the residual underflows and the quotient
// encodes to a zero of the right sign either way); signed zeros come out
// with the sign of x.  The saturating RNE pack of p is the code of the IEEE
// quotient; a NaN input gives the NaN code 0x7F.  The method is checked
// against IEEE division for every bf16 input on the CPU.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace dspark {

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ------------------------------------------------------------------ packed fp32 pairs
// Blackwell's paired fp32 FMA / multiply / add (fma.rn.f32x2 and friends)
// process two values per instruction; a pair lives in a 64-bit register.

__device__ __forceinline__ uint64_t pr(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void unpr(uint64_t v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// bf16 pair (element 2j in the low half) -> fp32 pair, exactly
__device__ __forceinline__ uint64_t bf2_to_f2(uint32_t w) { return pr(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u)); }

// fp32 pair -> bf16 pair, round to nearest even
__device__ __forceinline__ uint32_t f2_to_bf2(uint64_t v)
{
    float lo, hi;
    unpr(v, lo, hi);
    return pack_bf16x2(lo, hi);
}

// min(|w|, |bound|) per half with the sign of w XOR the sign of bound (a
// negative bound negates), NaN kept
__device__ __forceinline__ uint32_t clamp_bf2(uint32_t w, uint32_t bound)
{
    uint32_t d;
    asm("min.NaN.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(w), "r"(bound));
    return d;
}

// Four e4m3 codes in one word, element order a b c d from the low byte up,
// RNE with saturation.
__device__ __forceinline__ uint32_t e4m3x4(uint64_t ab, uint64_t cd)
{
    float a, b, c, d;
    unpr(ab, a, b);
    unpr(cd, c, d);
    uint32_t w;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 lo, %2, %1;\n\t"
        "cvt.rn.satfinite.e4m3x2.f32 hi, %4, %3;\n\t"
        "mov.b32 %0, {lo, hi};\n\t}"
        : "=r"(w)
        : "f"(a), "f"(b), "f"(c), "f"(d));
    return w;
}

// -x' / s correctly rounded for an fp32 pair x' (already clamped and
// negated): s2 = (s, s), n2 = (-RN(1/s), -RN(1/s)).
__device__ __forceinline__ uint64_t quotient2(uint64_t x, uint64_t s2, uint64_t n2)
{
    const uint64_t p0 = mul2(x, n2);
    const uint64_t e = fma2(p0, s2, x);
    return fma2(e, n2, p0);
}

// e4m3 codes of x / s for the 8 bf16 values of v (two 4-code words): nbound
// is the negated clamp bound as a bf16 pair, s2 = (s, s),
// n2 = (-RN(1/s), -RN(1/s)).
__device__ __forceinline__ uint2 quantise8(const uint4 &v, uint32_t nbound, uint64_t s2, uint64_t n2)
{
    const uint32_t w[4] = {clamp_bf2(v.x, nbound), clamp_bf2(v.y, nbound), clamp_bf2(v.z, nbound),
                           clamp_bf2(v.w, nbound)};
    uint64_t p[4];
#pragma unroll
    for (int j = 0; j < 4; j++)
        p[j] = quotient2(bf2_to_f2(w[j]), s2, n2);
    return make_uint2(e4m3x4(p[0], p[1]), e4m3x4(p[2], p[3]));
}


// Negated clamp bound of a scale: minus the smallest bf16 >= 512 s, as a
// bf16 pair.
__device__ __forceinline__ uint32_t fp8_bound_pair(float s)
{
    uint32_t u = __float_as_uint(512.0f * s);
    if (u & 0xffffu)
        u = (u & 0xffff0000u) + 0x10000u;
    return ((u >> 16) | 0x8000u) * 0x10001u;
}

// Everything quantise8 needs for one scale.
struct Fp8Scale {
    uint32_t bound;
    uint64_t s2, n2;
};

__device__ __forceinline__ Fp8Scale fp8_scale(float s)
{
    const float n = -__frcp_rn(s);
    return Fp8Scale{fp8_bound_pair(s), pr(s, s), pr(n, n)};
}

__device__ __forceinline__ uint2 quantise8(const uint4 &v, const Fp8Scale &q)
{
    return quantise8(v, q.bound, q.s2, q.n2);
}

}  // namespace dspark
