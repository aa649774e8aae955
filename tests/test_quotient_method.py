"""The fp8 path's quotient method against IEEE division, on the CPU.

The pipelined kernels form x / scale (the fp8 store's "x / scale", vLLM
DSpark context-KV writer page, module docstring) with Markstein's FMA
correction of a reciprocal-multiplied quotient.  x is clamped in magnitude to
a bound B >= 448 s (the bf16 value just above 512 s, so every clamped
quotient still saturates) and negated in the same instruction (min.xorsign.abs
against -B; NaN kept); with the negated reciprocal n = -RN(1/s):
    x' = -sign(x) min(|x|, B),  p0 = x' * n,  e = p0*s + x'  (exact by FMA),
    p = p0 + e*n  = -(x'/s) correctly rounded,  code = e4m3(p).
This test runs the same operations in C (the C library's correctly rounded
fmaf) for every bf16 value x, including +-0, subnormals, +-inf and NaN, and
many fp32 scales, and checks that
  * that code equals the e4m3 code (RNE, saturating, the oracle's encoder)
    of the IEEE quotient x / s -- so the kernels' fp8 codes can be bit-exact
    with the oracle's true division, signed zeros and NaN included;
  * p is the correctly rounded quotient wherever |x| and |x / s| are at
    least 2^-90 and x is not clamped (below, the FMA residual underflows;
    those quotients are far below e4m3's smallest step and encode to a zero
    of the right sign either way).
"""

import ctypes
import os
import subprocess
import tempfile

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SRC = r"""
#include <math.h>
#include <stdint.h>
#include <string.h>
uint8_t dspark_oracle_e4m3_rne_sat(float xf);
static float bf(uint16_t b) { uint32_t u = (uint32_t)b << 16; float f; memcpy(&f, &u, 4); return f; }
static uint32_t bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float clamp_neg(float v, float bound) {   /* min.NaN.xorsign.abs(v, -bound) */
    if (isnan(v)) return v;
    return copysignf(fminf(fabsf(v), bound), -v);
}
static float bf16_up(float v) {  /* smallest bf16 >= v > 0 */
    uint32_t u = bits(v);
    if (u & 0xffff) u = (u & 0xffff0000u) + 0x10000u;
    float f; memcpy(&f, &u, 4); return f;
}
/* counts code mismatches and (normal-range) quotient mismatches */
void check(const float *scales, int ns, long long *bad_code, long long *bad_q, long long *first) {
    *bad_code = *bad_q = 0; *first = -1;
    for (int j = 0; j < ns; j++) {
        const float s = scales[j];
        const volatile float one = 1.0f;
        const float n = -(one / s);
        const float bound = bf16_up(512.0f * s);
        for (uint32_t b = 0; b < 65536; b++) {
            const float x = bf((uint16_t)b);
            const volatile float xv = x;
            const float want = xv / s;
            const float xc = clamp_neg(x, bound);
            const float p0 = xc * n;
            const float e = fmaf(p0, s, xc);
            const float q = fmaf(e, n, p0);
            const uint8_t code = dspark_oracle_e4m3_rne_sat(q);
            const uint8_t want_code = dspark_oracle_e4m3_rne_sat(want);
            if (code != want_code) {
                if (*first < 0) *first = (long long)j << 16 | b;
                (*bad_code)++;
            }
            const float a = fabsf(want);
            if (fabsf(x) >= 0x1p-90f && a >= 0x1p-90f && fabsf(x) <= bound && bits(q) != bits(want)) (*bad_q)++;
        }
    }
}
"""


@pytest.fixture(scope="module")
def checker():
    d = tempfile.mkdtemp()
    c = os.path.join(d, "q.c")
    so = os.path.join(d, "q.so")
    open(c, "w").write(SRC)
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-shared", "-fPIC",
                    "-o", so, c, os.path.join(ROOT, "oracle", "ctx_kv_oracle.c"), "-lm"], check=True)
    lib = ctypes.CDLL(so)
    P = ctypes.POINTER(ctypes.c_longlong)
    lib.check.argtypes = [ctypes.c_void_p, ctypes.c_int, P, P, P]
    lib.check.restype = None
    return lib


def test_quotient_gives_the_true_division_codes(checker):
    rng = np.random.default_rng(0)
    scales = np.concatenate([
        rng.uniform(0.05, 0.5, 300),            # the workloads' scale range
        np.exp(rng.uniform(-30, 30, 200)),      # wide magnitudes
        [1.0, 0.5, 0.25, 3.0, 0.1, 1 / 3, 448.0, 1e-3, 7.0, 1e-30, 1e30, 1e35],
        # significands near 1 and near 2 (reciprocals near powers of two)
        np.float32(1.0) + np.arange(1, 50, dtype=np.float32) * np.float32(2**-23),
        np.float32(2.0) - np.arange(1, 50, dtype=np.float32) * np.float32(2**-22),
    ]).astype(np.float32)
    bc, bq, first = ctypes.c_longlong(), ctypes.c_longlong(), ctypes.c_longlong()
    checker.check(scales.ctypes.data, len(scales), ctypes.byref(bc), ctypes.byref(bq), ctypes.byref(first))
    assert bc.value == 0, (bc.value, first.value)
    assert bq.value == 0, bq.value
