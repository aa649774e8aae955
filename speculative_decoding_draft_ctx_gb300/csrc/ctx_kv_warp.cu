// sm_103a context-KV write with warp-private pipelines: the fast path for the
// pages' own layout (head dim 128, rotary dim 16, 32 or 64, a power-of-two
// block size, one slot mapping shared by every layer) with 4 or 8 KV heads.
// Every other layout runs on ctx_kv_tma.cu (or the fallbacks).
//
// Defining passage: vLLM DSpark context-KV writer page, module docstring (one
// launch for all draft layers: Gemma RMSNorm of K in fp32 materialised to
// bf16, partial NeoX RoPE at the token's position, K|V stored into each
// layer's [num_blocks, nkv, block_size, 256] cache as bf16 or fp8 e4m3 of
// x / scale, slots < 0 not written).
//
// Work split.  A unit is (P tokens, one layer) with P = 8 / nkv: the layer's
// 8 rows -- two groups of four -- of one token (8 KV heads) or of two
// consecutive tokens (4 KV heads).  The grid's warps are numbered so that
// warp gw owns layer gw % L and the token stream gw / L: units gw / L,
// gw / L + NS, ... (NS streams in all).  A warp keeps everything that depends
// on its layer in registers for the whole launch ((1 + w) of its lane's 16
// dims, the layer's cache base, the fp8 scale constants) and runs its own
// pipeline: a ring of S shared-memory stages, each filled by one bulk
// asynchronous copy per token of all_kv[t, l] (the layer's K and V rows of
// the token, nkv * 512 contiguous bytes) plus the token's cos|sin row,
// completing on the stage's mbarrier (transaction bytes).  The warp reads
// slots and positions of its next 32 units one batch ahead, issues copies up
// to S units ahead of the unit it computes, skips units whose tokens are all
// padding, and copies its first S units before their slots are known (a
// padded token among them is read and dropped).  No warp ever waits for
// another: there is no producer warp and no stage shared between warps, so
// the warps of an SM drift apart and keep its issue slots evenly busy.
//
// Compute mapping: 8 lanes per row, lane q holding dims [8q, 8q + 8) and
// [64 + 8q, 64 + 8q + 8) of K and of V; sum of squares on paired FMAs and 3
// xor shuffles; rsqrt.approx; RoPE partner r/16 lanes away (one xor shuffle)
// with a single rounding per output; fp8 as the correctly rounded fp32
// quotient (Markstein's correction of the reciprocal product, see
// ctx_kv_device.cuh) and a saturating RNE pack.
//
// Every mbarrier wait is bounded (globaltimer); on expiry the warp raises
// DSPARK_FLAG_TIMEOUT, stops, waits (bounded) for its own copies in flight
// and returns.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "ctx_kv_device.cuh"
#include "ctx_kv_internal.h"
#include "ctx_kv_pipe.cuh"

namespace dspark {
namespace {

using namespace pipe;

constexpr int kWarps = 4;      // warps per CTA (8 or 16 measured slower on the draft steps)
constexpr int kStagesW = 3;    // stages per warp
constexpr int kCsSlotW = 128;  // one token's cos|sin row (2r <= 128 bytes)
constexpr unsigned kFlagSlotW = 0x1u, kFlagPosW = 0x2u, kFlagTimeoutW = 0x4u;

// per-warp shared memory: S barriers, S headers (the unit's row offsets per
// token, < 0: padding), an abort word, then S stages
template <int P>
struct WarpSmem {
    static constexpr uint32_t kSlab = 8 * 512;  // the unit's K|V rows: 8 (token, head) rows of 512 B
    static constexpr uint32_t kStage = (kSlab + P * kCsSlotW + 127) / 128 * 128;
    static constexpr uint32_t kHead = 256;  // barriers, headers, abort word
    static constexpr uint32_t kBytes = kHead + kStagesW * kStage;
};

struct WarpParams {
    CtxKvParams p;
};

// A device word that nothing ever sets: the test hook's wait (test_hold_ns)
// runs out on it.
__device__ unsigned g_never_set_w = 0;

__device__ __forceinline__ void fence_proxy_async_shared()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ROT: the rotary dim (16, 32, 64).  P: tokens per unit (1: 8 KV heads, 2: 4).
template <int ROT, bool FP8, int P>
__global__ void __launch_bounds__(32 * kWarps, 4) ctx_kv_warp_kernel(const WarpParams wp)
{
    constexpr int H = 8 / P;                    // KV heads
    constexpr int kCacheRow = FP8 ? 256 : 512;  // bytes of one cache row
    constexpr int kPartner = ROT / 16;          // lanes between RoPE partners
    constexpr int kRotLanes = ROT / 8;          // lanes whose first chunk is rotated
    constexpr int S = kStagesW;
    constexpr uint32_t kTokRows = 2 * H * 256;  // one token's K|V rows of one layer
    using Sm = WarpSmem<P>;
    extern __shared__ __align__(128) unsigned char smem[];
    const CtxKvParams &p = wp.p;
    const int L = p.num_layers;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned char *mine = smem + (size_t)warp * Sm::kBytes;
    uint64_t *full = reinterpret_cast<uint64_t *>(mine);              // [S]
    long long *hdr = reinterpret_cast<long long *>(mine + 64);        // [S][P] row offsets
    volatile int *abort = reinterpret_cast<volatile int *>(mine + 192);
    unsigned char *stages = mine + Sm::kHead;

    if (lane == 0) {
        for (int s = 0; s < S; s++)
            mbar_init(full + s, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncwarp();

    const long long T = p.num_ctx;
    const long long U = (T + P - 1) / P;            // token units
    const long long NS = (long long)gridDim.x * kWarps / L;  // token streams
    const long long gw = (long long)blockIdx.x * kWarps + warp;
    const int l = (int)(gw % L);
    const long long ts = gw / L;
    const long long n_my = gw < NS * L && ts < U ? (U - ts + NS - 1) / NS : 0;  // units of this warp
    auto unit_of = [&](long long o) { return ts + o * NS; };
    auto unit_tokens = [&](long long u) { return (int)min((long long)P, T - u * P); };
    const unsigned char *kv_layer = reinterpret_cast<const unsigned char *>(p.all_kv) + (size_t)l * kTokRows;
    const size_t tok_stride = (size_t)L * kTokRows;  // bytes between consecutive tokens in all_kv
    // While the previous kernel drains: this warp's first S units' K|V rows,
    // and the slots and positions of its first 32 units, into L2 (hints
    // only; the copies below still follow griddepcontrol.wait).
    if (n_my > 0) {
        if (lane < S && lane < n_my) {
            const long long u = unit_of(lane);
            for (int j = 0; j < unit_tokens(u); j++)
                prefetch_l2_bulk(kv_layer + (size_t)(u * P + j) * tok_stride, kTokRows);
        }
        if (lane < n_my) {
            const long long t = unit_of(lane) * P;
            prefetch_l2(p.slot_mapping + t);
            prefetch_l2(p.positions + t);
        }
    }
    pdl_enter();  // launched with launch_pdl: above, only barriers and L2 prefetch hints
    if (n_my == 0)
        return;  // no units (or a warp beyond the last whole set of L streams): idle
    const uint64_t stream_once = evict_first_policy();  // all_kv: read exactly once
    const uint64_t keep = evict_last_policy();          // cos|sin rows: shared by many tokens
    unsigned flags = 0;

    if (p.test_hold_ns) {
        // test hook: a bounded wait on a word nothing sets, which runs out;
        // the warp then stops before issuing anything
        if (lane == 0) {
            const unsigned long long t0 = globaltimer();
            while (*reinterpret_cast<volatile unsigned *>(&g_never_set_w) == 0 && globaltimer() - t0 < p.test_hold_ns) {
            }
            if (p.error_flags)
                atomicOr(p.error_flags, kFlagTimeoutW);
        }
        return;
    }

    // ---- slots and positions, one batch of 32 units ahead
    auto row_off = [&](long long slot) {
        return ((slot >> p.block_size_log2) * H * ((long long)1 << p.block_size_log2) +
                (slot & (((long long)1 << p.block_size_log2) - 1))) *
               kCacheRow;
    };
    // lane j: the P tokens of unit o = base + j (slot < 0: padding, past the
    // last token, or out of range -- flagged)
    auto fetch = [&](long long base, long long (&slot)[P], long long (&pos)[P]) {
        const long long o = base + lane;
#pragma unroll
        for (int j = 0; j < P; j++) {
            slot[j] = -1;
            pos[j] = 0;
            if (o < n_my) {
                const long long t = unit_of(o) * P + j;
                if (t < T) {
                    slot[j] = __ldg(p.slot_mapping + t);
                    pos[j] = __ldg(p.positions + t);
                }
            }
        }
    };
    auto vet = [&](long long (&slot)[P], const long long (&pos)[P]) {
#pragma unroll
        for (int j = 0; j < P; j++) {
            if (slot[j] < 0)
                continue;
            if (pos[j] < 0 || pos[j] >= p.max_pos) {
                flags |= kFlagPosW;
                slot[j] = -1;
            } else if (slot[j] >= p.capacity) {
                flags |= kFlagSlotW;
                slot[j] = -1;
            }
        }
    };
    long long cur_s[P], cur_p[P], nxt_s[P], nxt_p[P];
    fetch(0, cur_s, cur_p);  // first: the cos|sin copies wait on these positions
    // the layer's norm weights, cache offset and scales: issued now, used below
    const int q = lane & 7;    // 8-dim chunk of each 64-dim half of the row
    uint4 wraw[2];
#pragma unroll
    for (int c = 0; c < 2; c++)
        wraw[c] = __ldg(reinterpret_cast<const uint4 *>(p.knorm_w + l * 128 + 64 * c + 8 * q));
    const long long loff = __ldg(p.cache_offsets + l);
    float ksf = 1.0f, vsf = 1.0f;
    if (FP8) {
        ksf = __ldg(reinterpret_cast<const float *>(__ldg(reinterpret_cast<const unsigned long long *>(p.k_scales) + l)));
        vsf = __ldg(reinterpret_cast<const float *>(__ldg(reinterpret_cast<const unsigned long long *>(p.v_scales) + l)));
    }

    // ---- first S units: copied before their slots are known
    const int nspec = (int)min((long long)S, n_my);
    if (lane == 0) {
        for (int i = 0; i < nspec; i++) {
            const long long u = unit_of(i);
            const int n = unit_tokens(u);
            mbar_expect_tx(full + i, (uint32_t)n * kTokRows);
            for (int j = 0; j < n; j++)
                bulk_g2s(stages + (size_t)i * Sm::kStage + j * kTokRows, kv_layer + (size_t)(u * P + j) * tok_stride,
                         kTokRows, full + i, stream_once);
        }
    }

    // ---- per-layer constants, in registers for the whole launch
    const int rr = lane >> 3;  // row of the 4-row group
    const bool rot_lane = q < kRotLanes;
    uint64_t w1[8];  // (1 + w[l, d]) in fp32 for the lane's dims, as pairs
#pragma unroll
    for (int c = 0; c < 2; c++) {
        const uint32_t ww[4] = {wraw[c].x, wraw[c].y, wraw[c].z, wraw[c].w};
#pragma unroll
        for (int j = 0; j < 4; j++)
            w1[4 * c + j] = pr(1.0f + __uint_as_float(ww[j] << 16), 1.0f + __uint_as_float(ww[j] & 0xffff0000u));
    }
    unsigned char *const lbase = p.cache0 + loff * (FP8 ? 1 : 2);
    Fp8Scale kq{}, vq{};
    if (FP8) {
        kq = fp8_scale(ksf);
        vq = fp8_scale(vsf);
    }
    const long long head_bytes = (long long)kCacheRow << p.block_size_log2;
    // the two row groups of a unit: token tg[g], head hh[g]
    constexpr int tg[2] = {0, P - 1};
    const int hh[2] = {rr, P == 1 ? 4 + rr : rr};
    uint32_t koff[2];  // byte offset of the group's K row in a stage
#pragma unroll
    for (int g = 0; g < 2; g++)
        koff[g] = (uint32_t)(tg[g] * kTokRows + hh[g] * 256);

    vet(cur_s, cur_p);
    if (n_my > 32) {
        fetch(32, nxt_s, nxt_p);
        vet(nxt_s, nxt_p);
    } else {
#pragma unroll
        for (int j = 0; j < P; j++)
            nxt_s[j] = -1, nxt_p[j] = 0;
    }
    // the speculatively copied units: their headers and cos|sin rows now
#pragma unroll 1
    for (int i = 0; i < nspec; i++) {
        long long sl[P], po[P];
        int nvalid = 0;
#pragma unroll
        for (int j = 0; j < P; j++) {
            sl[j] = __shfl_sync(0xffffffffu, cur_s[j], i);
            po[j] = __shfl_sync(0xffffffffu, cur_p[j], i);
            nvalid += sl[j] >= 0;
        }
        if (lane == 0) {
#pragma unroll
            for (int j = 0; j < P; j++)
                hdr[i * P + j] = sl[j] >= 0 ? row_off(sl[j]) : -1;
            unsigned char *dst = stages + (size_t)i * Sm::kStage;
            mbar_arrive_expect_tx(full + i, (uint32_t)nvalid * 2u * ROT);
#pragma unroll
            for (int j = 0; j < P; j++)
                if (sl[j] >= 0)
                    bulk_g2s(dst + P * kTokRows + j * kCsSlotW, p.cos_sin + po[j] * ROT, 2u * ROT, full + i, keep);
        }
    }
    __syncwarp();

    uint32_t issued = nspec, consumed = 0;  // stages issued / consumed so far
    long long ip = nspec;                    // next unit to consider for a copy
    bool ok = true;
    for (long long b = 0; b < n_my && ok; b += 32) {
#pragma unroll 1
        for (int jj = 0; jj < 32; jj++) {
            const long long o = b + jj;
            if (o >= n_my)
                break;
            // ---- compute unit o, if it holds a stage
            bool any = false;
#pragma unroll
            for (int j = 0; j < P; j++)
                any |= __shfl_sync(0xffffffffu, cur_s[j], jj) >= 0;
            if (o < nspec || any) {
                const int s = (int)(consumed % S);
                if (!mbar_wait(full + s, (consumed / S) & 1u, abort)) {
                    ok = false;
                    break;
                }
                const unsigned char *stage = stages + (size_t)s * Sm::kStage;
                long long dst[2];
#pragma unroll
                for (int g = 0; g < 2; g++)
                    dst[g] = hdr[s * P + tg[g]];
                // cos and sign * sin (bf16 pairs) of each group's token for the lane's first 8 dims
                uint32_t cw[2][4], sw[2][4];
#pragma unroll
                for (int g = 0; g < 2; g++) {
#pragma unroll
                    for (int j = 0; j < 4; j++)
                        cw[g][j] = sw[g][j] = 0;
                    if (g == 0 || P > 1) {
                        if (rot_lane) {
                            const unsigned char *cs =
                                stage + P * kTokRows + tg[g] * kCsSlotW + 16 * (q & (kPartner - 1));
                            const uint4 c4 = lds128(cs), s4 = lds128(cs + ROT);  // sin half: r/2 elements later
                            const uint32_t flip = (q & kPartner) ? 0u : 0x80008000u;  // lower half subtracts
                            cw[g][0] = c4.x, cw[g][1] = c4.y, cw[g][2] = c4.z, cw[g][3] = c4.w;
                            sw[g][0] = s4.x ^ flip, sw[g][1] = s4.y ^ flip, sw[g][2] = s4.z ^ flip,
                            sw[g][3] = s4.w ^ flip;
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; j++)
                            cw[g][j] = cw[0][j], sw[g][j] = sw[0][j];
                    }
                }
                // K: load, sum of squares
                uint64_t x2[2][8];
                float ss[2];
#pragma unroll
                for (int g = 0; g < 2; g++) {
#pragma unroll
                    for (int c = 0; c < 2; c++) {
                        const uint4 a = lds128(stage + koff[g] + 128 * c + 16 * q);
                        x2[g][4 * c] = bf2_to_f2(a.x), x2[g][4 * c + 1] = bf2_to_f2(a.y);
                        x2[g][4 * c + 2] = bf2_to_f2(a.z), x2[g][4 * c + 3] = bf2_to_f2(a.w);
                    }
                    uint64_t a0 = mul2(x2[g][0], x2[g][0]), a1 = mul2(x2[g][1], x2[g][1]);
#pragma unroll
                    for (int j = 2; j < 8; j += 2) {
                        a0 = fma2(x2[g][j], x2[g][j], a0);
                        a1 = fma2(x2[g][j + 1], x2[g][j + 1], a1);
                    }
                    float slo, shi;
                    unpr(add2(a0, a1), slo, shi);
                    ss[g] = slo + shi;
                }
#pragma unroll
                for (int m = 4; m >= 1; m >>= 1)
#pragma unroll
                    for (int g = 0; g < 2; g++)
                        ss[g] += __shfl_xor_sync(0xffffffffu, ss[g], m);
                uint32_t ko[2][8];
#pragma unroll
                for (int g = 0; g < 2; g++) {
                    float inv;  // ss/128 + eps >= eps > 0 (hardware reciprocal square root)
                    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(fmaf(ss[g], 1.0f / 128, p.eps)));
                    const uint64_t inv2 = pr(inv, inv);
                    // y = bf16((k * inv) * (1 + w))
#pragma unroll
                    for (int j = 0; j < 8; j++)
                        ko[g][j] = f2_to_bf2(mul2(mul2(x2[g][j], inv2), w1[j]));
                }
                // RoPE on the first chunk (dims 8q .. 8q+7); the partner is kPartner lanes away
#pragma unroll
                for (int g = 0; g < 2; g++)
#pragma unroll
                    for (int j = 0; j < 4; j++) {
                        const uint32_t yp = __shfl_xor_sync(0xffffffffu, ko[g][j], kPartner);
                        const uint32_t rv = f2_to_bf2(rope_bf2(ko[g][j], cw[g][j], yp, sw[g][j]));
                        ko[g][j] = rot_lane ? rv : ko[g][j];  // both computed: a select, not a branch
                    }
#pragma unroll
                for (int g = 0; g < 2; g++) {
                    if (dst[g] < 0)
                        continue;  // a padded token of the unit
                    unsigned char *dg = lbase + dst[g] + hh[g] * head_bytes;
                    const unsigned char *vrow = stage + koff[g] + H * 256;
                    if (!FP8) {
#pragma unroll
                        for (int c = 0; c < 2; c++)
                            st_stream_v4(dg + 128 * c + 16 * q,
                                         make_uint4(ko[g][4 * c], ko[g][4 * c + 1], ko[g][4 * c + 2], ko[g][4 * c + 3]));
#pragma unroll
                        for (int c = 0; c < 2; c++)
                            st_stream_v4(dg + 256 + 128 * c + 16 * q, lds128(vrow + 128 * c + 16 * q));
                    } else {
#pragma unroll
                        for (int c = 0; c < 2; c++)
                            st_stream_v2(dg + 64 * c + 8 * q,
                                         quantise8(make_uint4(ko[g][4 * c], ko[g][4 * c + 1], ko[g][4 * c + 2],
                                                              ko[g][4 * c + 3]),
                                                   kq));
#pragma unroll
                        for (int c = 0; c < 2; c++)
                            st_stream_v2(dg + 128 + 64 * c + 8 * q, quantise8(lds128(vrow + 128 * c + 16 * q), vq));
                    }
                }
                consumed++;
                __syncwarp();  // every lane's reads of the stage are done before it is refilled
            }
            // ---- copies up to S units ahead (within this batch and the next)
            const long long ip_end = min(n_my, b + 64);
            while (issued - consumed < (uint32_t)S && ip < ip_end) {
                const bool in_cur = ip < b + 32;
                const int src = (int)(ip - b) & 31;
                long long sl[P], po[P];
                int nvalid = 0;
#pragma unroll
                for (int j = 0; j < P; j++) {
                    sl[j] = __shfl_sync(0xffffffffu, in_cur ? cur_s[j] : nxt_s[j], src);
                    po[j] = __shfl_sync(0xffffffffu, in_cur ? cur_p[j] : nxt_p[j], src);
                    nvalid += sl[j] >= 0;
                }
                if (nvalid > 0) {
                    if (lane == 0) {
                        const int s = (int)(issued % S);
                        const long long u = unit_of(ip);
                        unsigned char *dst = stages + (size_t)s * Sm::kStage;
#pragma unroll
                        for (int j = 0; j < P; j++)
                            hdr[s * P + j] = sl[j] >= 0 ? row_off(sl[j]) : -1;
                        fence_proxy_async_shared();  // the stage's earlier reads before the copies refill it
                        mbar_arrive_expect_tx(full + s, (uint32_t)nvalid * (kTokRows + 2u * ROT));
#pragma unroll
                        for (int j = 0; j < P; j++)
                            if (sl[j] >= 0) {
                                bulk_g2s(dst + j * kTokRows, kv_layer + (size_t)(u * P + j) * tok_stride, kTokRows,
                                         full + s, stream_once);
                                bulk_g2s(dst + P * kTokRows + j * kCsSlotW, p.cos_sin + po[j] * ROT, 2u * ROT,
                                         full + s, keep);
                            }
                    }
                    issued++;
                }
                ip++;
            }
        }
        // advance the slot batches
#pragma unroll
        for (int j = 0; j < P; j++)
            cur_s[j] = nxt_s[j], cur_p[j] = nxt_p[j];
        if (b + 64 < n_my) {
            fetch(b + 64, nxt_s, nxt_p);
            vet(nxt_s, nxt_p);
        } else {
#pragma unroll
            for (int j = 0; j < P; j++)
                nxt_s[j] = -1, nxt_p[j] = 0;
        }
    }
    if (!ok) {
        flags |= kFlagTimeoutW;
        // drain: the copies still in flight land before the warp exits
        if (lane == 0) {
            for (uint32_t k = consumed; k < issued; k++) {
                const int s = (int)(k % S);
                const unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(full + s, (k / S) & 1u) && globaltimer() - t0 < kTimeoutNs) {
                }
            }
        }
        __syncwarp();
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (lane == 0 && flags && p.error_flags)
        atomicOr(p.error_flags, flags);
}

template <int P>
constexpr uint32_t warp_smem_bytes()
{
    return kWarps * WarpSmem<P>::kBytes;
}

template <int ROT, bool FP8, int P>
cudaError_t launch_warp_variant(const WarpParams &wp, cudaStream_t stream)
{
    static std::mutex mu;
    static int blocks_cache[64];
    static bool smem_set[64];
    constexpr uint32_t smem = warp_smem_bytes<P>();
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    int per_sm, sms;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!smem_set[dev]) {
            e = cudaFuncSetAttribute(ctx_kv_warp_kernel<ROT, FP8, P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem);
            if (e != cudaSuccess)
                return e;
            smem_set[dev] = true;
        }
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess)
            return e;
        if (blocks_cache[dev] == 0) {
            int b = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, ctx_kv_warp_kernel<ROT, FP8, P>, 32 * kWarps, smem);
            if (e != cudaSuccess)
                return e;
            blocks_cache[dev] = std::max(1, b);
        }
        per_sm = blocks_cache[dev];
    }
    // as many warps as fit, but no more streams than token units; at least
    // one whole set of L warps
    const long long L = wp.p.num_layers;
    const long long units = (wp.p.num_ctx + P - 1) / P;
    long long warps = (long long)per_sm * sms * kWarps;
    warps = std::min(warps, units * L);
    warps = std::max(warps, L);
    const int blocks = (int)((warps + kWarps - 1) / kWarps);
    return launch_pdl(ctx_kv_warp_kernel<ROT, FP8, P>, blocks, 32 * kWarps, smem, stream, wp);
}

template <bool FP8, int P>
cudaError_t launch_warp_rot(const WarpParams &wp, cudaStream_t stream)
{
    switch (wp.p.rotary_dim) {
    case 16:
        return launch_warp_variant<16, FP8, P>(wp, stream);
    case 32:
        return launch_warp_variant<32, FP8, P>(wp, stream);
    default:
        return launch_warp_variant<64, FP8, P>(wp, stream);
    }
}

}  // namespace

bool warp_path_supported(const CtxKvParams &p)
{
    const int H = p.num_kv_heads;
    return (H == 4 || H == 8) && !p.layer_slots && p.block_size_log2 >= 0 && p.num_layers >= 1 &&
           (p.rotary_dim == 16 || p.rotary_dim == 32 || p.rotary_dim == 64);
}

cudaError_t launch_ctx_kv_write_warp(const CtxKvParams &p, bool fp8, cudaStream_t stream)
{
    if (!warp_path_supported(p))
        return cudaErrorInvalidValue;
    WarpParams wp;
    wp.p = p;
    if (p.num_kv_heads == 8)
        return fp8 ? launch_warp_rot<true, 1>(wp, stream) : launch_warp_rot<false, 1>(wp, stream);
    return fp8 ? launch_warp_rot<true, 2>(wp, stream) : launch_warp_rot<false, 2>(wp, stream);
}

}  // namespace dspark
