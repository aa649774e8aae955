// sm_103a tensor-core kernel of the fused context-KV projection, alone or
// with the context-KV write in its epilogue.
//
// Defining passages: DSpark draft model page, precompute_and_store_context_kv
// (all_kv = _project_context_kv_token_major(context_states, ...), then the
// fused writer), and the context-KV writer page (module docstring: all_kv
// [num_ctx, L, 2, nkv, 128]; Gemma RMSNorm of K in fp32 materialised to bf16,
// partial NeoX RoPE, fp8 of x / scale, slots < 0 not written).
//
// all_kv[t, n] = bf16(sum_k x[t, k] w[n, k]) with x [T, hidden] (context
// states) and w [N, hidden] (N = L * 2 * nkv * 128, row ((l*2 + kv)*nkv + h)
// * 128 + d), both bf16 and K-major: a TN GEMM with an fp32 accumulator.
//
// Tiling.  A tile is 128 tokens x 256 columns: the K rows and the V rows of
// one (layer, head), i.e. exactly the two 128-element halves of the head's
// cache rows, so the write needs no other tile.  One persistent CTA per SM
// walks the tiles (groups of 16 column tiles, all row tiles of a group
// before the next, so the running CTAs share their weights and x rows in
// L2) with two tensor-memory accumulators: the epilogue of one tile runs
// while the MMAs of the next fill the other accumulator.  Per 64-wide k-block a
// TMA producer warp loads the x tile (128 x 64) and the two weight boxes
// (128 x 64 each) into a 4-stage shared-memory ring with 128-byte swizzle;
// one thread of an MMA warp issues four tcgen05.mma (M 128, N 256, K 16,
// bf16 in, fp32 accumulate in tensor memory) per k-block and frees the stage
// with tcgen05.commit; the last commit wakes four epilogue warps, which read
// the accumulator with tcgen05.ld (thread = token row) and either store the
// bf16 projection or run the write: round to bf16 (all_kv as the unfused
// path materialises it), Gemma norm of K, RoPE (both dims of a rotated pair
// sit in the same thread), bf16 or exact-quotient fp8 encode, and 512 / 256
// contiguous bytes per (token, head) into the layer's paged cache.  all_kv
// never reaches HBM.
//
// Tall tiles (calls of at most 2,048 tokens where they save a wave): 256
// tokens x 256 columns, two x boxes per k-block against the same weight
// boxes, eight MMAs per k-block into both accumulators, three 64 KB stages;
// the epilogue runs the same code over the two 128-row halves.
//
// Every mbarrier wait is bounded (globaltimer); on expiry the CTA raises
// DSPARK_FLAG_TIMEOUT, stops issuing, waits (bounded) for its own copies and
// MMAs in flight, frees its tensor memory and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdlib>
#include <cstring>
#include <mutex>

#include "ctx_kv_device.cuh"
#include "ctx_kv_internal.h"

namespace dspark {
namespace {

constexpr int BM = 128, BN = 256, BK = 64, kStages = 4;
constexpr int kThreadsG = 192;                             // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr uint32_t kABytes = BM * BK * 2;                  // 16 KB
constexpr uint32_t kBoxBytes = 128 * BK * 2;               // one 128-row weight box, 16 KB
constexpr uint32_t kTmemCols = 512;  // two 256-column accumulators: the epilogue of one tile overlaps the next
constexpr int kMaxLayersProj = 32;   // the (1 + w) table of every layer lives in shared memory
constexpr int kGroupN = 16;          // column tiles per rasterisation group
// Tile shape.  Short tiles (128 tokens) keep the two accumulators apart, so
// the epilogue of one tile overlaps the MMAs of the next.  Tall tiles (256
// tokens: two 128-row A boxes per k-block against the same two weight boxes,
// one accumulator each) hold 64 KB of operands per k-block for twice the
// flops of a short tile's 48 KB, and halve the tile count; their epilogue
// does not overlap the next tile's MMAs (both accumulators are in use).
template <bool TALL>
struct TileCfg {
    static constexpr int kRows = TALL ? 256 : BM;                       // tokens per tile
    static constexpr int kStagesC = TALL ? 3 : kStages;                 // k-blocks in flight
    static constexpr uint32_t kAPart = TALL ? 2 * kABytes : kABytes;    // x boxes of a stage
    static constexpr uint32_t kStage = kAPart + 2 * kBoxBytes;          // 64 KB / 48 KB
    static constexpr uint32_t kSmem = kStagesC * kStage + 1024 /* alignment pad */ + 256 /* barriers */ +
                                      kMaxLayersProj * 128 * 4 /* (1 + w) table */;
};
static_assert(TileCfg<true>::kSmem <= 227 * 1024 && TileCfg<false>::kSmem <= 227 * 1024, "shared memory");
constexpr unsigned kFlagSlot = 0x1u, kFlagPos = 0x2u, kFlagTimeout = 0x4u;
constexpr unsigned long long kTimeoutNs = 4000000000ull;
constexpr uint32_t kSuspendNs = 200000;

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5), A and B
// bf16 (bits 7-9, 10-12), both K-major (bits 15, 16 clear), N >> 3 at bit 17,
// M >> 4 at bit 24.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) |
                            ((uint32_t)(BM >> 4) << 24);

enum { kModeProject = 0, kModeWrite = 1 };

struct GemmParams {
    int64_t T;
    int32_t hidden, L, nkv, num_kb;
    uint16_t *all_kv_out;  // project: [T, L * 2 * nkv * 128]
    // write
    const uint16_t *knorm_w;
    const int64_t *positions, *slot_mapping;
    const uint16_t *cos_sin;
    unsigned char *cache0;
    const int64_t *cache_offsets;
    const float *const *k_scales;
    const float *const *v_scales;
    unsigned int *error_flags;
    int64_t max_pos, capacity;
    int32_t bsl;
    float eps;
};

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t saddr(const void *p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

__device__ __forceinline__ unsigned long long gtimer()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(saddr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_arrive(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(saddr(bar)), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(saddr(bar)), "r"(parity), "n"(kSuspendNs)
        : "memory");
    return ok != 0;
}

// Waits for the phase of `bar` with this parity; false after kTimeoutNs or
// once another warp of the CTA has given up (which it then records).
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile int *abort)
{
    if (mbar_try(bar, parity))
        return true;
    const unsigned long long t0 = gtimer();
    while (true) {
        if (mbar_try(bar, parity))
            return true;
        if (*abort)
            return false;
        if (gtimer() - t0 > kTimeoutNs) {
            *abort = 1;
            return false;
        }
    }
}

// 2-D tiled TMA load (x = inner coordinate, a multiple of 64 elements here).
__device__ __forceinline__ void tma_load(void *dst, const CUtensorMap *map, int32_t x, int32_t y, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            saddr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(saddr(bar))
        : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major tile written by TMA with
// 128-byte swizzle: rows of 64 bf16 (128 B), 8-row atoms 1024 B apart
// (stride byte offset), descriptor version 1 (bits 46-48), swizzle mode 2
// (128 B, bits 61-63); the leading byte offset is unused for this layout.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t addr)
{
    return (uint64_t)((addr & 0x3FFFFu) >> 4) | ((uint64_t)1 << 16) | ((uint64_t)(1024 >> 4) << 32) |
           ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}

__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(kIdesc), "r"(accumulate)
        : "memory");
}

// The mbarrier arrives once every tcgen05.mma this thread issued so far has completed.
__device__ __forceinline__ void mma_commit(uint64_t *bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(saddr(bar))
                 : "memory");
}

// 32 consecutive fp32 columns of the accumulator for this thread's lane.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}

__device__ __forceinline__ float bfl(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bfh(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// RoPE on a bf16 pair: y * c + yp * sn per half, one rounding (the partner
// product of two bf16 values is exact in fp32; an FMA with -0 keeps the sign
// of a zero product).
__device__ __forceinline__ uint32_t rope_pair(uint32_t y, uint32_t c, uint32_t yp, uint32_t sn)
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
    return pack_bf16x2(lo, hi);
}

__device__ __forceinline__ void st16(void *p, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    *reinterpret_cast<uint4 *>(p) = make_uint4(a, b, c, d);
}

// Tile order: groups of kGroupN column tiles (one (layer, head) each), all
// row tiles of a group before the next group, so that the CTAs running at
// any one time share a few MB of weights and x rows (both stay in L2).
__device__ __forceinline__ void tile_coords(int tile, int num_m, int num_n, int &m, int &n)
{
    const int per_group = kGroupN * num_m;
    const int g = tile / per_group;
    const int r = tile - g * per_group;
    const int gn = min(kGroupN, num_n - g * kGroupN);
    m = r / gn;
    n = g * kGroupN + (r - m * gn);
}

template <int MODE, int ROT, bool FP8, bool TALL>
__global__ void __launch_bounds__(kThreadsG, 1)
    proj_gemm_kernel(const __grid_constant__ CUtensorMap tmx, const __grid_constant__ CUtensorMap tmw,
                     const GemmParams p)
{
    using C = TileCfg<TALL>;
    constexpr int KS = C::kStagesC;
    constexpr int NH = TALL ? 2 : 1;  // 128-row accumulators per tile
    extern __shared__ unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (saddr(smem_raw) & 1023u)) & 1023u);  // 1024-aligned for the swizzle
    unsigned char *stages = smem;
    unsigned char *ctl = smem + KS * C::kStage;
    uint64_t *full = reinterpret_cast<uint64_t *>(ctl);  // TMA -> MMA, per stage
    uint64_t *empty = full + KS;                           // MMA -> TMA, per stage
    uint64_t *acc_full = empty + KS;                       // MMA -> epilogue, per accumulator (tall: the pair)
    uint64_t *acc_empty = acc_full + 2;                    // epilogue -> MMA, per accumulator
    uint64_t *done = acc_empty + 2;                        // every MMA of the CTA has completed
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(done + 1);
    volatile int *abort = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *w1 = reinterpret_cast<float *>(ctl + 256);      // (1 + w) of every layer, [L][128]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int num_m = (int)((p.T + C::kRows - 1) / C::kRows), num_n = p.L * p.nkv;
    const int num_tiles = num_m * num_n;

    if (threadIdx.x == 0) {
        for (int s = 0; s < KS; s++) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(acc_full + b, 1);
            mbar_init(acc_empty + b, 4);  // one arrive per epilogue warp
        }
        mbar_init(done, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmx)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmw)) : "memory");
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         saddr(const_cast<uint32_t *>(tmem_slot))),
                     "r"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    if (MODE == kModeWrite && warp >= 2) {
        for (int i = threadIdx.x - 64; i < p.L * 128; i += 128)
            w1[i] = 1.0f + bfl((uint32_t)__ldg(p.knorm_w + i));
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    unsigned flags = 0;

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            int issued = 0;  // k-blocks issued over all tiles
            bool ok = true;
            for (int tile = blockIdx.x; tile < num_tiles && ok; tile += gridDim.x) {
                int m, n;
                tile_coords(tile, num_m, num_n, m, n);
                const int l = n / p.nkv, h = n - l * p.nkv;
                const int nk = ((l * 2 + 0) * p.nkv + h) * 128, nv = ((l * 2 + 1) * p.nkv + h) * 128;
                for (int kb = 0; kb < p.num_kb; kb++) {
                    const int s = issued % KS;
                    if (!mbar_wait(empty + s, ((uint32_t)(issued / KS) & 1u) ^ 1u, abort)) {
                        ok = false;
                        break;
                    }
                    unsigned char *st = stages + s * C::kStage;
                    mbar_expect_arrive(full + s, C::kStage);
                    tma_load(st, &tmx, kb * BK, m * C::kRows, full + s);
                    if (TALL)  // rows past the end of x arrive as zeros
                        tma_load(st + kABytes, &tmx, kb * BK, m * C::kRows + BM, full + s);
                    tma_load(st + C::kAPart, &tmw, kb * BK, nk, full + s);
                    tma_load(st + C::kAPart + kBoxBytes, &tmw, kb * BK, nv, full + s);
                    issued++;
                }
            }
            // the copies of the last rounds may still be landing: wait (bounded)
            for (int it = issued > KS ? issued - KS : 0; it < issued; it++) {
                const unsigned long long t0 = gtimer();
                while (!mbar_try(full + it % KS, (uint32_t)(it / KS) & 1u) && gtimer() - t0 < kTimeoutNs) {
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int it = 0;  // k-blocks consumed over all tiles
            bool ok = true;
            for (int tile = blockIdx.x, i = 0; tile < num_tiles && ok; tile += gridDim.x, i++) {
                const int b = TALL ? 0 : i & 1;            // tall: the pair, every tile
                const uint32_t use = TALL ? i : (i >> 1);  // earlier uses of this accumulator
                // the epilogue has drained this accumulator (its previous use)
                if (!mbar_wait(acc_empty + b, (use & 1u) ^ 1u, abort))
                    break;
                tc_fence_after();
                const uint32_t d = tmem + (uint32_t)(b * BN);
                for (int kb = 0; kb < p.num_kb; kb++, it++) {
                    const int s = it % KS;
                    if (!mbar_wait(full + s, (uint32_t)(it / KS) & 1u, abort)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a = saddr(stages + s * C::kStage);
                    const uint32_t bb = a + C::kAPart;
#pragma unroll
                    for (int k = 0; k < BK / 16; k++) {  // 16 bf16 = 32 bytes per step along K
                        mma_bf16(d, sw128_desc(a + 32 * k), sw128_desc(bb + 32 * k), (kb | k) != 0);
                        if (TALL)  // rows 128..255 of the tile into the second accumulator
                            mma_bf16(d + BN, sw128_desc(a + kABytes + 32 * k), sw128_desc(bb + 32 * k), (kb | k) != 0);
                    }
                    mma_commit(empty + s);
                }
                if (ok)
                    mma_commit(acc_full + b);
            }
            mma_commit(done);  // fires once every MMA issued above has completed
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int q4 = warp & 3;  // the TMEM lane quarter this warp may access
        const int row = q4 * 32 + lane;
        for (int tile = blockIdx.x, i = 0; tile < num_tiles; tile += gridDim.x, i++) {
            const int b = TALL ? 0 : i & 1;            // tall: the pair, every tile
            const uint32_t use = TALL ? i : (i >> 1);  // earlier uses of this accumulator
            int m, n;
            tile_coords(tile, num_m, num_n, m, n);
            const int l = n / p.nkv, h = n - l * p.nkv;
            // this thread's token in each 128-row half of the tile, with its
            // slot and position (loaded before the accumulator is ready)
            int64_t t_h[NH], slot_h[NH], pos_h[NH];
#pragma unroll
            for (int hf = 0; hf < NH; hf++) {
                const int64_t t = (int64_t)m * C::kRows + hf * BM + row;
                int64_t slot = -1, pos = 0;
                if (MODE == kModeWrite && t < p.T) {
                    slot = __ldg(p.slot_mapping + t);
                    if (slot >= 0) {
                        pos = __ldg(p.positions + t);
                        if (slot >= p.capacity) {
                            if (n == 0)
                                flags |= kFlagSlot;
                            slot = -1;
                        } else if (pos < 0 || pos >= p.max_pos) {
                            if (n == 0)
                                flags |= kFlagPos;
                            slot = -1;
                        }
                    }
                }
                t_h[hf] = t, slot_h[hf] = slot, pos_h[hf] = pos;
            }
            bool ok = mbar_wait(acc_full + b, use & 1u, abort);
            ok = __all_sync(0xffffffffu, ok) && !*abort;
            if (!ok)
                break;
            tc_fence_after();
#pragma unroll 1
            for (int hf = 0; hf < NH; hf++) {
                const int64_t t = t_h[hf], slot = slot_h[hf], pos = pos_h[hf];
                const bool last = hf == NH - 1;  // the tile's last read hands its accumulator(s) back
                const uint32_t trow = tmem + (uint32_t)((b + hf) * BN) + ((uint32_t)(q4 * 32) << 16);
                if (MODE == kModeProject) {
                    const int64_t N = (int64_t)p.L * 2 * p.nkv * 128;
                    const int nk = ((l * 2 + 0) * p.nkv + h) * 128, nv = ((l * 2 + 1) * p.nkv + h) * 128;
#pragma unroll 1
                    for (int c = 0; c < 8; c++) {
                        uint32_t r[32];
                        tmem_ld32(trow + 32 * c, r);  // every lane: the load is warp-wide
                        if (c == 7 && last) {                 // the accumulator is read: hand it back
                            tc_fence_before();
                            __syncwarp();
                            if (lane == 0)
                                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(acc_empty + b))
                                             : "memory");
                        }
                        if (t < p.T) {
                            uint32_t pk[16];
#pragma unroll
                            for (int j = 0; j < 16; j++)
                                pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                            uint16_t *dst = p.all_kv_out + t * N + (c < 4 ? nk + 32 * c : nv + 32 * (c - 4));
#pragma unroll
                            for (int k = 0; k < 4; k++)
                                st16(dst + 8 * k, pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                        }
                    }
                    continue;
                }
                // K: bf16 as the projection materialises it, then the Gemma norm in fp32
                uint32_t kw[64];
                float ss = 0.0f;
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    uint32_t r[32];
                    tmem_ld32(trow + 32 * c, r);
#pragma unroll
                    for (int j = 0; j < 16; j++) {
                        const uint32_t pk = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                        kw[16 * c + j] = pk;
                        ss = fmaf(bfl(pk), bfl(pk), ss);
                        ss = fmaf(bfh(pk), bfh(pk), ss);
                    }
                }
                float inv;  // ss/128 + eps >= eps > 0 (hardware reciprocal square root)
                asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(fmaf(ss, 1.0f / kHeadDim, p.eps)));
                const float *wl = w1 + l * 128;
#pragma unroll
                for (int j = 0; j < 64; j++)
                    kw[j] = pack_bf16x2((bfl(kw[j]) * inv) * wl[2 * j], (bfh(kw[j]) * inv) * wl[2 * j + 1]);
                unsigned char *dst = nullptr;
                Fp8Scale vq;
                if (slot >= 0) {
                    // RoPE: dims j and j + r/2 (both in this thread), cos|sin of the token's position
                    uint32_t cs[ROT / 2];
                    const uint4 *src = reinterpret_cast<const uint4 *>(p.cos_sin + pos * ROT);
#pragma unroll
                    for (int k = 0; k < ROT / 8; k++) {
                        const uint4 v = __ldg(src + k);
                        cs[4 * k] = v.x, cs[4 * k + 1] = v.y, cs[4 * k + 2] = v.z, cs[4 * k + 3] = v.w;
                    }
#pragma unroll
                    for (int j = 0; j < ROT / 4; j++) {
                        const uint32_t a = kw[j], bb = kw[j + ROT / 4], c = cs[j], s = cs[ROT / 4 + j];
                        kw[j] = rope_pair(a, c, bb, s ^ 0x80008000u);  // a c - b s
                        kw[j + ROT / 4] = rope_pair(bb, c, a, s);      // b c + a s
                    }
                    const int64_t rowel =
                        ((((slot >> p.bsl) * p.nkv + h) << p.bsl) + (slot & ((int64_t(1) << p.bsl) - 1))) * kRowElems;
                    dst = p.cache0 + (__ldg(p.cache_offsets + l) + rowel) * (FP8 ? 1 : 2);
                    if (FP8) {
                        const Fp8Scale kq = fp8_scale(__ldg(reinterpret_cast<const float *>(
                            __ldg(reinterpret_cast<const unsigned long long *>(p.k_scales) + l))));
                        vq = fp8_scale(__ldg(reinterpret_cast<const float *>(
                            __ldg(reinterpret_cast<const unsigned long long *>(p.v_scales) + l))));
#pragma unroll
                        for (int k = 0; k < 8; k++) {
                            const uint2 lo =
                                quantise8(make_uint4(kw[8 * k], kw[8 * k + 1], kw[8 * k + 2], kw[8 * k + 3]), kq);
                            const uint2 hi =
                                quantise8(make_uint4(kw[8 * k + 4], kw[8 * k + 5], kw[8 * k + 6], kw[8 * k + 7]), kq);
                            st16(dst + 16 * k, lo.x, lo.y, hi.x, hi.y);
                        }
                    } else {
#pragma unroll
                        for (int k = 0; k < 16; k++)
                            st16(dst + 16 * k, kw[4 * k], kw[4 * k + 1], kw[4 * k + 2], kw[4 * k + 3]);
                    }
                }
                // V: bf16 as materialised, stored as it is (or encoded); after its
                // last read the accumulator is handed back to the MMA warp
#pragma unroll
                for (int c = 0; c < 4; c++) {
                    uint32_t r[32];
                    tmem_ld32(trow + 128 + 32 * c, r);
                    if (c == 3 && last) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(saddr(acc_empty + b)) : "memory");
                    }
                    if (slot >= 0) {
                        uint32_t pk[16];
#pragma unroll
                        for (int j = 0; j < 16; j++)
                            pk[j] = pack_bf16x2(__uint_as_float(r[2 * j]), __uint_as_float(r[2 * j + 1]));
                        if (FP8) {
#pragma unroll
                            for (int k = 0; k < 2; k++) {
                                const uint2 lo =
                                    quantise8(make_uint4(pk[8 * k], pk[8 * k + 1], pk[8 * k + 2], pk[8 * k + 3]), vq);
                                const uint2 hi =
                                    quantise8(make_uint4(pk[8 * k + 4], pk[8 * k + 5], pk[8 * k + 6], pk[8 * k + 7]), vq);
                                st16(dst + 128 + 32 * c + 16 * k, lo.x, lo.y, hi.x, hi.y);
                            }
                        } else {
#pragma unroll
                            for (int k = 0; k < 4; k++)
                                st16(dst + 256 + 64 * c + 16 * k, pk[4 * k], pk[4 * k + 1], pk[4 * k + 2], pk[4 * k + 3]);
                        }
                    }
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) {
        // every MMA has completed before the accumulators are freed (the
        // epilogue may have stopped waiting after an abort)
        if (lane == 0) {
            const unsigned long long t0 = gtimer();
            while (!mbar_try(done, 0) && gtimer() - t0 < kTimeoutNs) {
            }
        }
        __syncwarp();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
    }
    if (threadIdx.x == 0 && *abort)
        flags |= kFlagTimeout;
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (lane == 0 && flags && p.error_flags)
        atomicOr(p.error_flags, flags);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// A [outer, inner] bf16 row-major matrix as 64 x 128 boxes with 128-byte swizzle.
bool encode_kmajor(CUtensorMap *map, const void *ptr, uint64_t inner, uint64_t outer)
{
    const PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
    if (!fn)
        return false;
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {inner * 2};
    const cuuint32_t box[2] = {(cuuint32_t)BK, 128u};
    const cuuint32_t es[2] = {1u, 1u};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box, es,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gemm_sms(cudaError_t &e)
{
    static std::mutex mu;
    static int sms_cache[64];
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return 0;
    if (dev < 0 || dev >= 64) {
        e = cudaErrorInvalidDevice;
        return 0;
    }
    std::lock_guard<std::mutex> lock(mu);
    if (sms_cache[dev] == 0)
        e = cudaDeviceGetAttribute(&sms_cache[dev], cudaDevAttrMultiProcessorCount, dev);
    return sms_cache[dev];
}

// Tall tiles where they save whole waves on a small call: the short tiles'
// waves against 1.4 x the tall tiles' (a tall tile is twice the work at
// about 1.4 x the short tile's time, being fed 50% more flops per operand
// byte), up to 2,048 tokens; larger calls keep the overlapped epilogue.
bool use_tall(int64_t T, int64_t num_n, int sms)
{
    const char *env = std::getenv("DSPARK_PROJ_TILE");  // tests: "tall" or "short" pins one
    if (env && std::strcmp(env, "tall") == 0)
        return true;
    if (env && std::strcmp(env, "short") == 0)
        return false;
    if (T > 2048 || sms <= 0)
        return false;
    const int64_t waves_short = (num_n * ((T + BM - 1) / BM) + sms - 1) / sms;
    const int64_t waves_tall = (num_n * ((T + 255) / 256) + sms - 1) / sms;
    return (double)waves_short > 1.4 * (double)waves_tall;
}

template <int MODE, int ROT, bool FP8, bool TALL>
cudaError_t launch_gemm(const CUtensorMap &tx, const CUtensorMap &tw, const GemmParams &p, int sms,
                        cudaStream_t stream)
{
    using C = TileCfg<TALL>;
    static std::mutex mu;
    static bool attr_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (!attr_set[dev]) {
            e = cudaFuncSetAttribute(proj_gemm_kernel<MODE, ROT, FP8, TALL>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::kSmem);
            if (e != cudaSuccess)
                return e;
            attr_set[dev] = true;
        }
    }
    // persistent: one CTA per SM (the shared-memory ring holds one), each
    // walking the tile order with a stride of the grid
    const int64_t tiles = (int64_t)p.L * p.nkv * ((p.T + C::kRows - 1) / C::kRows);
    const int grid = (int)(tiles < sms ? tiles : sms);
    proj_gemm_kernel<MODE, ROT, FP8, TALL><<<grid, kThreadsG, C::kSmem, stream>>>(tx, tw, p);
    return cudaGetLastError();
}

template <int MODE, int ROT, bool FP8>
cudaError_t launch_gemm(const CUtensorMap &tx, const CUtensorMap &tw, const GemmParams &p, cudaStream_t stream)
{
    cudaError_t e = cudaSuccess;
    const int sms = gemm_sms(e);
    if (e != cudaSuccess)
        return e;
    return use_tall(p.T, (int64_t)p.L * p.nkv, sms) ? launch_gemm<MODE, ROT, FP8, true>(tx, tw, p, sms, stream)
                                                     : launch_gemm<MODE, ROT, FP8, false>(tx, tw, p, sms, stream);
}

}  // namespace

cudaError_t launch_proj(const ProjArgs &a, cudaStream_t stream)
{
    CUtensorMap tx, tw;
    const int64_t N = (int64_t)a.L * 2 * a.nkv * 128;
    if (!encode_kmajor(&tx, a.x, (uint64_t)a.hidden, (uint64_t)a.T) ||
        !encode_kmajor(&tw, a.w_kv, (uint64_t)a.hidden, (uint64_t)N))
        return cudaErrorInvalidValue;
    GemmParams p{};
    p.T = a.T;
    p.hidden = a.hidden;
    p.L = a.L;
    p.nkv = a.nkv;
    p.num_kb = (a.hidden + BK - 1) / BK;
    p.all_kv_out = a.all_kv_out;
    p.knorm_w = a.knorm_w;
    p.positions = a.positions;
    p.slot_mapping = a.slot_mapping;
    p.cos_sin = a.cos_sin;
    p.cache0 = a.cache0;
    p.cache_offsets = a.cache_offsets;
    p.k_scales = a.k_scales;
    p.v_scales = a.v_scales;
    p.error_flags = a.error_flags;
    p.max_pos = a.max_pos;
    p.capacity = a.capacity;
    p.bsl = a.block_size_log2;
    p.eps = a.eps;
    if (a.all_kv_out)
        return launch_gemm<kModeProject, 16, false>(tx, tw, p, stream);
    if (a.L > kMaxLayersProj)
        return cudaErrorInvalidValue;
    switch (a.rotary_dim) {
    case 16:
        return a.fp8 ? launch_gemm<kModeWrite, 16, true>(tx, tw, p, stream)
                     : launch_gemm<kModeWrite, 16, false>(tx, tw, p, stream);
    case 32:
        return a.fp8 ? launch_gemm<kModeWrite, 32, true>(tx, tw, p, stream)
                     : launch_gemm<kModeWrite, 32, false>(tx, tw, p, stream);
    case 64:
        return a.fp8 ? launch_gemm<kModeWrite, 64, true>(tx, tw, p, stream)
                     : launch_gemm<kModeWrite, 64, false>(tx, tw, p, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace dspark
