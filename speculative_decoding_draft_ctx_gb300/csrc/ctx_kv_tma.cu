// sm_103a pipelined kernel of the DSpark fused context-KV write (the fast
// path; ctx_kv_kernel.cu and ctx_kv_general.cu keep the fallbacks).
//
// Defining passage: vLLM DSpark context-KV writer page, module docstring (one
// launch for all draft layers: Gemma RMSNorm of K in fp32 materialised to
// bf16, partial NeoX RoPE at the token's position, K|V stored into each
// layer's [num_blocks, nkv, block_size, 2D] cache as bf16 or fp8 e4m3 of
// x / scale, slots < 0 not written).  The pages' head dim D is 128; this
// kernel also takes 64 and 256, any even rotary_dim up to D and any block
// size (the layouts their writer hands to the unfused path).
//
// Data movement.  all_kv[t, l0 : l0 + Lp] -- every K and V row of Lp layers of
// one token -- is one contiguous block of Lp * nkv * 4D bytes.  Each CTA runs
// a ring of shared-memory stages: a producer warp reads the slot and position
// of its next tokens, skips padding (a padded token's K|V is not copied, save
// among the CTA's first S units, which are copied before their slots are
// known and dropped if padded), and for each valid (token, layer piece)
// issues one bulk asynchronous copy
// (cp.async.bulk, completing on an mbarrier) of the block, plus one of the
// token's cos|sin row when r is 16, 32 or 64.  Eight consumer warps wait on
// the stage's barrier, compute from shared memory and store straight to the
// caches, then release the stage.  Bytes in flight per SM are bounded by
// shared memory, not by registers, so the HBM queue stays full with few
// warps.  A slot's (block, offset) comes from a shift and a mask for a
// power-of-two block size, else from a multiply-high by the host's
// Granlund-Montgomery magic number.  The kernel is launched with
// programmatic dependent launch (launch_pdl): it waits for the stream's
// previous kernel before its first global load or store, and before that
// wait only prefetches its first slabs, slots and positions into L2.
//
// Compute mapping.  A consumer warp handles 4 rows per instruction: 8 lanes
// per row, each lane holding the D/64 chunks [64k + 8q, 64k + 8q + 8) of K
// and of V (q = lane % 8), so every 16-byte shared load is conflict-free and
// every 16-byte (bf16) or 8-byte (fp8) global store of a warp covers 4 whole
// 128-byte (64-byte) segments.  Sum of squares: paired FMAs + 3 xor shuffles
// within the row's 8 lanes.  RoPE with r = 16 or 64: the partner of dim d is
// d +- r/2, r/16 lanes away within the row's 8 lanes (one xor shuffle).
// r = 32 maps K differently: lane q holds dims [32k + 4q, 32k + 4q + 4) for
// k = 0..3, so the 32 rotated dims are four on every lane of the row and
// each lane's first segment rotates against lane q ^ 4 (with 8-dim chunks
// only half the lanes would hold rotated dims, the other half computing a
// rotation they throw away).  In these three modes (head dim 128) a consumer
// warp copies its rows of the stage (at most two groups) and the token's
// cos|sin words into registers and releases the stage before computing, so
// the producer refills it while the warp computes.
// Any other even r: the normed row goes to a per-warp shared scratch (rows
// padded by 4 bytes, so the warp's partner reads hit 32 different banks), and
// after a __syncwarp each rotated dim reads its partner there; the token's
// cos|sin row is staged per warp from global memory (a row of 2r bytes need
// not be a multiple of the 16 a bulk copy moves).  fp8: the
// quotient x / scale is formed from the correctly rounded reciprocal of the
// scale with one FMA correction step (Markstein's method: q0 = x*(1/s),
// e = x - q0*s exactly, q = q0 + e*(1/s)), which yields the correctly rounded
// fp32 quotient, then a saturating RNE pack to e4m3 pairs.
//
// Per-layer slot mappings (drafts whose layers span several KV-cache
// groups): the producer prefetches each unit's per-layer slots one batch
// ahead into a double-buffered shared table, where each lane turns its
// unit's slots into row offsets (< 0: that layer is padding); when the unit
// is issued, one lane per layer copies them into the stage, and only the
// runs of layers that have a slot are copied from all_kv (a layer padded in
// its own mapping is neither read nor written; the consumers skip its
// rows).
//
// Every wait on an mbarrier is bounded (globaltimer); on expiry the CTA sets
// DSPARK_FLAG_TIMEOUT, stops, waits (bounded) for its own copies in flight
// and returns.
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "ctx_kv_device.cuh"
#include "ctx_kv_internal.h"
#include "ctx_kv_pipe.cuh"

namespace dspark {
namespace {

using namespace pipe;

constexpr int kConsumerWarps = 8;
constexpr int kThreads = 32 * (kConsumerWarps + 1);  // last warp is the producer
constexpr int kCsBytes = 128;                        // cos|sin row slot (r <= 64 bf16)
constexpr unsigned kFlagSlot = 0x1u;
constexpr unsigned kFlagPos = 0x2u;
constexpr unsigned kFlagTimeout = 0x4u;
constexpr unsigned kFlagCounter = 0x8u;
constexpr int kMaxTmaLayers = 32;

// A device word that nothing ever sets: the test hook's wait (test_hold_ns)
// runs out on it.
__device__ unsigned g_never_set = 0;

// What the producer tells the consumers about a stage.
struct StageHdr {
    long long dst;  // byte offset of the token's row for head 0 within a layer's cache
    long long pos;  // the token's position (rotary dims other than 16 / 32 / 64)
    int l0;         // first layer in the stage
    int rows;       // rows in the stage (layers * nkv); < 0: end of work
};

// Shared-memory layout (dynamic): barriers and headers, per-layer tables,
// then the stages (128-byte aligned).
struct Layout {
    uint32_t full, empty, hdr, abort, w1, off, scl, pls, lsp, pdst, csw, stages, stage_bytes, slab_bytes, total;
};

__host__ __device__ inline uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// pl: layers per unit when every layer has its own slot mapping (then the
// producer prefetches each unit's per-layer slots into a double-buffered
// [2][32][pl] table and hands the consumers per-layer row offsets [S][pl]),
// else 0.  D: the head dim.  xor_rot: r is 16, 32 or 64 (the cos|sin row is
// bulk-copied into each stage); else every consumer warp stages it in its own
// 2D-byte slot.
__host__ __device__ inline Layout make_layout(int L, int S, uint32_t slab_bytes, int pl, int D, bool xor_rot)
{
    Layout y;
    uint32_t o = 0;
    y.full = o;
    o += 8 * S;
    y.empty = o;
    o += 8 * S;
    y.hdr = align_up(o, 16);
    o = y.hdr + sizeof(StageHdr) * S;
    y.abort = o;
    o += 16;
    y.w1 = align_up(o, 16);
    o = y.w1 + 4 * D * L;  // D / 4 float4 slots per layer
    y.off = align_up(o, 8);  // per layer: its cache's base address
    o = y.off + 8 * L;
    y.scl = align_up(o, 16);  // per layer, 48 bytes: (k, k), (v, v), (-1/k, -1/k), (-1/v, -1/v), k bound, v bound
    o = y.scl + 48 * L;
    y.pls = align_up(o, 16);
    o = y.pls + 2 * 32 * 8 * pl;
    y.lsp = align_up(o, 16);  // per layer: its slot mapping's address (per-layer mappings)
    o = y.lsp + (pl ? 8 * L : 0);
    y.pdst = align_up(o, 16);
    o = y.pdst + 8 * S * pl;
    // per consumer warp (rotary dims other than 16/32/64): the token's cos|sin
    // row (2D bytes) and its 4 rows' normed K, each padded by 4 bytes so the
    // warp's partner reads spread over all 32 banks
    y.csw = align_up(o, 16);
    o = y.csw + (xor_rot ? 0 : kConsumerWarps * (10 * D + 64));
    y.stages = align_up(o, 128);
    y.slab_bytes = slab_bytes;
    y.stage_bytes = align_up(slab_bytes + (xor_rot ? kCsBytes : 0), 128);
    y.total = y.stages + y.stage_bytes * S;
    return y;
}

struct TmaParams {
    CtxKvParams p;
    int32_t layers_per_piece;  // Lp
    int32_t pieces;            // ceil(L / Lp)
    int32_t stages;            // S
    uint64_t h_magic;          // ceil(2^32 / nkv): row / nkv = (row * h_magic) >> 32 for row < 2^16
    // dynamic tail (work_counter != null): units [0, static_units) go to the
    // CTAs in grid-stride order, the rest in runs of claim_units to whichever
    // CTA claims the next run from work_counter[0]; work_counter[1] counts
    // finished CTAs, and the last one leaves both at zero for the next launch
    unsigned long long *work_counter;
    long long static_units;
    int32_t claim_units;       // consecutive units per claim (1..32)
    int32_t prefetch_units;    // units whose slabs go to L2 before the dependency wait (<= 32)
};

// w1 table: float4 slot of (layer l, half jj of an 8-dim chunk, chunk c of
// the D/8 chunks): lane q reads slots c = 8k + q (dims 64k + 8q..), so the 8
// lanes of a row read 128 contiguous bytes per load.
template <int D>
__device__ __forceinline__ int w1_slot(int l, int jj, int c)
{
    return l * (D / 4) + jj * (D / 8) + c;
}

// D: the head dim (64, 128, 256).  ROT: the rotary dim when it is 16, 32 or
// 64 (partners one xor shuffle away), or 0: any even p.rotary_dim up to D
// (partners through shared memory).  PL: every layer has its own slot
// mapping (p.layer_slots).  Template parameters, so each path carries none
// of the others' branches.
template <int D, int ROT, bool FP8, bool PL>
__global__ void __launch_bounds__(kThreads, 2) ctx_kv_tma_kernel(const TmaParams tp)
{
    constexpr int NC = D / 64;                  // 8-dim chunks of K (and of V) per lane
    constexpr uint32_t kRowIn = 4 * D;          // bytes of one K|V row pair in all_kv
    constexpr int kCacheRow = FP8 ? 2 * D : 4 * D;  // bytes of one cache row
    constexpr bool kXor = ROT != 0;
    // r = 32: K in the segmented mapping -- lane q holds dims 32k + 4q .. + 3
    // (k = 0..3), so the rotated dims 0..31 are four on every lane of a row
    // and each lane's first segment rotates with lane q ^ 4 (V keeps the
    // 16-byte chunks)
    constexpr bool kSeg = ROT == 32 && D == 128;
    extern __shared__ __align__(128) unsigned char smem[];
    const CtxKvParams &p = tp.p;
    const int L = p.num_layers, H = p.num_kv_heads, S = tp.stages, NP = tp.pieces, Lp = tp.layers_per_piece;
    const Layout lay = make_layout(L, S, (uint32_t)Lp * H * kRowIn, PL ? Lp : 0, D, kXor);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + lay.full);
    uint64_t *empty = reinterpret_cast<uint64_t *>(smem + lay.empty);
    StageHdr *hdr = reinterpret_cast<StageHdr *>(smem + lay.hdr);
    volatile int *abort = reinterpret_cast<volatile int *>(smem + lay.abort);
    float4 *w1 = reinterpret_cast<float4 *>(smem + lay.w1);
    unsigned char **layer_base = reinterpret_cast<unsigned char **>(smem + lay.off);
    uint32_t *scl = reinterpret_cast<uint32_t *>(smem + lay.scl);
    unsigned char *stages = smem + lay.stages;
    long long *pls = reinterpret_cast<long long *>(smem + lay.pls);    // [2][32][Lp] prefetched per-layer slots
    long long *pdst = reinterpret_cast<long long *>(smem + lay.pdst);  // [S][Lp] per-layer row offsets (< 0: none)
    const int64_t **lsp = reinterpret_cast<const int64_t **>(smem + lay.lsp);  // [L] per-layer slot mappings

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        for (int s = 0; s < S; s++) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, kConsumerWarps);
        }
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    if (warp == kConsumerWarps) {
        // While the previous kernel drains: the K|V slabs of this CTA's first
        // prefetch_units units, and the slots and positions of its first 32,
        // into L2 (hints only; every copy below still follows
        // griddepcontrol.wait).
        const long long u_end = tp.work_counter ? tp.static_units : p.num_ctx * (long long)NP;
        const long long u = blockIdx.x + (long long)lane * gridDim.x;
        if (u < u_end) {
            const long long t = NP == 1 ? u : u / NP;
            if (lane < tp.prefetch_units) {
                const int l0 = (NP == 1 ? 0 : (int)(u - t * NP)) * Lp;
                prefetch_l2_bulk(p.all_kv + (t * L + l0) * 2LL * H * D, (uint32_t)min(Lp, L - l0) * H * kRowIn);
            }
            if (!PL)
                prefetch_l2(p.slot_mapping + t);
            prefetch_l2(p.positions + t);
        }
    }
    pdl_enter();  // launched with launch_pdl: above, only barriers and L2 prefetch hints

    const long long units = p.num_ctx * (long long)NP;
    const long long G = gridDim.x;
    unsigned flags = 0;

    if (warp == kConsumerWarps) {
        // ---------------------------------------------------------- producer
        // Starts at once: the consumers build their tables meanwhile.  The
        // CTA's units come in batches: its static units in grid-stride order
        // (32 per batch), then, with a work counter, runs of consecutive units
        // claimed from the shared tail until the counter runs past the end.  Slots
        // and positions of the next batch are fetched while the current one
        // is issued.
        struct Batch {
            long long first, stride;  // units first + j * stride, j < count
            int count;
            bool dyn;
        };
        const long long u_first = blockIdx.x, step = G;
        const long long u_static = tp.work_counter ? tp.static_units : units;
        auto static_batch = [&](long long base) {
            Batch b{base, step, 0, false};
            if (base < u_static)
                b.count = (int)min(32LL, (u_static - base + step - 1) / step);
            return b;
        };
        // runs of the shared tail; a launch makes at most runs + G claims
        // (every CTA's last one finds the tail empty), so a larger claim
        // number means the counter was not zero at launch: no unit is taken
        // from it and the call is flagged
        const unsigned long long runs =
            tp.work_counter ? (unsigned long long)((units - u_static + tp.claim_units - 1) / tp.claim_units) : 0;
        auto claim = [&]() {  // the whole warp; lane 0 takes the next run of units
            unsigned long long c = 0;
            if (lane == 0)
                c = atomicAdd(tp.work_counter, 1ull);
            c = __shfl_sync(0xffffffffu, c, 0);
            Batch b{0, 1, 0, true};
            if (c < runs) {
                b.first = u_static + (long long)c * tp.claim_units;
                b.count = (int)min((long long)tp.claim_units, units - b.first);
            } else if (c >= runs + (unsigned long long)G) {
                flags |= kFlagCounter;
            }
            return b;
        };
        auto next_batch = [&](const Batch &b) {
            if (!b.dyn) {
                const Batch n = static_batch(b.first + 32 * step);
                if (n.count > 0 || !tp.work_counter)
                    return n;
            }
            return claim();
        };
        // byte offset of a slot's (block, offset) row for head 0 within a
        // layer's cache: a power-of-two block size shifts, any other divides
        // by a multiply-high with the host's magic number
        auto row_off = [&](long long slot) {
            long long blk, off;
            if (p.block_size_log2 >= 0) {
                blk = slot >> p.block_size_log2;
                off = slot & ((1LL << p.block_size_log2) - 1);
            } else {
                blk = (long long)(__umul64hi((unsigned long long)slot, p.bs_magic) >> p.bs_magic_shift);
                off = slot - blk * p.block_size;
            }
            return (blk * H * p.block_size + off) * kCacheRow;
        };
        // Slot and position of unit base + lane * step.  With per-layer
        // mappings the unit's layers' slots go to the prefetch table (buffer
        // buf) and `slot` only says whether any of them is valid.
        auto fetch = [&](const Batch &b, long long &slot, long long &pos, int buf) {
            const long long u = b.first + (long long)lane * b.stride;
            slot = -1;
            pos = 0;
            if (lane < b.count) {
                const long long t = NP == 1 ? u : u / NP;
                pos = __ldg(p.positions + t);
                if (PL) {
                    // the unit's per-layer slots land in the prefetch table by
                    // asynchronous copies (no register waits on them here);
                    // vet() waits for them a batch later
                    const int l0 = (NP == 1 ? 0 : (int)(u - t * NP)) * Lp;
                    const int n = min(Lp, L - l0);
                    long long *e = pls + (buf * 32 + lane) * Lp;
                    for (int j = 0; j < n; j++)
                        asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(e + j)),
                                     "l"(lsp[l0 + j] + t)
                                     : "memory");
                    slot = 0;  // vet() decides
                } else {
                    slot = __ldg(p.slot_mapping + t);
                }
            }
        };
        auto vet = [&](const Batch &b, long long &slot, long long pos, int buf) {
            if (slot < 0)
                return;
            const long long u = b.first + (long long)lane * b.stride;
            const bool first_piece = NP == 1 || u % NP == 0;  // a token is reported once
            if (pos < 0 || pos >= p.max_pos) {
                if (first_piece)
                    flags |= kFlagPos;
                slot = -1;
            } else if (PL) {
                const long long t = NP == 1 ? u : u / NP;
                const int n = min(Lp, L - (NP == 1 ? 0 : (int)(u - t * NP)) * Lp);
                long long *e = pls + (buf * 32 + lane) * Lp;  // this lane's own copies (waited for below)
                bool any = false;
                // each layer's slot becomes its row offset here, one unit per
                // lane, so the issuing lane only copies them
                for (int j = 0; j < n; j++) {
                    if (e[j] >= p.capacity) {
                        flags |= kFlagSlot;
                        e[j] = -1;
                    }
                    any |= e[j] >= 0;
                    e[j] = e[j] >= 0 ? row_off(e[j]) : -1;
                }
                if (!any)
                    slot = -1;
            } else if (slot >= p.capacity) {
                if (first_piece)
                    flags |= kFlagSlot;
                slot = -1;
            }
        };
        const uint64_t stream_once = evict_first_policy();  // all_kv: read exactly once
        const uint64_t keep = evict_last_policy();          // cos|sin rows: shared by many tokens
        uint32_t k = 0;  // stages issued so far (the sentinel excluded)
        int ps = 0;          // ring slot of round k
        uint32_t pph = 0;    // phase parity of round k in that slot
        bool ok = true;
        long long cur_slot, cur_pos, nxt_slot = -1, nxt_pos = 0;
        // The first S units of the CTA get their K|V block copied before
        // their slots are known (each takes a stage whatever its slot), which
        // hides the slot fetch behind the first copies; a padded one among
        // them has been read all the same and is dropped (its stage released
        // with no rows).
        auto unit_span = [&](long long u, long long &t, int &l0, uint32_t &slab) {
            t = NP == 1 ? u : u / NP;
            l0 = (NP == 1 ? 0 : (int)(u - t * NP)) * Lp;
            slab = (uint32_t)min(Lp, L - l0) * H * kRowIn;
        };
        int nspec = 0;
        for (long long u = u_first; u < u_static && nspec < S; u += step)
            nspec++;
        if (p.test_hold_ns) {
            // test hook: a bounded wait on a word nothing sets, which runs out;
            // the CTA then stops before issuing anything
            if (lane == 0) {
                const unsigned long long t0 = globaltimer();
                while (*reinterpret_cast<volatile unsigned *>(&g_never_set) == 0 &&
                       globaltimer() - t0 < p.test_hold_ns) {
                }
                *abort = 1;
            }
            ok = false;
            nspec = 0;
        }
        if (lane == 0) {
            for (int i = 0; i < nspec; i++) {
                long long t;
                int l0;
                uint32_t slab;
                unit_span(u_first + i * step, t, l0, slab);
                mbar_expect_tx(full + i, slab);
                bulk_g2s(stages + (size_t)i * lay.stage_bytes, p.all_kv + (t * L + l0) * 2LL * H * D, slab,
                         full + i, stream_once);
            }
        }
        long long ordinal = 0;  // index of the batch's first unit in this CTA's sequence
        int buf = 0;            // prefetch-table buffer of the current batch
        if (PL) {  // the layers' slot mapping addresses, once
            for (int j = lane; j < L; j += 32)
                lsp[j] = reinterpret_cast<const int64_t *>(
                    __ldg(reinterpret_cast<const unsigned long long *>(p.layer_slots) + j));
            __syncwarp();
        }
        Batch cur = static_batch(u_first);
        if (cur.count == 0 && tp.work_counter && ok)
            cur = claim();
        if (ok && cur.count > 0) {
            fetch(cur, cur_slot, cur_pos, buf);
            if (PL)
                asm volatile("cp.async.commit_group;" ::: "memory");
        }
        for (; cur.count > 0 && ok; buf ^= 1) {
            const Batch nxt = next_batch(cur);
            if (nxt.count > 0) {
                fetch(nxt, nxt_slot, nxt_pos, buf ^ 1);
                if (PL) {
                    asm volatile("cp.async.commit_group;" ::: "memory");
                    asm volatile("cp.async.wait_group 1;" ::: "memory");  // this batch's, not the next one's
                }
            } else if (PL) {
                asm volatile("cp.async.wait_group 0;" ::: "memory");
            }
            vet(cur, cur_slot, cur_pos, buf);
            __syncwarp();  // lane 0 reads the other lanes' prefetched slots below
            for (int i = 0; i < cur.count; i++) {
                const long long u = cur.first + (long long)i * cur.stride;
                const long long slot = __shfl_sync(0xffffffffu, cur_slot, i);
                const long long pos = __shfl_sync(0xffffffffu, cur_pos, i);
                const bool spec = ordinal + i < nspec;
                if (slot < 0 && !spec)
                    continue;  // padding (or out of range): K|V not copied, nothing written
                bool ready = true;
                uint32_t vmask = 0;  // per-layer mappings: the unit's layers that have a slot
                if constexpr (PL) {
                    // the stage is free before its per-layer row offsets are
                    // rewritten, one lane per layer; the ballot gives the mask of
                    // the unit's layers that have a slot
                    if (lane == 0)
                        ready = spec || mbar_wait(empty + ps, pph ^ 1u, abort);
                    ready = __shfl_sync(0xffffffffu, ready, 0);
                    long long t_;
                    int l0_;
                    uint32_t slab_;
                    unit_span(u, t_, l0_, slab_);
                    const int n = (int)(slab_ / kRowIn) / H;
                    const long long off = lane < n ? pls[(buf * 32 + i) * Lp + lane] : -1;
                    if (ready && slot >= 0 && lane < n)
                        pdst[ps * Lp + lane] = off;
                    vmask = __ballot_sync(0xffffffffu, off >= 0);
                    __syncwarp();
                }
                if (lane == 0) {
                    const int s = ps;
                    ok = PL ? ready : spec || mbar_wait(empty + s, pph ^ 1u, abort);
                    if (ok) {
                        long long t;
                        int l0;
                        uint32_t slab;
                        unit_span(u, t, l0, slab);
                        unsigned char *dst = stages + (size_t)s * lay.stage_bytes;
                        if (slot < 0) {
                            hdr[s].rows = 0;  // a speculatively copied padded unit: dropped
                            mbar_arrive(full + s);
                        } else {
                            if (!PL)
                                hdr[s].dst = row_off(slot);
                            hdr[s].l0 = l0;
                            hdr[s].pos = pos;
                            hdr[s].rows = (int)(slab / kRowIn);
                            // the cos|sin row rides along in the xor modes (2r = 32, 64 or
                            // 128 bytes); otherwise the consumers fetch it themselves
                            const uint32_t cs_bytes = kXor ? 2u * ROT : 0u;
                            if (spec) {
                                if (kXor)
                                    mbar_arrive_expect_tx(full + s, cs_bytes);
                                else
                                    mbar_arrive(full + s);
                            } else if (PL) {
                                // only the runs of layers that have a slot (bits of vmask): a
                                // layer padded in its own mapping is neither read nor written
                                const uint32_t layer_bytes = (uint32_t)H * kRowIn;
                                mbar_arrive_expect_tx(full + s, (uint32_t)__popc(vmask) * layer_bytes + cs_bytes);
                                for (uint32_t m = vmask; m;) {
                                    const int j = __ffs(m) - 1;
                                    // the run of set bits from j (64-bit: a run may hold all 32 layers)
                                    const int len = __ffsll((long long)~((unsigned long long)m >> j)) - 1;
                                    bulk_g2s(dst + (size_t)j * layer_bytes, p.all_kv + (t * L + l0 + j) * 2LL * H * D,
                                             (uint32_t)len * layer_bytes, full + s, stream_once);
                                    m &= ~(uint32_t)(((1ull << len) - 1ull) << j);
                                }
                            } else {
                                mbar_arrive_expect_tx(full + s, slab + cs_bytes);
                                bulk_g2s(dst, p.all_kv + (t * L + l0) * 2LL * H * D, slab, full + s, stream_once);
                            }
                            if (kXor)
                                bulk_g2s(dst + lay.slab_bytes, p.cos_sin + pos * ROT, 2u * ROT, full + s, keep);
                        }
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok)
                    break;
                k++;
                if (++ps == S) {
                    ps = 0;
                    pph ^= 1u;
                }
            }
            ordinal += cur.count;
            cur_slot = nxt_slot;
            cur_pos = nxt_pos;
            cur = nxt;
        }
        if (PL)
            asm volatile("cp.async.wait_group 0;" ::: "memory");  // no prefetch copy outlives the CTA
        uint32_t rounds = k;  // barrier rounds used, the sentinel included
        if (lane == 0) {
            if (ok) {
                const int s = ps;
                if (mbar_wait(empty + s, pph ^ 1u, abort)) {
                    hdr[s].rows = -1;
                    mbar_arrive(full + s);
                    rounds = k + 1;
                }
            }
            if (*abort)
                flags |= kFlagTimeout;
        }
        __syncwarp();
        __syncthreads();
        // drain: every copy this CTA issued has landed before the CTA exits.
        // Only the last S rounds can be pending, and a round whose stage was
        // reused since has completed (its barrier moved on).
        if (lane == 0) {
            const uint32_t first = rounds > (uint32_t)S ? rounds - S : 0;
            for (uint32_t j = first; j < k; j++) {
                const int s = (int)(j % S);
                const unsigned long long t0 = globaltimer();
                while (!mbar_try_wait(full + s, (j / S) & 1u) && globaltimer() - t0 < kTimeoutNs) {
                }
            }
        }
    } else {
        // ---------------------------------------------------------- consumers
        // per-layer tables: (1 + w) in fp32, cache offsets, scale constants
        for (int i = tid; i < L * D; i += 32 * kConsumerWarps) {
            const int l = i / D, d = i % D;
            const int c = d / 8, j = d % 8;  // chunk c holds dims 8c .. 8c+7
            // segmented mode (r = 32): dims in natural order, float4 slot
            // l * D/4 + 8k + q holding the lane's dims 32k + 4q .. + 3
            const int at = kSeg ? i : w1_slot<D>(l, j / 4, c) * 4 + (j % 4);
            reinterpret_cast<float *>(w1)[at] = 1.0f + __uint_as_float((uint32_t)__ldg(p.knorm_w + i) << 16);
        }
        for (int l = tid; l < L; l += 32 * kConsumerWarps) {
            layer_base[l] = p.cache0 + __ldg(p.cache_offsets + l) * (FP8 ? 1 : 2);
            float ks = 1.0f, vs = 1.0f;
            if (FP8) {
                ks = __ldg(reinterpret_cast<const float *>(
                    __ldg(reinterpret_cast<const unsigned long long *>(p.k_scales) + l)));
                vs = __ldg(reinterpret_cast<const float *>(
                    __ldg(reinterpret_cast<const unsigned long long *>(p.v_scales) + l)));
            }
            const float kn = -__frcp_rn(ks), vn = -__frcp_rn(vs);
            uint32_t *e = scl + 12 * l;
            e[0] = e[1] = __float_as_uint(ks);
            e[2] = e[3] = __float_as_uint(vs);
            e[4] = e[5] = __float_as_uint(kn);
            e[6] = e[7] = __float_as_uint(vn);
            e[8] = fp8_bound_pair(ks);
            e[9] = fp8_bound_pair(vs);
        }
        asm volatile("bar.sync 1, %0;" ::"n"(32 * kConsumerWarps) : "memory");

        const int q = lane & 7;      // 8-dim chunk of each 64-dim segment of the row
        const int rr = lane >> 3;    // row of the 4-row group
        constexpr int kPartner = kXor ? ROT / 16 : 1;
        constexpr int kRotLanes = ROT / 8;
        const bool rot_lane = kXor && q < kRotLanes;
        const int rdim = kXor ? ROT : p.rotary_dim, half = rdim >> 1;
        uint16_t *csw = reinterpret_cast<uint16_t *>(smem + lay.csw + warp * (10 * D + 64));  // cos|sin row
        // this lane's row of the warp's normed-K scratch: rows D + 2 elements
        // apart, so lane (q, rr)'s 2-byte element 8q + e falls in bank
        // 4q + rr + e/2 and the warp's 32 lanes hit 32 different banks
        uint16_t *yrow = csw + D + rr * (D + 2);
        // bytes between the rows of consecutive heads in a cache
        const long long head_bytes = (long long)kCacheRow * p.block_size;
        int gmod = 0;  // row groups seen so far, over all stages, modulo the consumer warps
        int s = 0;          // ring slot of the current round
        uint32_t ph = 0;    // its phase parity
        for (;; s = (s + 1 == S) ? 0 : s + 1, ph ^= (s == 0)) {
            if (!mbar_wait(full + s, ph, abort))
                break;
            const StageHdr h_s = hdr[s];
            const int R = h_s.rows;
            if (R < 0)
                break;
            const int ngroups = (R + 3) >> 2;
            const int first = (warp - gmod) & (kConsumerWarps - 1);  // this warp's first group here
            gmod = (gmod + ngroups) & (kConsumerWarps - 1);
            if constexpr (kXor) {
                // Early release: the warp copies its rows (a 32 KB stage holds at
                // most 8192 / D rows, so at most 256 / D groups per warp) and the
                // token's cos|sin words into registers, releases the stage so
                // that the producer can refill it at once, then computes.
                constexpr int kMaxG = 256 / D;
                uint4 kd[kMaxG][NC], vd[kMaxG][NC];
                long long gdst[kMaxG];
                int gl[kMaxG], gh[kMaxG];
                bool gact[kMaxG];  // the lane's row exists in the group
                uint32_t cw[4] = {0, 0, 0, 0}, sw[4] = {0, 0, 0, 0};
                const unsigned char *stage = stages + (size_t)s * lay.stage_bytes;
                if (first < ngroups) {
                    if constexpr (kSeg) {
                        // the lane's 4 rotated dims 4q .. 4q+3: cos and sin of dims 4 (q & 3) .. + 3
                        const unsigned char *cs = stage + lay.slab_bytes + 8 * (q & 3);
                        const uint2 c2 = *reinterpret_cast<const uint2 *>(cs);
                        const uint2 s2 = *reinterpret_cast<const uint2 *>(cs + ROT);
                        const uint32_t flip = (q & 4) ? 0u : 0x80008000u;  // lower half subtracts
                        cw[0] = c2.x, cw[1] = c2.y;
                        sw[0] = s2.x ^ flip, sw[1] = s2.y ^ flip;
                    } else if (rot_lane) {
                        const unsigned char *cs = stage + lay.slab_bytes + 16 * (q & (kPartner - 1));
                        const uint4 c4 = lds128(cs), s4 = lds128(cs + ROT);  // sin half: r/2 elements later
                        const uint32_t flip = (q & kPartner) ? 0u : 0x80008000u;  // lower half subtracts
                        cw[0] = c4.x, cw[1] = c4.y, cw[2] = c4.z, cw[3] = c4.w;
                        sw[0] = s4.x ^ flip, sw[1] = s4.y ^ flip, sw[2] = s4.z ^ flip, sw[3] = s4.w ^ flip;
                    }
#pragma unroll
                    for (int gi = 0; gi < kMaxG; gi++) {
                        const int g = first + gi * kConsumerWarps;
                        gact[gi] = false;
                        gdst[gi] = -1;
                        gl[gi] = gh[gi] = 0;
                        if (g < ngroups) {
                            const int row = g * 4 + rr;
                            gact[gi] = row < R;
                            const int rc = gact[gi] ? row : R - 1;
                            const int lr = (int)(((uint64_t)(uint32_t)rc * tp.h_magic) >> 32);
                            gh[gi] = rc - lr * H;
                            gl[gi] = h_s.l0 + lr;
                            gdst[gi] = PL ? pdst[s * Lp + lr] : h_s.dst;
                            const unsigned char *krow = stage + ((size_t)(2 * lr) * H + gh[gi]) * (2 * D);
                            const unsigned char *vrow = krow + (size_t)H * (2 * D);
#pragma unroll
                            for (int k = 0; k < NC; k++) {
                                if constexpr (kSeg) {  // segments 2k, 2k + 1
                                    const uint2 a = *reinterpret_cast<const uint2 *>(krow + 128 * k + 8 * q);
                                    const uint2 b = *reinterpret_cast<const uint2 *>(krow + 128 * k + 64 + 8 * q);
                                    kd[gi][k] = make_uint4(a.x, a.y, b.x, b.y);
                                } else {
                                    kd[gi][k] = lds128(krow + 128 * k + 16 * q);
                                }
                                vd[gi][k] = lds128(vrow + 128 * k + 16 * q);
                            }
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty + s);
#pragma unroll
                for (int gi = 0; gi < kMaxG; gi++) {
                    if (first + gi * kConsumerWarps >= ngroups)
                        break;  // warp-uniform
                    const int l = gl[gi], h = gh[gi];
                    uint64_t x2[4 * NC];
#pragma unroll
                    for (int k = 0; k < NC; k++) {
                        const uint4 a = kd[gi][k];
                        x2[4 * k] = bf2_to_f2(a.x), x2[4 * k + 1] = bf2_to_f2(a.y);
                        x2[4 * k + 2] = bf2_to_f2(a.z), x2[4 * k + 3] = bf2_to_f2(a.w);
                    }
                    uint64_t a0 = mul2(x2[0], x2[0]), a1 = mul2(x2[1], x2[1]);
#pragma unroll
                    for (int j = 2; j < 4 * NC; j += 2) {
                        a0 = fma2(x2[j], x2[j], a0);
                        a1 = fma2(x2[j + 1], x2[j + 1], a1);
                    }
                    float slo, shi;
                    unpr(add2(a0, a1), slo, shi);
                    float ss = slo + shi;
                    ss += __shfl_xor_sync(0xffffffffu, ss, 4);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                    ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                    float inv;  // ss/D + eps >= eps > 0 (hardware reciprocal square root)
                    asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(fmaf(ss, 1.0f / D, p.eps)));
                    const uint64_t inv2 = pr(inv, inv);
                    uint32_t ko[4 * NC];
#pragma unroll
                    for (int k = 0; k < NC; k++) {
                        float4 wa, wb;
                        if constexpr (kSeg) {
                            wa = w1[l * (D / 4) + 16 * k + q];      // dims 64k + 4q .. + 3 (segment 2k)
                            wb = w1[l * (D / 4) + 16 * k + 8 + q];  // segment 2k + 1
                        } else {
                            wa = w1[w1_slot<D>(l, 0, 8 * k + q)], wb = w1[w1_slot<D>(l, 1, 8 * k + q)];
                        }
                        ko[4 * k] = f2_to_bf2(mul2(mul2(x2[4 * k], inv2), pr(wa.x, wa.y)));
                        ko[4 * k + 1] = f2_to_bf2(mul2(mul2(x2[4 * k + 1], inv2), pr(wa.z, wa.w)));
                        ko[4 * k + 2] = f2_to_bf2(mul2(mul2(x2[4 * k + 2], inv2), pr(wb.x, wb.y)));
                        ko[4 * k + 3] = f2_to_bf2(mul2(mul2(x2[4 * k + 3], inv2), pr(wb.z, wb.w)));
                    }
                    if constexpr (kSeg) {
                        // segment 0 (dims 4q .. 4q+3) rotates on every lane; the partner is 4 lanes away
#pragma unroll
                        for (int j = 0; j < 2; j++) {
                            const uint32_t yp = __shfl_xor_sync(0xffffffffu, ko[j], 4);
                            ko[j] = f2_to_bf2(rope_bf2(ko[j], cw[j], yp, sw[j]));
                        }
                    } else {
#pragma unroll
                        for (int j = 0; j < 4; j++) {
                            const uint32_t yp = __shfl_xor_sync(0xffffffffu, ko[j], kPartner);
                            const uint32_t rv = f2_to_bf2(rope_bf2(ko[j], cw[j], yp, sw[j]));
                            ko[j] = rot_lane ? rv : ko[j];  // both computed: a select, not a branch
                        }
                    }
                    if (!gact[gi] || gdst[gi] < 0)
                        continue;  // past the stage's rows, or a layer padded in its own mapping
                    unsigned char *dg = layer_base[l] + gdst[gi] + h * head_bytes;
                    if constexpr (kSeg) {
                        // K: 4 dims per segment, 4 segments; V: 16-byte chunks
                        if (!FP8) {
#pragma unroll
                            for (int k = 0; k < 4; k++)
                                st_stream_v2(dg + 64 * k + 8 * q, make_uint2(ko[2 * k], ko[2 * k + 1]));
#pragma unroll
                            for (int k = 0; k < NC; k++)
                                st_stream_v4(dg + 2 * D + 128 * k + 16 * q, vd[gi][k]);
                        } else {
                            const ulonglong2 sv = reinterpret_cast<const ulonglong2 *>(scl + 12 * l)[0];
                            const ulonglong2 nv = reinterpret_cast<const ulonglong2 *>(scl + 12 * l)[1];
                            const uint2 b2 = *reinterpret_cast<const uint2 *>(scl + 12 * l + 8);
#pragma unroll
                            for (int k = 0; k < NC; k++) {
                                const uint2 c = quantise8(
                                    make_uint4(ko[4 * k], ko[4 * k + 1], ko[4 * k + 2], ko[4 * k + 3]), b2.x, sv.x, nv.x);
                                st_stream_v1(dg + 64 * k + 4 * q, c.x);
                                st_stream_v1(dg + 64 * k + 32 + 4 * q, c.y);
                            }
#pragma unroll
                            for (int k = 0; k < NC; k++)
                                st_stream_v2(dg + D + 64 * k + 8 * q, quantise8(vd[gi][k], b2.y, sv.y, nv.y));
                        }
                        continue;
                    }
                    if (!FP8) {
#pragma unroll
                        for (int k = 0; k < NC; k++)
                            st_stream_v4(dg + 128 * k + 16 * q, make_uint4(ko[4 * k], ko[4 * k + 1], ko[4 * k + 2],
                                                                          ko[4 * k + 3]));
#pragma unroll
                        for (int k = 0; k < NC; k++)
                            st_stream_v4(dg + 2 * D + 128 * k + 16 * q, vd[gi][k]);
                    } else {
                        const ulonglong2 sv = reinterpret_cast<const ulonglong2 *>(scl + 12 * l)[0];
                        const ulonglong2 nv = reinterpret_cast<const ulonglong2 *>(scl + 12 * l)[1];
                        const uint2 b2 = *reinterpret_cast<const uint2 *>(scl + 12 * l + 8);
#pragma unroll
                        for (int k = 0; k < NC; k++)
                            st_stream_v2(dg + 64 * k + 8 * q,
                                         quantise8(make_uint4(ko[4 * k], ko[4 * k + 1], ko[4 * k + 2], ko[4 * k + 3]),
                                                   b2.x, sv.x, nv.x));
#pragma unroll
                        for (int k = 0; k < NC; k++)
                            st_stream_v2(dg + D + 64 * k + 8 * q, quantise8(vd[gi][k], b2.y, sv.y, nv.y));
                    }
                }
            } else {
                if (first < ngroups) {
                    // any other even rotary dim: partners through the warp's shared row
                    const unsigned char *stage = stages + (size_t)s * lay.stage_bytes;
                    {
                        // the token's cos|sin row into this warp's slot, as 4-byte words (r is even)
                        const uint32_t *src = reinterpret_cast<const uint32_t *>(p.cos_sin + h_s.pos * rdim);
                        uint32_t *dst = reinterpret_cast<uint32_t *>(csw);
                        for (int k = lane; k < half; k += 32)
                            dst[k] = __ldg(src + k);
                        __syncwarp();
                    }
                    for (int g = first; g < ngroups; g += kConsumerWarps) {
                        const int row = g * 4 + rr;
                        const bool active = row < R;
                        const int rc = active ? row : R - 1;
                        const int lr = (int)(((uint64_t)(uint32_t)rc * tp.h_magic) >> 32);
                        const int h = rc - lr * H;
                        const int l = h_s.l0 + lr;
                        const unsigned char *krow = stage + ((size_t)(2 * lr) * H + h) * (2 * D);
                        const unsigned char *vrow = krow + (size_t)H * (2 * D);
                        uint64_t x2[4 * NC];
#pragma unroll
                        for (int k = 0; k < NC; k++) {
                            const uint4 a = lds128(krow + 128 * k + 16 * q);
                            x2[4 * k] = bf2_to_f2(a.x), x2[4 * k + 1] = bf2_to_f2(a.y);
                            x2[4 * k + 2] = bf2_to_f2(a.z), x2[4 * k + 3] = bf2_to_f2(a.w);
                        }
                        // sum of squares: two accumulator chains of packed FMAs
                        uint64_t a0 = mul2(x2[0], x2[0]), a1 = mul2(x2[1], x2[1]);
#pragma unroll
                        for (int j = 2; j < 4 * NC; j += 2) {
                            a0 = fma2(x2[j], x2[j], a0);
                            a1 = fma2(x2[j + 1], x2[j + 1], a1);
                        }
                        float slo, shi;
                        unpr(add2(a0, a1), slo, shi);
                        float ss = slo + shi;
                        ss += __shfl_xor_sync(0xffffffffu, ss, 4);
                        ss += __shfl_xor_sync(0xffffffffu, ss, 2);
                        ss += __shfl_xor_sync(0xffffffffu, ss, 1);
                        float inv;  // ss/D + eps >= eps > 0 (hardware reciprocal square root)
                        asm("rsqrt.approx.ftz.f32 %0, %1;" : "=f"(inv) : "f"(fmaf(ss, 1.0f / D, p.eps)));
                        const uint64_t inv2 = pr(inv, inv);
                        // y = bf16((k * inv) * (1 + w))
                        uint32_t y[4 * NC];
#pragma unroll
                        for (int k = 0; k < NC; k++) {
                            const float4 wa = w1[w1_slot<D>(l, 0, 8 * k + q)], wb = w1[w1_slot<D>(l, 1, 8 * k + q)];
                            y[4 * k] = f2_to_bf2(mul2(mul2(x2[4 * k], inv2), pr(wa.x, wa.y)));
                            y[4 * k + 1] = f2_to_bf2(mul2(mul2(x2[4 * k + 1], inv2), pr(wa.z, wa.w)));
                            y[4 * k + 2] = f2_to_bf2(mul2(mul2(x2[4 * k + 2], inv2), pr(wb.x, wb.y)));
                            y[4 * k + 3] = f2_to_bf2(mul2(mul2(x2[4 * k + 3], inv2), pr(wb.z, wb.w)));
                        }
                        uint32_t ko[4 * NC];
                        {
                            // the normed row into the warp's scratch (the row's 8 lanes own it; the
                            // previous group's partner reads are done first), then each rotated dim
                            // d reads its partner d +- r/2 there
                            __syncwarp();
#pragma unroll
                            for (int k = 0; k < NC; k++)
#pragma unroll
                                for (int w = 0; w < 4; w++)  // 4-byte stores: the rows are only 4-byte aligned
                                    reinterpret_cast<uint32_t *>(yrow + 64 * k + 8 * q)[w] = y[4 * k + w];
                            __syncwarp();
#pragma unroll
                            for (int k = 0; k < NC; k++) {
                                const int d0 = 64 * k + 8 * q;
#pragma unroll
                                for (int j = 0; j < 4; j++) {
                                    ko[4 * k + j] = y[4 * k + j];
                                    if (d0 + 2 * j < rdim) {
                                        float o[2];
#pragma unroll
                                        for (int b = 0; b < 2; b++) {
                                            const int d = d0 + 2 * j + b;  // d < r: r is even
                                            const bool lower = d < half;
                                            const int fi = lower ? d : d - half;
                                            const float yd = __uint_as_float(b ? (y[4 * k + j] & 0xffff0000u)
                                                                               : (y[4 * k + j] << 16));
                                            const float c = __uint_as_float((uint32_t)csw[fi] << 16);
                                            const float sn = __uint_as_float((uint32_t)csw[half + fi] << 16);
                                            const float yp = __uint_as_float((uint32_t)yrow[lower ? d + half : d - half] << 16);
                                            o[b] = fmaf(yd, c, lower ? -(yp * sn) : yp * sn);
                                        }
                                        ko[4 * k + j] = pack_bf16x2(o[0], o[1]);
                                    }
                                }
                            }
                        }
                        const long long roff = PL ? pdst[s * Lp + lr] : h_s.dst;
                        if (!active || roff < 0)
                            continue;  // past the stage's rows, or a layer padded in its own mapping
                        unsigned char *dg = layer_base[l] + roff + h * head_bytes;
                        if (!FP8) {
#pragma unroll
                            for (int k = 0; k < NC; k++)
                                st_stream_v4(dg + 128 * k + 16 * q, make_uint4(ko[4 * k], ko[4 * k + 1], ko[4 * k + 2],
                                                                              ko[4 * k + 3]));
#pragma unroll
                            for (int k = 0; k < NC; k++)
                                st_stream_v4(dg + 2 * D + 128 * k + 16 * q, lds128(vrow + 128 * k + 16 * q));
                        } else {
                            const ulonglong2 sv = reinterpret_cast<const ulonglong2 *>(scl + 12 * l)[0];
                            const ulonglong2 nv = reinterpret_cast<const ulonglong2 *>(scl + 12 * l)[1];
                            const uint2 b2 = *reinterpret_cast<const uint2 *>(scl + 12 * l + 8);
                            const uint64_t ks2 = sv.x, vs2 = sv.y, kn2 = nv.x, vn2 = nv.y;
#pragma unroll
                            for (int k = 0; k < NC; k++)
                                st_stream_v2(dg + 64 * k + 8 * q,
                                             quantise8(make_uint4(ko[4 * k], ko[4 * k + 1], ko[4 * k + 2], ko[4 * k + 3]),
                                                       b2.x, ks2, kn2));
#pragma unroll
                            for (int k = 0; k < NC; k++)
                                st_stream_v2(dg + D + 64 * k + 8 * q, quantise8(lds128(vrow + 128 * k + 16 * q), b2.y, vs2, vn2));
                        }
                    }
                }
                __syncwarp();
                if (lane == 0)
                    mbar_arrive(empty + s);
            }
        }
        __syncwarp();
        __syncthreads();
    }
    flags = __reduce_or_sync(0xffffffffu, flags);
    if (lane == 0 && flags && p.error_flags)
        atomicOr(p.error_flags, flags);
    if (tp.work_counter) {
        // every claim of this CTA is done (its producer has left its loop);
        // the last CTA to finish leaves the counter at zero for the next launch
        __syncthreads();
        __threadfence();
        if (threadIdx.x == 0 && atomicAdd(tp.work_counter + 1, 1ull) == gridDim.x - 1) {
            tp.work_counter[0] = 0;
            tp.work_counter[1] = 0;
            __threadfence();
        }
    }
}

constexpr int kMaxSlabBytes = 32 * 1024;
constexpr int kStageBudget = 106 * 1024;  // per CTA, two CTAs per SM
constexpr int kStages = 3;

struct Plan {
    int Lp, NP, S;
    Layout lay;
};

// xor modes: r = 16, 32 or 64 (the rotated dims all in each lane's first
// chunk, partners r/16 lanes away) for every head dim; any other rotary dim
// takes the shared-memory RoPE (ROT = 0).
bool xor_mode(int head_dim, int rotary_dim)
{
    return (head_dim == 64 || head_dim == 128 || head_dim == 256) &&
           (rotary_dim == 16 || rotary_dim == 32 || rotary_dim == 64);
}

bool plan_for(const CtxKvParams &p, int head_dim, Plan &pl)
{
    const int L = p.num_layers, H = p.num_kv_heads;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256)
        return false;
    const int row_bytes = H * 4 * head_dim;
    if (row_bytes > kMaxSlabBytes || L > kMaxTmaLayers)
        return false;
    pl.Lp = std::min(L, kMaxSlabBytes / row_bytes);
    pl.NP = (L + pl.Lp - 1) / pl.Lp;
    const int pl_tab = p.layer_slots ? pl.Lp : 0;
    const bool xr = xor_mode(head_dim, p.rotary_dim);
    // Three stages measured best on the bf16 long-context workload and as good
    // as four on the fp8 prefill one (a deeper ring of reads in flight slowed
    // the write-heavy bf16 workload); fewer when three would not leave room
    // for two CTAs per SM.
    const Layout one = make_layout(L, 1, (uint32_t)pl.Lp * row_bytes, pl_tab, head_dim, xr);
    const int fixed = (int)one.stages;
    int S = (kStageBudget - fixed) / (int)one.stage_bytes;
    S = S < 2 ? 2 : (S > kStages ? kStages : S);
    pl.S = S;
    pl.lay = make_layout(L, S, (uint32_t)pl.Lp * row_bytes, pl_tab, head_dim, xr);
    return pl.lay.total <= 113 * 1024;
}

int tma_sms(cudaError_t &e)
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

template <int D, int ROT, bool FP8, bool PL>
cudaError_t launch_tma_variant(const TmaParams &tp, uint32_t smem_bytes, cudaStream_t stream)
{
    static std::mutex mu;
    static int sms_cache[64];
    static uint32_t smem_set[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= 64)
        return cudaErrorInvalidDevice;
    int sms;
    {
        std::lock_guard<std::mutex> lock(mu);
        if (sms_cache[dev] == 0) {
            e = cudaDeviceGetAttribute(&sms_cache[dev], cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess)
                return e;
        }
        if (smem_set[dev] < smem_bytes) {
            e = cudaFuncSetAttribute(ctx_kv_tma_kernel<D, ROT, FP8, PL>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     (int)smem_bytes);
            if (e != cudaSuccess)
                return e;
            smem_set[dev] = smem_bytes;
        }
        sms = sms_cache[dev];
    }
    const long long units = tp.p.num_ctx * (long long)tp.pieces;
    const long long want = 2LL * sms;
    const int blocks = (int)(units < want ? units : want);
    return launch_pdl(ctx_kv_tma_kernel<D, ROT, FP8, PL>, blocks, kThreads, smem_bytes, stream, tp);
}

template <int D, int ROT, bool PL>
cudaError_t launch_dtype(const TmaParams &tp, bool fp8, uint32_t smem, cudaStream_t stream)
{
    return fp8 ? launch_tma_variant<D, ROT, true, PL>(tp, smem, stream)
               : launch_tma_variant<D, ROT, false, PL>(tp, smem, stream);
}

template <int D, bool PL>
cudaError_t launch_rot(const TmaParams &tp, int rotary_dim, bool fp8, uint32_t smem, cudaStream_t stream)
{
    switch (xor_mode(D, rotary_dim) ? rotary_dim : 0) {
    case 16:
        return launch_dtype<D, 16, PL>(tp, fp8, smem, stream);
    case 32:
        return launch_dtype<D, 32, PL>(tp, fp8, smem, stream);
    case 64:
        return launch_dtype<D, 64, PL>(tp, fp8, smem, stream);
    default:
        return launch_dtype<D, 0, PL>(tp, fp8, smem, stream);
    }
}

template <bool PL>
cudaError_t launch_layout(const TmaParams &tp, int head_dim, int rotary_dim, bool fp8, uint32_t smem,
                          cudaStream_t stream)
{
    switch (head_dim) {
    case 64:
        return launch_rot<64, PL>(tp, rotary_dim, fp8, smem, stream);
    case 128:
        return launch_rot<128, PL>(tp, rotary_dim, fp8, smem, stream);
    case 256:
        return launch_rot<256, PL>(tp, rotary_dim, fp8, smem, stream);
    default:
        return cudaErrorInvalidValue;
    }
}

}  // namespace

bool tma_path_supported(const CtxKvParams &p, int head_dim)
{
    Plan pl;
    return plan_for(p, head_dim, pl);
}

cudaError_t launch_ctx_kv_write_tma(const CtxKvParams &p, int head_dim, bool fp8, cudaStream_t stream)
{
    Plan pl;
    if (!plan_for(p, head_dim, pl))
        return cudaErrorInvalidValue;
    TmaParams tp;
    tp.p = p;
    tp.layers_per_piece = pl.Lp;
    tp.pieces = pl.NP;
    tp.stages = pl.S;
    tp.h_magic = (0x100000000ull + p.num_kv_heads - 1) / (uint64_t)p.num_kv_heads;
    tp.work_counter = nullptr;
    tp.static_units = 0;
    tp.claim_units = 1;
    cudaError_t e = cudaSuccess;
    const int sms = tma_sms(e);
    if (e != cudaSuccess)
        return e;
    const long long units = p.num_ctx * (long long)pl.NP;
    const long long G = 2LL * sms;
    // slabs prefetched ahead of the dependency wait: the first S units (the
    // ones copied at once after it); 12 on large calls, where a deeper start
    // measured 0.7% faster (long context 208.5 -> 206.9 us) and on prefill
    // 1-3% slower
    tp.prefetch_units = units >= 64 * G ? 12 : pl.S;
    if (p.work_counter) {
        // CTAs of a static launch end up to 6% apart and the slowest one ends
        // it, so on large calls the last tenth of the units is handed out in
        // runs of 4 to whichever CTA is free (long context 211.8 -> 209.5 us,
        // per-layer mappings 222.8 -> 220.4 us).  Below 64 units per CTA the
        // claims cost more than they recover (prefill, 27 units per CTA: 1-3
        // us slower with any tail share and run length tried), so those calls
        // keep the static order.
        if (units >= 64 * G) {
            tp.work_counter = p.work_counter;
            tp.static_units = units * 9 / 10 / G * G;
            tp.claim_units = 4;
        }
    }
    const uint32_t smem = pl.lay.total;
    if (p.layer_slots)
        return launch_layout<true>(tp, head_dim, p.rotary_dim, fp8, smem, stream);
    return launch_layout<false>(tp, head_dim, p.rotary_dim, fp8, smem, stream);
}

}  // namespace dspark
