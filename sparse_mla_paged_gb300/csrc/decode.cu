// The selected-index NoPE MLA paged decode kernel (attend.rs, decode_attention).
//
// One CTA per SM, persistent over a static slot-space partition (see common.cuh). Work
// unit = (decode row, group of 64 query heads). Tiles of 128 resolved tokens stream
// through a 3-tile shared-memory ring (1 tile when K and V are separate buffers):
//
//   gather   warps 0-3   cp.async 16-byte copies of each token's 512-byte E4M3 latent row,
//                        each warp a quarter of every tile (byte offsets resolved by the
//                        prologue; the next tile's offsets are loaded while waiting for a
//                        free slot), written in the 128-byte-swizzled operand layout, 8
//                        tokens (4 KB) per swizzle group.
//   QK^T     warp 4      tcgen05.mma kind::f8f6f4, M = 128 query rows (64 heads x {hi, lo}
//                        terms, A in tensor memory), N = 128 tokens, K = 512: S -> TMEM.
//   softmax  warps 5-12  the hi and lo rows of a head sit in neighbouring TMEM lanes, so
//                        one shuffle gives each thread the full scores of one head for 32
//                        tokens. A head's reference max is raised only when a tile exceeds
//                        it by more than kRescaleMargin (one barrier-reduction per tile
//                        decides for the CTA); then O is rescaled in TMEM. P' =
//                        2^(x - m + kPBias) is stored as two E4M3 terms (hi = top 4 bits,
//                        lo = rest).
//   P.V      warp 3      O^T[512 dims x 64 heads] += V^T * P'^T in TMEM: the ring slot read
//                        as an MN-major operand (K and V are the same bytes).
//   epilogue warps 4-11  O / l * v_scale -> BF16 output, or (O/l, lse) partials, transposed
//                        per warp through shared memory into 16-byte stores.
//
// The contraction is exact in its inputs: keys and values are the cached E4M3 codes
// themselves (k_scale and v_scale are applied outside the MMA), queries are split into
// two E4M3 terms that reproduce the BF16 value (see prologue.cu), probabilities into two
// terms that carry about 8 significant bits. Accumulation is FP32 in TMEM.
//
// Shared memory 226 KB, TMEM 512 columns: O^T at 0..255 (chunk c of 128 dims at 64c),
// query operand at 256..383, S at 384..511. Every wait is bounded (see ptx.cuh); on a
// timeout the CTA records DSA_ERR_TIMEOUT, skips the remaining waits and finishes.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

// This file is compiled once per tile size (DSA_TILE = 64 or 128); each build lives in its
// own namespace and exports decode_kernel_setup_<tile> and launch_decode_<tile>.
#ifndef DSA_TILE
#define DSA_TILE 128
#endif
#define DSA_CAT2(a, b) a##b
#define DSA_CAT(a, b) DSA_CAT2(a, b)

namespace dsa {
namespace DSA_CAT(tile, DSA_TILE) {

constexpr int kTileTokens = DSA_TILE;                     // tokens per decode tile = MMA N of QK
constexpr int kKvTileBytes = kTileTokens * kLatent;       // E4M3 bytes per tile

constexpr int kProducerWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kSoftmaxWarp0 = 5;
constexpr int kSoftmaxWarps = 8;
// 416 threads: one gather warp per SM sub-partition (their copies are issue-bound per
// warp, and a fourth warp measured faster than three on every large workload) and two
// softmax warps each; thirteen warps leave 128 registers per thread.
constexpr int kThreads = (kSoftmaxWarp0 + kSoftmaxWarps) * 32;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;

constexpr int kBarSoftmax = 1;  // named barrier over the softmax warps
constexpr int kBarPair0 = 2;    // 2..5: the two softmax warps of TMEM lane quarter q (64 threads)

// Operand layout of a tile: token tk at (tk/8)*4096 + kb*1024 + (tk%8)*128 for its
// 128-dim block kb, 16-byte chunks of each 128-byte row permuted by tk%8 (128-byte
// swizzle); 8-token groups are the swizzle atoms (stride kGroupBytes).
constexpr int kGroupBytes = 8 * kLatent;  // 4 KB
constexpr int kRingBytes = 192 * 1024;                           // ring of tiles (K == V)
constexpr int kSlotsKV = kRingBytes / kKvTileBytes;              // tiles in flight when K == V
constexpr int kSBufs = 128 / kTileTokens;                        // S buffers in TMEM columns 384..511
constexpr int kHalfCols = kTileTokens / 2;                       // S columns per softmax warp
constexpr int kScores = kHalfCols / 2;                           // scores per softmax thread per tile
constexpr int kPTermBytes = kHeadsPerCta * kTileTokens;          // one E4M3 term of P'^T
static_assert(kSlotsKV <= 6 && kSBufs >= 1 && kScores % 16 == 0, "tile geometry");
constexpr int kOffRing = 0;
constexpr int kOffP = kOffRing + kRingBytes;                     // P' [2 buffers][hi, lo]; epilogue staging
constexpr int kOffHm = kOffP + 4 * kPTermBytes;                  // float [2 token halves][64] tile maxima
constexpr int kOffAlpha = kOffHm + 2 * kHeadsPerCta * 4;         // float [2 tile parities][64] rescale factors
constexpr int kOffL = kOffAlpha + 2 * kHeadsPerCta * 4;          // float [2 token halves][64] row sums
constexpr int kOffF = kOffL + 2 * kHeadsPerCta * 4;              // float [64] output factors
constexpr int kOffFlags = kOffF + kHeadsPerCta * 4;              // u32 [2 tile parities][4 lane quarters]
constexpr int kOffBars = kOffFlags + 2 * 4 * 4;
enum {
    BAR_FULL0 = 0,    // 6: ring slot gathered
    BAR_EMPTY0 = 6,   // 6: ring slot free again (its P.V is done)
    BAR_SFULL0 = 12,  // 2: S buffer written by QK
    BAR_SEMPTY0 = 14, // 2: S buffer read by the softmax warps
    BAR_PFULL0 = 16,  // 2: P buffer written
    BAR_PVDONE0 = BAR_PFULL0 + 2,  // 2: the P.V reading a P buffer is done
    BAR_QFULL = BAR_PVDONE0 + 2,
    BAR_QEMPTY,
    BAR_OEMPTY,
    BAR_DRAIN,
    BAR_DONE,
    kNumBars
};
constexpr int kOffTmemSlot = kOffBars + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kSmemUsed = kOffAbort + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for the 1024-byte alignment
static_assert(kSmemBytes <= 227 * 1024, "shared memory");

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemQ = 256;
constexpr uint32_t kTmemS = 384;

constexpr float kNegInf = -__builtin_huge_valf();

// Optional per-CTA timeline (clock64 values), compiled in only with -DDSA_TRACE: slot i of
// CTA c is trace[c*128 + i].
#ifdef DSA_TRACE
#define DSA_TRACE_AT(p, i)                                                                               \
    do {                                                                                                 \
        if ((p).trace && (i) < 128) (p).trace[static_cast<int64_t>(blockIdx.x) * 128 + (i)] = clock64(); \
    } while (0)
#else
#define DSA_TRACE_AT(p, i) \
    do {                   \
    } while (0)
#endif

struct Tiles {
    int32_t n;       // resolved tokens of this segment
    int64_t t0;      // first resolved token
    int32_t ntiles;
};

// Resolved tokens of a segment: positions [s0, s1) of the row's resolved list, clipped to
// its count U (the list holds the U distinct ids first).
__device__ __forceinline__ Tiles segment_tokens(const DecodeParams& p, const Segment& s) {
    const int64_t U = p.cnt[s.row];
    Tiles t;
    t.t0 = s.s0 < U ? s.s0 : U;
    const int64_t t1 = s.s1 < U ? s.s1 : U;
    t.n = static_cast<int32_t>(t1 - t.t0);
    t.ntiles = (t.n + kTileTokens - 1) / kTileTokens;
    return t;
}

__device__ __forceinline__ void fail(const DecodeParams& p, volatile int* abort_flag, int code) {
    atomicCAS(p.status, 0, code);
    *abort_flag = 1;
}

// Every lane of the warp waits for the phase (each acquires it), then the warp is
// reconverged before any warp-aligned tcgen05 or barrier instruction that follows.
__device__ __forceinline__ void warp_wait(const DecodeParams& p, uint32_t bar, uint32_t parity,
                                          volatile int* abort_flag) {
    if (!mbar_wait(bar, parity, abort_flag, p.wait_limit_ns)) fail(p, abort_flag, kStatusTimeout);
    __syncwarp();
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    return f32x2_to_e4m3x2(a, b) | (f32x2_to_e4m3x2(c, d) << 16);
}

// x rounded to 4 significant bits (sign, exponent and the top three mantissa bits, round
// half up on the magnitude): an E4M3-representable value for magnitudes in E4M3's normal
// range, leaving a remainder of at most half a unit in its last place.
__device__ __forceinline__ float hi_part(float x) {
    return __uint_as_float((__float_as_uint(x) + 0x00080000u) & 0xFFF00000u);
}

__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Ring geometry: with K and V in one buffer each slot holds one tile; otherwise a slot
// holds a K tile followed by the V tile.
struct Ring {
    int slots;
    uint32_t slot_bytes;
    __device__ explicit Ring(int kv_same)
        : slots(kv_same ? kSlotsKV : kSlotsKV / 2), slot_bytes(kv_same ? kKvTileBytes : 2 * kKvTileBytes) {}
};

// ------------------------------------------------------------------------------------
// gather warps
// ------------------------------------------------------------------------------------
// Rows of a tile taken by gather warp w: [w*kWarpRows, min((w+1)*kWarpRows, kTileTokens)).
constexpr int kWarpRows = (kTileTokens + kProducerWarps - 1) / kProducerWarps;

__device__ void run_producer(const DecodeParams& p, uint32_t sbase, volatile int* abort_flag, int nseg,
                             const Segment& seg0) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const Ring ring(p.kv_same);
    const int64_t W = p.part.width;
    const int r0 = warp * kWarpRows;
    const int nr = min(kWarpRows, kTileTokens - r0);
    uint32_t tau = 0;
    if (tid == 0) DSA_TRACE_AT(p, 2);
    for (int i = 0; i < nseg; ++i) {
        const Segment s = i == 0 ? seg0 : cta_segment(p.part, blockIdx.x, i);
        if (tid == 0 && i == 0) DSA_TRACE_AT(p, 3);
        // The segment's tokens start at position s0 of the row's resolved list, so the first
        // tile's offsets are requested together with the row's count (positions past the
        // count hold stale values and are masked once it arrives).
        const long long* offs = p.offs + static_cast<int64_t>(s.row) * W + s.s0;
        const int32_t span = static_cast<int32_t>(s.s1 - s.s0);
        const long long pa = (r0 + lane < span) ? offs[r0 + lane] : -1;
        const long long pb = (lane + 32 < nr && r0 + 32 + lane < span) ? offs[r0 + 32 + lane] : -1;
        const Tiles tl = segment_tokens(p, s);
        if (tid == 0 && i == 0 && tl.n >= 0) DSA_TRACE_AT(p, 4);
        if (tl.n <= 0) continue;
        // This lane's rows of tile t: r0 + lane and r0 + 32 + lane (the latter for lane < nr - 32).
        auto load = [&](int t, long long& a, long long& b) {
            const int ta = t * kTileTokens + r0 + lane, tb = ta + 32;
            a = (t < tl.ntiles && ta < tl.n) ? offs[ta] : -1;
            b = (t < tl.ntiles && lane + 32 < nr && tb < tl.n) ? offs[tb] : -1;
        };
        long long oa = (r0 + lane < tl.n) ? pa : -1;
        long long ob = (lane + 32 < nr && r0 + 32 + lane < tl.n) ? pb : -1;
        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            const long long ca = oa, cb = ob;
            if (tid == 0 && t == 0 && i == 0 && ca != 12345) DSA_TRACE_AT(p, 5);
            load(t + 1, oa, ob);  // next tile's rows, before the slot wait
            if (tid == 0 && t == 0 && i == 0) DSA_TRACE_AT(p, 6);
            if ((ca < 0 && t * kTileTokens + r0 + lane < tl.n) ||
                (cb < 0 && lane + 32 < nr && t * kTileTokens + r0 + 32 + lane < tl.n))
                atomicCAS(p.status, 0, kStatusBounds);
            if (tid == 0 && t == 0 && i == 0) DSA_TRACE_AT(p, 7);
            const int e = static_cast<int>(tau % ring.slots);
            const uint32_t use = tau / ring.slots;
            if (tau >= static_cast<uint32_t>(ring.slots))
                warp_wait(p, sbase + kOffBars + 8 * (BAR_EMPTY0 + e), (use - 1) & 1, abort_flag);
            if (tid == 0 && tau < 8) DSA_TRACE_AT(p, 40 + tau);
            const uint32_t kdst = sbase + kOffRing + e * ring.slot_bytes;
            const uint32_t vdst = kdst + kKvTileBytes;
            // Branch-free copy loop (a branch on the shuffled offset would serialise the
            // copies): rows without a token (o < 0) are zero-filled by a source size of 0.
            // Each row's offset is broadcast from the lane holding it. Offsets below 64 GiB
            // travel as 32-bit counts of 16-byte units (one shuffle per row; 0xFFFFFFFF marks
            // a row without token); a tile with a larger offset takes the 64-bit path.
            const uint8_t* kbase = p.k_cache + lane * 16;
            const uint8_t* vbase = p.v_cache + lane * 16;
            auto copy_row = [&](long long o, int tk) {
                const uint32_t d = (tk >> 3) * kGroupBytes + (lane >> 3) * 1024 + (tk & 7) * 128 +
                                   (((lane & 7) ^ (tk & 7)) << 4);
                const bool ok = o >= 0;
                const uint64_t src = ok ? static_cast<uint64_t>(o) : 0;
                cp_async_16_zfill(kdst + d, kbase + src, ok ? 16u : 0u);
                if (!p.kv_same) cp_async_16_zfill(vdst + d, vbase + src, ok ? 16u : 0u);
            };
            constexpr long long kNarrow = 1ll << 36;
            if (!__any_sync(0xffffffffu, ca >= kNarrow || cb >= kNarrow)) {
                auto to16 = [](long long o) { return o >= 0 ? static_cast<uint32_t>(o >> 4) : 0xFFFFFFFFu; };
                auto from16 = [](uint32_t u) { return u != 0xFFFFFFFFu ? static_cast<long long>(u) << 4 : -1ll; };
                const uint32_t ua = to16(ca), ub = to16(cb);
#pragma unroll 8
                for (int j = 0; j < min(nr, 32); ++j) copy_row(from16(__shfl_sync(0xffffffffu, ua, j)), r0 + j);
                if (kWarpRows > 32)
                    for (int j = 32; j < nr; ++j) copy_row(from16(__shfl_sync(0xffffffffu, ub, j - 32)), r0 + j);
            } else {
#pragma unroll 4
                for (int j = 0; j < min(nr, 32); ++j) copy_row(__shfl_sync(0xffffffffu, ca, j), r0 + j);
                if (kWarpRows > 32)
                    for (int j = 32; j < nr; ++j) copy_row(__shfl_sync(0xffffffffu, cb, j - 32), r0 + j);
            }
            // One arrival per lane, made when the lane's copies so far have landed (.noinc: the
            // arrival counts toward the barrier's expected 96 per tile).
            cp_async_arrive_noinc(sbase + kOffBars + 8 * (BAR_FULL0 + e));
            if (tid == 0 && tau < 8) DSA_TRACE_AT(p, 48 + tau);
        }
    }
    cp_async_wait_all();
}

// ------------------------------------------------------------------------------------
// gather by tensor map (pages of block_size*512 bytes: token row = page*block_size + slot)
// ------------------------------------------------------------------------------------
// Warp 0 alone: lane l (l < kGroups4) fetches tokens 4l..4l+3 of every tile with one
// tile::gather4 per 128-dim block, straight into the 128-byte-swizzled operand layout
// (the swizzle follows the shared-memory address, and each token group's rows sit at
// (tk/8)*4096 + kb*1024 + (tk%8)*128 of the slot). Rows without a token take index -1
// and are zero-filled. One arrive.expect_tx per tile arms the slot's full barrier.
constexpr int kGroups4 = kTileTokens / 4;

__device__ void run_producer_tma(const DecodeParams& p, const CUtensorMap* kmap, const CUtensorMap* vmap,
                                 uint32_t sbase, volatile int* abort_flag, int nseg, const Segment& seg0) {
    const int lane = threadIdx.x & 31;
    const Ring ring(p.kv_same);
    const int64_t W = p.part.width;
    const uint32_t tile_bytes = (p.kv_same ? 1u : 2u) * static_cast<uint32_t>(kKvTileBytes);
    const bool active = lane < kGroups4;
    const uint32_t lane_dst = ((4 * lane) >> 3) * kGroupBytes + ((4 * lane) & 7) * 128;
    uint32_t tau = 0;
    bool stop = false;
    for (int i = 0; i < nseg && !stop; ++i) {
        const Segment s = i == 0 ? seg0 : cta_segment(p.part, blockIdx.x, i);
        const long long* offs = p.offs + static_cast<int64_t>(s.row) * W + s.s0;
        const int32_t span = static_cast<int32_t>(s.s1 - s.s0);
        // The first tile's offsets are requested together with the row's count.
        long long o4[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) o4[k] = (active && 4 * lane + k < span) ? offs[4 * lane + k] : -1;
        const Tiles tl = segment_tokens(p, s);
        if (tl.n <= 0) continue;
        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            int32_t y[4];
            bool bad = false;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const bool in = active && t * kTileTokens + 4 * lane + k < tl.n;
                y[k] = (in && o4[k] >= 0) ? static_cast<int32_t>(o4[k] >> 9) : -1;
                bad |= in && o4[k] < 0;
            }
            if (bad) atomicCAS(p.status, 0, kStatusBounds);
            // next tile's offsets, before the slot wait
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int j = (t + 1) * kTileTokens + 4 * lane + k;
                o4[k] = (active && t + 1 < tl.ntiles && j < tl.n) ? offs[j] : -1;
            }
            const int e = static_cast<int>(tau % ring.slots);
            const uint32_t use = tau / ring.slots;
            if (tau >= static_cast<uint32_t>(ring.slots))
                warp_wait(p, sbase + kOffBars + 8 * (BAR_EMPTY0 + e), (use - 1) & 1, abort_flag);
            // After a failed wait nothing more is issued: every copy in flight then targets a
            // slot whose previous contents were consumed, and the drain below finds it.
            if (__shfl_sync(0xffffffffu, *abort_flag, 0)) {
                stop = true;
                break;
            }
            if (tau < 8 && lane == 0) DSA_TRACE_AT(p, 40 + tau);
            const uint32_t full = sbase + kOffBars + 8 * (BAR_FULL0 + e);
            if (lane == 0) mbar_arrive_expect_tx(full, tile_bytes);
            __syncwarp();
            const uint32_t kdst = sbase + kOffRing + e * ring.slot_bytes + lane_dst;
            if (active) {
#pragma unroll
                for (int kb = 0; kb < 4; ++kb)
                    tma_gather4(kdst + kb * 1024, kmap, kb * 128, y[0], y[1], y[2], y[3], full);
                if (!p.kv_same) {
#pragma unroll
                    for (int kb = 0; kb < 4; ++kb)
                        tma_gather4(kdst + kKvTileBytes + kb * 1024, vmap, kb * 128, y[0], y[1], y[2], y[3], full);
                }
            }
            if (tau < 8 && lane == 0) DSA_TRACE_AT(p, 48 + tau);
        }
    }
    // Drain: only the last ring.slots tiles can still be landing; wait for each one's
    // bytes (bounded) so that no copy into shared memory is in flight when the CTA exits.
    if (lane == 0) {
        const uint32_t first = tau > static_cast<uint32_t>(ring.slots) ? tau - ring.slots : 0;
        for (uint32_t k = first; k < tau; ++k) {
            const uint32_t bar = sbase + kOffBars + 8 * (BAR_FULL0 + static_cast<int>(k % ring.slots));
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(bar, (k / ring.slots) & 1) && globaltimer_ns() - t0 < kDrainLimitNs) {
            }
        }
    }
    __syncwarp();
}

// ------------------------------------------------------------------------------------
// MMA warp (one thread issues)
// ------------------------------------------------------------------------------------
// Warp-uniform wait: every lane polls, the warp leaves together (lane 0 decides timeouts).
__device__ __forceinline__ bool warp_poll(uint32_t bar, uint32_t parity) {
    return __all_sync(0xffffffffu, mbar_try_wait(bar, parity) != 0);
}
// Slow path of mma_wait, out of line (see mbar_wait).
static __device__ __noinline__ void mma_wait_slow(const DecodeParams& p, uint32_t bar, uint32_t parity,
                                           volatile int* abort_flag) {
    if (p.wait_limit_ns < kPollHintNs) {  // below the polling interval: the test has failed
        fail(p, abort_flag, kStatusTimeout);
        return;
    }
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        mbar_try_wait_hint(bar, parity, kPollHintNs);
        if (warp_poll(bar, parity)) return;
        const bool give_up =
            __shfl_sync(0xffffffffu, (*abort_flag != 0) || globaltimer_ns() - t0 > p.wait_limit_ns, 0);
        if (give_up) {
            fail(p, abort_flag, kStatusTimeout);
            return;
        }
    }
}
__device__ __forceinline__ void mma_wait(const DecodeParams& p, uint32_t bar, uint32_t parity,
                                         volatile int* abort_flag) {
    // Below the polling interval a single non-blocking test decides.
    const bool done = p.wait_limit_ns < kPollHintNs ? __all_sync(0xffffffffu, mbar_test_wait(bar, parity) != 0)
                                                     : warp_poll(bar, parity);
    if (!done) mma_wait_slow(p, bar, parity, abort_flag);
}

// The whole MMA warp runs this loop converged; the elected lane issues.
__device__ void run_mma(const DecodeParams& p, uint32_t sbase, uint32_t tmem, volatile int* abort_flag, int nseg,
                        const Segment& seg0) {
    const Ring ring(p.kv_same);
    const uint32_t idq = idesc_e4m3(128, kTileTokens, false, false);
    const uint32_t idp = idesc_e4m3(128, kHeadsPerCta, true, false);
    const uint32_t el = elect_one();
    auto barp = [&](int b) { return sbase + kOffBars + 8 * b; };
    int qseg = 0;  // non-empty units entered so far

    // Descriptors are formed once per tile and stepped by immediate offsets (the start
    // address field counts 16-byte units).
    const uint64_t pdesc0 = smem_desc(sbase + kOffP, 1024, 128, kSwizzleNone);
    auto issue_pv = [&](uint32_t tp, bool first) {
        const int pb = tp & 1;
        mma_wait(p, barp(BAR_PFULL0 + pb), (tp >> 1) & 1, abort_flag);
        if (first && qseg > 0) mma_wait(p, barp(BAR_OEMPTY), (qseg - 1) & 1, abort_flag);
        tc_fence_after();
        const int e = static_cast<int>(tp % ring.slots);
        const uint32_t vbase = sbase + kOffRing + e * ring.slot_bytes + (p.kv_same ? 0u : kKvTileBytes);
        // V^T: 128 dims of block mc x 32 tokens (4 swizzle groups), MN-major. P'^T: 64 heads
        // x 32 tokens, K-major core matrices (token chunk stride 1 KB, head group 128 B).
        const uint64_t vdesc = smem_desc(vbase, 1024, kGroupBytes, kSwizzle128B);
        const uint64_t pdesc = pdesc0 + static_cast<uint64_t>((pb * 2 * kPTermBytes) >> 4);
#pragma unroll
        for (int mc = 0; mc < 4; ++mc) {
#pragma unroll
            for (int ks = 0; ks < kTileTokens / 32; ++ks) {
                const uint64_t a = vdesc + static_cast<uint64_t>((ks * 4 * kGroupBytes + mc * 1024) >> 4);
                const uint64_t bh = pdesc + static_cast<uint64_t>((ks * 2048) >> 4);
                const uint64_t bl = pdesc + static_cast<uint64_t>((kPTermBytes + ks * 2048) >> 4);
                const uint32_t d = tmem + kTmemO + mc * 64;
                if (ks == 0)
                    mma_e4m3_el(d, a, bh, idp, first ? 0u : 1u, el);
                else
                    mma_e4m3_acc_el(d, a, bh, idp, el);
                mma_e4m3_acc_el(d, a, bl, idp, el);
            }
        }
        tc_commit_el(barp(BAR_PVDONE0 + pb), el);
        tc_commit_el(barp(BAR_EMPTY0 + e), el);
    };

    auto issue_qk = [&](uint32_t tq) {
        const int e = static_cast<int>(tq % ring.slots);
        fence_proxy_async_smem();
        tc_fence_after();
        // K: 128 tokens x 32 dims of block ks/4, K-major (8-token group stride 4 KB).
        const uint64_t kdesc = smem_desc(sbase + kOffRing + e * ring.slot_bytes, 16, kGroupBytes, kSwizzle128B);
        const int sb = static_cast<int>(tq % kSBufs);
        const uint32_t d = tmem + kTmemS + sb * kTileTokens;
        mma_e4m3_ta_el(d, tmem + kTmemQ, kdesc, idq, 0u, el);
#pragma unroll
        for (int ks = 1; ks < 16; ++ks)
            mma_e4m3_ta_acc_el(d, tmem + kTmemQ + ks * 8,
                               kdesc + static_cast<uint64_t>(((ks >> 2) * 1024 + (ks & 3) * 32) >> 4), idq, el);
        tc_commit_el(barp(BAR_SFULL0 + sb), el);
    };
    // QK of tile tq may start once its ring slot is full and its S buffer has been read.
    auto qk_ready = [&](uint32_t tq) {
        const int e = static_cast<int>(tq % ring.slots);
        return warp_poll(barp(BAR_FULL0 + e), (tq / ring.slots) & 1) &&
               (tq < kSBufs || warp_poll(barp(BAR_SEMPTY0 + static_cast<int>(tq % kSBufs)), ((tq / kSBufs) - 1) & 1));
    };

    uint32_t tau = 0;
    Tiles tl_next = segment_tokens(p, seg0);
    for (int i = 0; i < nseg; ++i) {
        const Tiles tl = tl_next;
        // The next unit's count is read a unit ahead, its latency hidden behind this unit.
        if (i + 1 < nseg) tl_next = segment_tokens(p, cta_segment(p.part, blockIdx.x, i + 1));
        if (tl.n <= 0) continue;
        mma_wait(p, barp(BAR_QFULL), qseg & 1, abort_flag);
        tc_fence_after();
        const uint32_t tau0 = tau;
        // QK(t) and PV(t-1) are independent: issue whichever becomes ready first.
        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            bool qk_done = false, pv_done = (t == 0);
            const uint64_t t_start = globaltimer_ns();
            while (!qk_done || !pv_done) {
                if (!qk_done && qk_ready(tau)) {
                    if (tau < 8) DSA_TRACE_AT(p, 56 + tau);
                    issue_qk(tau);
                    if (t == tl.ntiles - 1) tc_commit_el(barp(BAR_QEMPTY), el);
                    qk_done = true;
                }
                if (!pv_done && warp_poll(barp(BAR_PFULL0 + ((tau - 1) & 1)), ((tau - 1) >> 1) & 1)) {
                    if (tau - 1 < 8) DSA_TRACE_AT(p, 64 + tau - 1);
                    issue_pv(tau - 1, tau - 1 == tau0);
                    pv_done = true;
                }
                if (!qk_done || !pv_done) {
                    const bool give_up = __shfl_sync(0xffffffffu,
                                                     (*abort_flag != 0) || p.wait_limit_ns < kPollHintNs ||
                                                         globaltimer_ns() - t_start > p.wait_limit_ns,
                                                     0);
                    if (give_up) {
                        fail(p, abort_flag, kStatusTimeout);
                        break;
                    }
                    // Sleep briefly on the barrier still awaited instead of spinning.
                    if (!pv_done)
                        mbar_try_wait_hint(barp(BAR_PFULL0 + ((tau - 1) & 1)), ((tau - 1) >> 1) & 1, kPollHintNs);
                    else
                        mbar_try_wait_hint(barp(BAR_FULL0 + static_cast<int>(tau % ring.slots)),
                                           (tau / ring.slots) & 1, kPollHintNs);
                }
            }
        }
        issue_pv(tau - 1, tl.ntiles == 1);
        ++qseg;
    }
    DSA_TRACE_AT(p, 10);
}

// ------------------------------------------------------------------------------------
// softmax / epilogue warps
// ------------------------------------------------------------------------------------

// Writes a warp's 32 dims x 32 heads block (dims on lanes, v[k] = head h0+k, scaled by
// f[k]) to row-major global rows (row stride kLatent elements) through the warp's 2 KB
// staging area (one staging round for all 32 heads), with 16-byte stores. T is bf16
// (output) or f16 (partials). Heads at or beyond hvalid are not written.
template <typename T>
__device__ __forceinline__ void store_block(T* rows, int h0, int hvalid, int dim0, const float* v, const float* f,
                                            uint8_t* stage, int lane) {
    constexpr int kPer16 = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte store
    constexpr int kLanesPerRow = 32 / kPer16;                 // lanes covering one head's 32 dims
    constexpr int kRowsPerPass = 32 / kLanesPerRow;           // heads per warp-wide store
    static_assert(32 * 32 * sizeof(T) <= 2048, "staging area");
    T* stg = reinterpret_cast<T*>(stage);                     // [32 heads][32 dims]
#pragma unroll
    for (int k = 0; k < 32; ++k) {
        const float x = v[k] * f[k];
        if constexpr (std::is_same<T, __half>::value) {
            stg[k * 32 + lane] = __float2half_rn(x);
        } else {
            stg[k * 32 + lane] = __float2bfloat16_rn(x);
        }
    }
    __syncwarp();
#pragma unroll
    for (int pass = 0; pass < 32 / kRowsPerPass; ++pass) {
        const int hk = pass * kRowsPerPass + lane / kLanesPerRow;
        const int c = (lane % kLanesPerRow) * kPer16;
        const uint4 val = *reinterpret_cast<const uint4*>(stg + hk * 32 + c);
        if (h0 + hk < hvalid)
            *reinterpret_cast<uint4*>(rows + static_cast<int64_t>(h0 + hk) * kLatent + dim0 + c) = val;
    }
    __syncwarp();
}

__device__ void run_softmax(const DecodeParams& p, uint8_t* smem, uint32_t sbase, uint32_t tmem,
                            volatile int* abort_flag, int nseg, const Segment& seg0) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sw = warp - kSoftmaxWarp0;      // 0..7
    const int q4 = warp & 3;                  // TMEM lane quarter of this warp
    const int half = sw >> 2;                 // token half of each tile: kHalfCols columns
    const int term = lane & 1;                // 0: hi row, 1: lo row
    const int hq = 16 * q4 + (lane >> 1);     // head of this thread within the unit
    const int st = sw * 32 + lane;            // 0..255
    float* hm_s = reinterpret_cast<float*>(smem + kOffHm);
    float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
    float* l_s = reinterpret_cast<float*>(smem + kOffL);
    float* f_s = reinterpret_cast<float*>(smem + kOffF);
    uint32_t* flag_s = reinterpret_cast<uint32_t*>(smem + kOffFlags);
    static_assert(kSoftmaxWarps * 2048 <= 4 * kPTermBytes, "epilogue staging fits the P buffers");
    uint8_t* stage = smem + kOffP + sw * 2048;  // epilogue staging (2 KB per warp)
    auto barp = [&](int b) { return sbase + kOffBars + 8 * b; };
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    // This thread's first 16-byte row in a P' term buffer: K-major core matrices of 8 heads
    // x 16 tokens, token chunk kc = (half*kHalfCols + term*kScores)/16 (+1 per further 16
    // tokens), head group hq/8 (chunk stride 1 KB, group stride 128 B).
    const uint32_t p_off = (((half * kHalfCols + term * kScores) / 16) * 8 + (hq >> 3)) * 128 + (hq & 7) * 16;
    uint32_t tau = 0;
    int qseg = 0;

    // Query operand of a unit into TMEM (the previous unit's QKs must be done).
    auto load_q = [&](int32_t unit) {
        // Chunk-major image (chunk c of row r at c*2048 + r*16): each load of the warp is 512
        // contiguous bytes.
        const uint4* src = reinterpret_cast<const uint4*>(p.qimg + static_cast<int64_t>(unit) * kQImageBytes +
                                                          half * 16 * 2048 + (q4 * 32 + lane) * 16);
        // All sixteen loads are issued before either store: one memory round trip.
        uint32_t a[2][32];
#pragma unroll
        for (int hc = 0; hc < 2; ++hc)
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const uint4 v = src[(hc * 8 + c) * (2048 / 16)];
                a[hc][4 * c] = v.x;
                a[hc][4 * c + 1] = v.y;
                a[hc][4 * c + 2] = v.z;
                a[hc][4 * c + 3] = v.w;
            }
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) tmem_st_x32(tmem + lane_base + kTmemQ + half * 64 + hc * 32, a[hc]);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(barp(BAR_QFULL));
    };
    // The next unit's row count and query scale are read at the start of the current one
    // (plain loads whose latency the unit's tiles hide).
    Segment s_next = seg0;
    Tiles tl_next = segment_tokens(p, seg0);
    bool q_loaded = false;  // the current unit's query operand was loaded during the previous unit
    float c_next = p.qscale[static_cast<int64_t>(seg0.unit) * kHeadsPerCta + hq];
    bool pv_seen = false;   // the P.V two tiles back was already waited for (rescale or epilogue)
    for (int i = 0; i < nseg; ++i) {
        const Segment s = s_next;
        const Tiles tl = tl_next;
        const float c = c_next;
        if (i + 1 < nseg) {
            s_next = cta_segment(p.part, blockIdx.x, i + 1);
            tl_next = segment_tokens(p, s_next);
            c_next = p.qscale[static_cast<int64_t>(s_next.unit) * kHeadsPerCta + hq];
        }
        const int hvalid = min(kHeadsPerCta, p.heads - s.group * kHeadsPerCta);
        const int64_t head0 = static_cast<int64_t>(s.row) * p.heads + s.group * kHeadsPerCta;
        if (tl.n <= 0) {
            // Empty selection: the output is zero; a partial carries weight zero.
            if (s.part < 0) {
                uint4* o = reinterpret_cast<uint4*>(p.out + head0 * kLatent);
                for (int e = st; e < hvalid * kLatent / 8; e += kSoftmaxThreads) o[e] = make_uint4(0, 0, 0, 0);
            } else {
                uint4* po = reinterpret_cast<uint4*>(p.part_o + static_cast<int64_t>(s.part) * kHeadsPerCta * kLatent);
                for (int e = st; e < kHeadsPerCta * kLatent / 8; e += kSoftmaxThreads) po[e] = make_uint4(0, 0, 0, 0);
                if (st < kHeadsPerCta) p.part_lse[s.part * kHeadsPerCta + st] = kNegInf;
            }
            continue;
        }
        // Query operand of this unit into TMEM, once the previous unit's QKs are done
        // (already there when it was loaded before the previous unit's epilogue).
        if (!q_loaded) {
            if (qseg > 0) warp_wait(p, barp(BAR_QEMPTY), (qseg - 1) & 1, abort_flag);
            load_q(s.unit);
        }
        q_loaded = false;
        float m_ref = kNegInf;  // reference max of head hq (log2 units)
        float m_top = kNegInf;  // highest reference of head hq so far
        float l_part = 0.0f;    // this thread's share of the row sum of P'

        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            // The next unit's query image was written by the prologue long before and has
            // left L2 under the gather stream: fetch it back a few tiles before it is read.
            if (st < 16 && i + 1 < nseg && tl_next.n > 0 && t == max(0, tl.ntiles - 3))
                bulk_prefetch_l2(p.qimg + static_cast<int64_t>(s_next.unit) * kQImageBytes + st * (kQImageBytes / 16),
                                 kQImageBytes / 16);
            const int sb = static_cast<int>(tau % kSBufs);
            warp_wait(p, barp(BAR_SFULL0 + sb), (tau / kSBufs) & 1, abort_flag);
            if (st == 0 && tau < 8) DSA_TRACE_AT(p, 24 + tau);
            tc_fence_after();
            uint32_t v[kHalfCols];
#pragma unroll
            for (int k = 0; k < kHalfCols / 32; ++k)
                tmem_ld_x32(tmem + lane_base + kTmemS + sb * kTileTokens + half * kHalfCols + 32 * k,
                            *reinterpret_cast<uint32_t(*)[32]>(v + 32 * k));
            if (st == 0 && (tau == 2 || tau == 3)) DSA_TRACE_AT(p, 72 + 8 * (tau - 2));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(barp(BAR_SEMPTY0 + sb));

            // Scores of head hq for tokens tok0 .. tok0+kScores-1: this lane's term plus the
            // neighbouring lane's other term. The hi lane keeps the first kScores columns of
            // its half, the lo lane the last kScores.
            const int tok0 = t * kTileTokens + half * kHalfCols + term * kScores;
            float x[kScores];
            float hm4[4] = {kNegInf, kNegInf, kNegInf, kNegInf};  // four independent max chains
#pragma unroll
            for (int j = 0; j < kScores; ++j) {
                const float send = __uint_as_float(term ? v[j] : v[kScores + j]);
                const float mine = __uint_as_float(term ? v[kScores + j] : v[j]);
                const float other = __shfl_xor_sync(0xffffffffu, send, 1);
                x[j] = (mine + other) * c;
            }
            if (t == tl.ntiles - 1) {  // only the last tile can hold positions past the count
#pragma unroll
                for (int j = 0; j < kScores; ++j)
                    if (tok0 + j >= tl.n) x[j] = kNegInf;
            }
#pragma unroll
            for (int j = 0; j < kScores; ++j) hm4[j & 3] = fmaxf(hm4[j & 3], x[j]);
            // Max of head hq over the tile: this warp's half (both term lanes), then the
            // other half from the partner warp of the lane quarter (64-thread barrier; the
            // buffer is rewritten only after the block barrier below, which the partner
            // passes after reading it).
            float hmax = fmaxf(fmaxf(hm4[0], hm4[1]), fmaxf(hm4[2], hm4[3]));
            hmax = fmaxf(hmax, __shfl_xor_sync(0xffffffffu, hmax, 1));
            if (term == 0) hm_s[half * kHeadsPerCta + hq] = hmax;
            named_bar_sync_id(kBarPair0 + q4, 64);
            const float tm = fmaxf(hm_s[hq], hm_s[kHeadsPerCta + hq]);
            if (st == 0 && (tau == 2 || tau == 3)) DSA_TRACE_AT(p, 73 + 8 * (tau - 2));
            // Reset the reference of head hq when the tile max exceeds it by more than the
            // margin, or lies more than kRescaleDrop below it; O and the row sums are
            // rescaled by 2^(m_old - m_new). Every thread of the head's pair computes the
            // same values; the factors are published (double-buffered by tile parity: a
            // buffer is rewritten two tiles later, after every reader passed the next
            // block barrier) and one block barrier tells every warp whether any changed.
            const bool change = tm > m_ref + kRescaleMargin || (tm < m_ref - kRescaleDrop && m_ref > m_top - kRescaleFloor);
            float alpha = 1.0f;
            if (change) {
                const float m_new = fmaxf(tm + kRescaleSlack, m_top - kRescaleFloor);
                alpha = m_ref == kNegInf ? 0.0f : ex2_approx(m_ref - m_new);
                l_part *= alpha;
                m_ref = m_new;
                m_top = fmaxf(m_top, m_new);
            }
            const float* alpha_t = alpha_s + (tau & 1) * kHeadsPerCta;
            if (term == 0 && half == 0) alpha_s[(tau & 1) * kHeadsPerCta + hq] = alpha;
            // Which of this lane quarter's 16 heads changed (both warps of the pair agree).
            const uint32_t changed = __ballot_sync(0xffffffffu, change);
            if (half == 0 && lane == 0) flag_s[(tau & 1) * 4 + q4] = changed;
            const bool any_change = named_bar_any<kBarSoftmax, kSoftmaxThreads>(change);
            if (st == 0 && (tau == 2 || tau == 3)) DSA_TRACE_AT(p, 77 + 8 * (tau - 2));
            // 32-head blocks of O^T that need rescaling before this tile's P.V: heads 0-31
            // live in lane quarters 0-1, heads 32-63 in 2-3 (uniform over the softmax warps).
            bool resc[2] = {false, false};
            if (any_change && t > 0) {
                const uint4 f = *reinterpret_cast<const uint4*>(flag_s + (tau & 1) * 4);
                resc[0] = (f.x | f.y) != 0u;
                resc[1] = (f.z | f.w) != 0u;
            }

            // P' = 2^(x - m + kPBias) as two E4M3 terms, 16 tokens per 16-byte row.
            uint32_t hw[kScores / 4], lw[kScores / 4];
            float ls4[4] = {0.0f, 0.0f, 0.0f, 0.0f};  // four independent sum chains
            const float off = kPBias - m_ref;
#pragma unroll
            for (int g = 0; g < kScores / 4; ++g) {
                float ph[4], pl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float pp = ex2_approx(x[4 * g + e] + off);
                    ls4[e] += pp;
                    ph[e] = hi_part(pp);
                    pl[e] = pp - ph[e];
                }
                hw[g] = pack_e4m3x4(ph[0], ph[1], ph[2], ph[3]);
                lw[g] = pack_e4m3x4(pl[0], pl[1], pl[2], pl[3]);
            }
            l_part += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
            if (st == 0 && (tau == 2 || tau == 3)) DSA_TRACE_AT(p, 74 + 8 * (tau - 2));
            // P buffer tau%2 is free once the P.V two tiles back has finished reading it.
            if (tau >= 2 && !pv_seen) warp_wait(p, barp(BAR_PVDONE0 + (tau & 1)), ((tau >> 1) - 1) & 1, abort_flag);
            pv_seen = false;
            if (st == 0 && (tau == 2 || tau == 3)) DSA_TRACE_AT(p, 75 + 8 * (tau - 2));
            const uint32_t pb = sbase + kOffP + (tau & 1) * 2 * kPTermBytes;
#pragma unroll
            for (int c = 0; c < kScores / 16; ++c) {
                st_shared_v4(pb + p_off + c * 1024, hw[4 * c], hw[4 * c + 1], hw[4 * c + 2], hw[4 * c + 3]);
                st_shared_v4(pb + kPTermBytes + p_off + c * 1024, lw[4 * c], lw[4 * c + 1], lw[4 * c + 2], lw[4 * c + 3]);
            }
            fence_proxy_async_smem();
            if (resc[0] || resc[1]) {
                // O^T columns are heads: this warp rescales its lanes of chunks 2*half and
                // 2*half + 1 once the P.V before this tile is done. Doing it after the P
                // write lets that P.V run while this tile's probabilities are formed; this
                // tile's P.V waits for the rescale through the P-full barrier below.
                warp_wait(p, barp(BAR_PVDONE0 + ((tau - 1) & 1)), ((tau - 1) >> 1) & 1, abort_flag);
                pv_seen = true;  // the next tile's P buffer is free
                tc_fence_after();
                // Both dim chunks of a 32-head block are loaded together (one load latency
                // per block instead of one per chunk) and share the block's 32 factors.
#pragma unroll 1
                for (int hh = 0; hh < 2; ++hh) {
                    if (!resc[hh]) continue;
                    const uint32_t ta = tmem + lane_base + kTmemO + 2 * half * 64 + hh * 32;
                    uint32_t o0[32], o1[32];
                    tmem_ld_2x32(ta, ta + 64, o0, o1);
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const float f = alpha_t[hh * 32 + k];
                        o0[k] = __float_as_uint(__uint_as_float(o0[k]) * f);
                        o1[k] = __float_as_uint(__uint_as_float(o1[k]) * f);
                    }
                    tmem_st_x32(ta, o0);
                    tmem_st_x32(ta + 64, o1);
                }
                tmem_wait_st();
            }
            if (st == 0 && (tau == 2 || tau == 3)) DSA_TRACE_AT(p, 76 + 8 * (tau - 2));
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(barp(BAR_PFULL0 + (tau & 1)));
            if (st == 0 && tau < 8) DSA_TRACE_AT(p, 32 + tau);
        }

        // The next unit's query operand goes into TMEM now, while this unit's last P.V
        // runs (this unit's last QK completed QEMPTY phase qseg), so that the next unit's
        // first QK runs during the epilogue below.
        if (i + 1 < nseg && tl_next.n > 0) {
            warp_wait(p, barp(BAR_QEMPTY), qseg & 1, abort_flag);
            load_q(s_next.unit);
            q_loaded = true;
        }

        // ---- epilogue ----
        warp_wait(p, barp(BAR_PVDONE0 + ((tau - 1) & 1)), ((tau - 1) >> 1) & 1, abort_flag);
        pv_seen = true;
        if (st == 0 && i == 0) DSA_TRACE_AT(p, 17);
        tc_fence_after();
        const float lpair = l_part + __shfl_xor_sync(0xffffffffu, l_part, 1);
        if (term == 0) l_s[half * kHeadsPerCta + hq] = lpair;
        named_bar_sync<kBarSoftmax, kSoftmaxThreads>();
        const bool whole = s.part < 0;
        if (st == 0 && i == 0) DSA_TRACE_AT(p, 12);
        if (term == 0 && half == 0) {
            const float l = l_s[hq] + l_s[kHeadsPerCta + hq];
            f_s[hq] = (whole ? p.v_scale : 1.0f) / l;
            if (!whole) p.part_lse[s.part * kHeadsPerCta + hq] = m_ref + __log2f(l);
        }
        named_bar_sync<kBarSoftmax, kSoftmaxThreads>();
        if (st == 0 && i == 0) DSA_TRACE_AT(p, 13);
#pragma unroll 1
        for (int mc2 = 0; mc2 < 2; ++mc2) {
            const int mc = 2 * half + mc2;
            const int dim0 = mc * 128 + q4 * 32;
            // All 64 head columns of this lane's dim in one load and one wait.
            uint32_t v64[64];
            tmem_ld_x64(tmem + lane_base + kTmemO + mc * 64, v64);
            if (st == 0 && i == 0 && mc2 == 0) DSA_TRACE_AT(p, 14);
            if (whole) {
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    float o[32], f[32];
#pragma unroll
                    for (int k = 0; k < 32; k += 4) {
                        const float4 f4 = *reinterpret_cast<const float4*>(f_s + hh * 32 + k);
                        f[k] = f4.x;
                        f[k + 1] = f4.y;
                        f[k + 2] = f4.z;
                        f[k + 3] = f4.w;
                    }
#pragma unroll
                    for (int k = 0; k < 32; ++k) o[k] = __uint_as_float(v64[hh * 32 + k]);
                    __nv_bfloat16* rows = reinterpret_cast<__nv_bfloat16*>(p.out) + head0 * kLatent;
                    store_block(rows, hh * 32, hvalid, dim0, o, f, stage, lane);
                }
            } else {
                // A partial is [16 blocks of 32 dims][8 head groups][32 dims][8 heads] f16:
                // this lane's dim holds all 64 heads, and each store instruction of the warp
                // writes one head group of its 32 dims, 512 contiguous bytes, straight from
                // registers (dim0 is a multiple of 32: the warp's dims are one dim block).
                __half* part = reinterpret_cast<__half*>(p.part_o) + static_cast<int64_t>(s.part) * kHeadsPerCta * kLatent;
#pragma unroll
                for (int k = 0; k < kHeadsPerCta; k += 8) {
                    const float4 fa = *reinterpret_cast<const float4*>(f_s + k);
                    const float4 fb = *reinterpret_cast<const float4*>(f_s + k + 4);
                    const __half2 h0 = __floats2half2_rn(__uint_as_float(v64[k]) * fa.x, __uint_as_float(v64[k + 1]) * fa.y);
                    const __half2 h1 = __floats2half2_rn(__uint_as_float(v64[k + 2]) * fa.z, __uint_as_float(v64[k + 3]) * fa.w);
                    const __half2 h2 = __floats2half2_rn(__uint_as_float(v64[k + 4]) * fb.x, __uint_as_float(v64[k + 5]) * fb.y);
                    const __half2 h3 = __floats2half2_rn(__uint_as_float(v64[k + 6]) * fb.z, __uint_as_float(v64[k + 7]) * fb.w);
                    *reinterpret_cast<uint4*>(part + ((static_cast<int64_t>(dim0 / 32) * 8 + k / 8) * 32 + lane) * 8) =
                        make_uint4(*reinterpret_cast<const uint32_t*>(&h0), *reinterpret_cast<const uint32_t*>(&h1),
                                   *reinterpret_cast<const uint32_t*>(&h2), *reinterpret_cast<const uint32_t*>(&h3));
                }
            }
        }
        if (st == 0 && i == 0) DSA_TRACE_AT(p, 15);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(barp(BAR_OEMPTY));
        if (st == 0 && i == 0) DSA_TRACE_AT(p, 18);
        // The staging area is the P buffer and l_s / f_s are reused: the next unit starts
        // only after every softmax warp is done here.
        named_bar_sync<kBarSoftmax, kSoftmaxThreads>();
        ++qseg;
    }
    if (st == 0) DSA_TRACE_AT(p, 19);
}

// kTma: gather by tensor map (warp 0) or by per-thread copies (warps 0-3). The two are
// separate kernels so that each carries only its own gather code (the warps of one CTA
// run different code at once and share the SM's instruction cache) and the per-thread
// copy kernel takes no tensor maps.
template <bool kTma>
__device__ __forceinline__ void decode_body(const DecodeParams& p, const CUtensorMap* kmap, const CUtensorMap* vmap) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
    if (tid == 0) DSA_TRACE_AT(p, 0);

    if (tid == 0) {
        const uint32_t b = sbase + kOffBars;
        for (int e = 0; e < kSlotsKV; ++e) {
            // tensor-map gather: one arrive.expect_tx per tile; per-thread copies: one
            // copy-completion arrival per gather lane
            mbar_init(b + 8 * (BAR_FULL0 + e), kTma ? 1 : 32 * kProducerWarps);
            mbar_init(b + 8 * (BAR_EMPTY0 + e), 1);
        }
        for (int k = 0; k < kSBufs; ++k) {
            mbar_init(b + 8 * (BAR_SFULL0 + k), 1);
            mbar_init(b + 8 * (BAR_SEMPTY0 + k), kSoftmaxWarps);
        }
        for (int k = 0; k < 2; ++k) {
            mbar_init(b + 8 * (BAR_PFULL0 + k), kSoftmaxWarps);
            mbar_init(b + 8 * (BAR_PVDONE0 + k), 1);
        }
        mbar_init(b + 8 * BAR_QFULL, kSoftmaxWarps);
        mbar_init(b + 8 * BAR_QEMPTY, 1);
        mbar_init(b + 8 * BAR_OEMPTY, kSoftmaxWarps);
        mbar_init(b + 8 * BAR_DRAIN, 1);
        mbar_init(b + 8 * BAR_DONE, kSoftmaxWarps);
        *abort_flag = 0;
        fence_mbar_init();
        if (kTma) {
            prefetch_tmap(kmap);
            if (!p.kv_same) prefetch_tmap(vmap);
        }
    }
    if (warp == kMmaWarp) {
        tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);
    // The partition is arithmetic on the launch parameters (64-bit divisions): the first
    // segment is worked out here, overlapping the prologue, and pinned before the wait.
    int64_t first_unit;
    const int nseg = cta_segments(p.part, blockIdx.x, &first_unit);
    const Segment seg0 = cta_segment(p.part, blockIdx.x, 0);
    asm volatile("" ::"r"(nseg), "r"(seg0.unit), "r"(seg0.row), "r"(seg0.group), "l"(seg0.s0), "l"(seg0.s1),
                 "r"(seg0.part));
    // Everything above overlaps the prologue; its results are read only after this.
    griddep_wait();
    if (tid == 0) DSA_TRACE_AT(p, 1);
    // Long decodes let the next kernel on the stream launch once every CTA has passed here
    // (it waits for this grid's completion before reading its results); short ones at the end.
    if (p.early_dependents) griddep_launch_dependents();

    if (warp < kProducerWarps) {
        if constexpr (!kTma)
            run_producer(p, sbase, abort_flag, nseg, seg0);
        else if (warp == 0)
            run_producer_tma(p, kmap, vmap, sbase, abort_flag, nseg, seg0);
    } else if (warp == kMmaWarp) {
        run_mma(p, sbase, tmem, abort_flag, nseg, seg0);
        // Wait (bounded, regardless of abort) until every issued MMA has completed and the
        // softmax warps have finished reading TMEM.
        const uint32_t db = sbase + kOffBars + 8 * BAR_DRAIN;
        tc_commit_el(db, elect_one());
        uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(db, 0) && globaltimer_ns() - t0 < kDrainLimitNs) {
        }
        DSA_TRACE_AT(p, 11);
        const uint32_t done = sbase + kOffBars + 8 * BAR_DONE;
        t0 = globaltimer_ns();
        while (!mbar_try_wait(done, 0) && globaltimer_ns() - t0 < kDrainLimitNs) {
        }
        __syncwarp();
    } else {
        run_softmax(p, smem, sbase, tmem, abort_flag, nseg, seg0);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sbase + kOffBars + 8 * BAR_DONE);
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) DSA_TRACE_AT(p, 20);
    if (!p.early_dependents) griddep_launch_dependents();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeParams p) {
    decode_body<false>(p, nullptr, nullptr);
}

__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel_tma(const DecodeParams p, const __grid_constant__ CUtensorMap kmap,
                      const __grid_constant__ CUtensorMap vmap) {
    decode_body<true>(p, &kmap, &vmap);
}

}  // namespace DSA_CAT(tile, DSA_TILE)

using namespace DSA_CAT(tile, DSA_TILE);

template <typename K>
cudaError_t setup_instance(K kernel) {
    // The register cap above must leave room for all kThreads threads of the block.
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, kernel);
    if (e != cudaSuccess) return e;
    if (attr.maxThreadsPerBlock < kThreads) return cudaErrorInvalidConfiguration;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

cudaError_t DSA_CAT(decode_kernel_setup_, DSA_TILE)() {
    const cudaError_t e = setup_instance(decode_kernel);
    return e != cudaSuccess ? e : setup_instance(decode_kernel_tma);
}

cudaError_t DSA_CAT(launch_decode_, DSA_TILE)(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                                              cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.part.ctas);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return p.use_tma ? cudaLaunchKernelEx(&cfg, decode_kernel_tma, p, kmap, vmap)
                     : cudaLaunchKernelEx(&cfg, decode_kernel, p);
}

}  // namespace dsa
