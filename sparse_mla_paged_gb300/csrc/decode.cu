// The selected-index NoPE MLA paged decode kernel (attend.rs, decode_attention).
//
// One CTA per SM, persistent over a static slot-space partition (see common.cuh). Work
// unit = (decode row, group of 64 query heads). For each tile of 128 resolved tokens:
//
//   gather   warps 0-3   cp.async 16-byte copies of each token's 512-byte E4M3 latent row
//                        (byte offsets resolved by the prologue; the next tile's offsets are
//                        loaded while waiting for a free slot) into a 2-slot ring, written in
//                        the 128-byte-swizzled K-major operand layout. (Per 512-byte row,
//                        16-byte copies from 32 lanes sustain a higher gather rate on this
//                        part than TMA tile::gather4 loads, whose per-instruction cost
//                        limits an SM to about 17 GB/s.)
//   QK^T     warp 4      tcgen05.mma kind::f8f6f4, M = 128 tokens, N = 128 (64 heads x
//                        {hi, lo} query terms), K = 512: S^T -> TMEM (double buffered).
//   softmax  warps 5-12  two warps per TMEM lane quarter, each thread one token and 32
//                        heads: s = hi + lo, per-head scale, column max over the 128 tokens
//                        (redux.sync.max per warp + a 4-way exchange), online rescale,
//                        P' = 256*exp2(x - m) stored as two E4M3 terms (hi = top 4 bits,
//                        lo = rest); the row sums stay per thread until the epilogue,
//                        the running maxima in shared memory.
//   P.V      warp 4      O^T[512 dims x 64 heads] += V^T * P'^T in TMEM: the same ring slot
//                        read as an MN-major operand (K and V are the same bytes).
//   epilogue warps 5-12  O / (256 l) * v_scale -> BF16 output, or (O/l, lse) partials,
//                        transposed per warp through shared memory into 16-byte stores.
//
// The contraction is exact in its inputs: keys and values are the cached E4M3 codes
// themselves (k_scale and v_scale are applied outside the MMA), queries are split into
// two E4M3 terms that reproduce the BF16 value (see prologue.cu), probabilities into two
// terms that carry about 8 significant bits. Accumulation is FP32 in TMEM.
//
// Shared memory 212 KB, TMEM 512 columns: O^T at 0..255 (chunk c of 128 dims at 64c),
// S^T buffers at 256 and 384. Every wait is bounded (see ptx.cuh); on a timeout the CTA
// records DSA_ERR_TIMEOUT, skips the remaining waits and finishes.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kProducerWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kSoftmaxWarp0 = 5;
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = (kSoftmaxWarp0 + kSoftmaxWarps) * 32;  // 416
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kSoftmaxThreads = kSoftmaxWarps * 32;

// Named barriers (0 is __syncthreads): one per head half of the softmax warps, one for
// all softmax warps.
constexpr int kBarHalf0 = 1;
constexpr int kBarSoftmax = 3;

constexpr int kOffRing = 0;
constexpr int kOffQ = 2 * kKvTileBytes;
constexpr int kOffP = kOffQ + kQImageBytes;              // P' hi (8 KB) then lo (8 KB)
constexpr int kPTermBytes = kTileTokens * kHeadsPerCta;  // 8 KB
constexpr int kOffRed = kOffP + 2 * kPTermBytes;         // float [2 parity][4 quarters][64 heads]
constexpr int kOffCs = kOffRed + 2 * 4 * kHeadsPerCta * 4;
constexpr int kOffM = kOffCs + kHeadsPerCta * 4;         // float [2 parity][64 heads] running max
constexpr int kOffBars = kOffM + 2 * kHeadsPerCta * 4;
enum {
    BAR_FULL0, BAR_FULL1, BAR_EMPTY0, BAR_EMPTY1, BAR_SFULL0, BAR_SFULL1, BAR_SEMPTY0, BAR_SEMPTY1,
    BAR_PFULL, BAR_PVDONE, BAR_QFULL, BAR_QEMPTY, BAR_OEMPTY, BAR_DRAIN, BAR_DONE, kNumBars
};
constexpr int kOffTmemSlot = kOffBars + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kSmemUsed = kOffAbort + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for the 1024-byte alignment

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;

constexpr float kNegInf = -__builtin_huge_valf();

// Optional per-CTA timeline (clock64 values), compiled in only with -DDSA_TRACE: slot i of
// CTA c is trace[c*64 + i].
#ifdef DSA_TRACE
#define DSA_TRACE_AT(p, i)                                                                             \
    do {                                                                                               \
        if ((p).trace && (i) < 64) (p).trace[static_cast<int64_t>(blockIdx.x) * 64 + (i)] = clock64(); \
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

__device__ __forceinline__ Tiles segment_tokens(const DecodeParams& p, const Segment& s) {
    const int64_t U = p.cnt[s.row];
    const int64_t W = p.part.width;
    Tiles t;
    t.t0 = s.s0 * U / W;
    const int64_t t1 = s.s1 * U / W;
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
    if (!mbar_wait(bar, parity, abort_flag)) fail(p, abort_flag, kStatusTimeout);
    __syncwarp();
}

// Barrier over the four softmax warps that share a head half.
__device__ __forceinline__ void half_bar_sync(int hh) {
    if (hh == 0)
        named_bar_sync<kBarHalf0, 128>();
    else
        named_bar_sync<kBarHalf0 + 1, 128>();
}

__device__ __forceinline__ float redux_max(float x) {
    float r;
    asm volatile("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(x));
    return r;
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    return f32x2_to_e4m3x2(a, b) | (f32x2_to_e4m3x2(c, d) << 16);
}

// Keeps sign, exponent and the top three mantissa bits (an E4M3-representable value for
// magnitudes in E4M3's normal range).
__device__ __forceinline__ float hi_part(float x) {
    return __uint_as_float(__float_as_uint(x) & 0xFFF00000u);
}

__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------------------------
// gather warps
// ------------------------------------------------------------------------------------
__device__ void run_producer(const DecodeParams& p, uint32_t sbase, volatile int* abort_flag, int nseg) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nslot = p.kv_same ? 2 : 1;
    const int64_t W = p.part.width;
    const uint32_t chunk = (lane >> 3) * kKBlockBytes;  // K-block of this lane's 16-byte chunk
    uint32_t tau = 0;
    int qseg = 0;
    for (int i = 0; i < nseg; ++i) {
        const Segment s = cta_segment(p.part, blockIdx.x, i);
        const Tiles tl = segment_tokens(p, s);
        if (tl.n <= 0) continue;
        if (tid == 0) {
            if (qseg > 0 && !mbar_wait(sbase + kOffBars + 8 * BAR_QEMPTY, (qseg - 1) & 1, abort_flag))
                fail(p, abort_flag, kStatusTimeout);
            const uint32_t qbar = sbase + kOffBars + 8 * BAR_QFULL;
            mbar_arrive_expect_tx(qbar, kQImageBytes);
            const uint8_t* src = p.qimg + static_cast<int64_t>(s.unit) * kQImageBytes;
#pragma unroll
            for (int k = 0; k < 4; ++k) bulk_g2s(sbase + kOffQ + k * 16384, src + k * 16384, 16384, qbar);
            if (qseg == 0) DSA_TRACE_AT(p, 3);
        }
        __syncwarp();
        ++qseg;
        const long long* offs = p.offs + static_cast<int64_t>(s.row) * W + tl.t0;
        const int tok = warp * 32 + lane;  // this lane's token of each tile
        long long nx = tok < tl.n ? offs[tok] : -1;
        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            const long long o_mine = nx;
            const int32_t next = (t + 1) * kTileTokens + tok;
            if (t + 1 < tl.ntiles) nx = next < tl.n ? offs[next] : -1;  // before the slot wait
            if (t * kTileTokens + tok < tl.n && o_mine < 0) atomicCAS(p.status, 0, kStatusBounds);
            const int slot = static_cast<int>(tau % nslot);
            const uint32_t use = tau / nslot;
            if (tau >= static_cast<uint32_t>(nslot))
                warp_wait(p, sbase + kOffBars + 8 * (BAR_EMPTY0 + slot), (use - 1) & 1, abort_flag);
            if (tid == 0 && tau < 8) DSA_TRACE_AT(p, 40 + tau);
            const uint32_t kdst = sbase + kOffRing + slot * kKvTileBytes;
            const uint32_t vdst = p.kv_same ? kdst : sbase + kOffRing + kKvTileBytes;
#pragma unroll 4
            for (int j = 0; j < 32; ++j) {
                const long long o = __shfl_sync(0xffffffffu, o_mine, j);
                const int tk = warp * 32 + j;
                const uint32_t d = chunk + tk * 128 + (((lane & 7) ^ (tk & 7)) << 4);
                if (o >= 0) {
                    cp_async_16(kdst + d, p.k_cache + o + lane * 16);
                    if (!p.kv_same) cp_async_16(vdst + d, p.v_cache + o + lane * 16);
                } else {
                    st_shared_v4(kdst + d, 0u, 0u, 0u, 0u);
                    if (!p.kv_same) st_shared_v4(vdst + d, 0u, 0u, 0u, 0u);
                }
            }
            const uint32_t fb = sbase + kOffBars + 8 * (BAR_FULL0 + slot);
            cp_async_arrive_noinc(fb);
            mbar_arrive(fb);
            if (tid == 0 && tau == 0) DSA_TRACE_AT(p, 4);
            if (tid == 0 && tau < 8) DSA_TRACE_AT(p, 48 + tau);
        }
    }
    if (tid == 0) DSA_TRACE_AT(p, 5);
    cp_async_wait_all();
}

// ------------------------------------------------------------------------------------
// MMA warp (one thread issues)
// ------------------------------------------------------------------------------------
__device__ void run_mma(const DecodeParams& p, uint32_t sbase, uint32_t tmem, volatile int* abort_flag, int nseg) {
    const int nslot = p.kv_same ? 2 : 1;
    const uint32_t idq = idesc_e4m3(128, 128, false, false);
    const uint32_t idp = idesc_e4m3(128, 64, true, true);
    auto barp = [&](int b) { return sbase + kOffBars + 8 * b; };
    uint32_t tau = 0;
    int qseg = 0;

    auto issue_pv = [&](uint32_t tp, bool first) {
        if (!mbar_wait(barp(BAR_PFULL), tp & 1, abort_flag)) fail(p, abort_flag, kStatusTimeout);
        if (tp == 0) DSA_TRACE_AT(p, 9);
        if (first && qseg > 0 && !mbar_wait(barp(BAR_OEMPTY), (qseg - 1) & 1, abort_flag))
            fail(p, abort_flag, kStatusTimeout);
        tc_fence_after();
        const int slot = static_cast<int>(tp % nslot);
        const uint32_t vbase = sbase + kOffRing + (p.kv_same ? slot * kKvTileBytes : kKvTileBytes);
#pragma unroll
        for (int mc = 0; mc < 4; ++mc) {
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                const uint64_t a = smem_desc(vbase + mc * kKBlockBytes + ks * 4096, kKBlockBytes, 1024, kSwizzle128B);
                const uint64_t bh = smem_desc(sbase + kOffP + ks * 512, 128, 2048, kSwizzleNone);
                const uint64_t bl = smem_desc(sbase + kOffP + kPTermBytes + ks * 512, 128, 2048, kSwizzleNone);
                mma_e4m3(tmem + kTmemO + mc * 64, a, bh, idp, (first && ks == 0) ? 0u : 1u);
                mma_e4m3(tmem + kTmemO + mc * 64, a, bl, idp, 1u);
            }
        }
        tc_commit(barp(BAR_PVDONE));
        tc_commit(barp(BAR_EMPTY0 + slot));
    };

    auto issue_qk = [&](uint32_t tq) {
        const int slot = static_cast<int>(tq % nslot);
        const int sb = tq & 1;
        fence_proxy_async_smem();
        tc_fence_after();
        const uint32_t kbase = sbase + kOffRing + slot * kKvTileBytes;
#pragma unroll
        for (int ks = 0; ks < 16; ++ks) {
            const uint32_t off = (ks >> 2) * kKBlockBytes + (ks & 3) * 32;
            mma_e4m3(tmem + kTmemS + sb * 128, smem_desc(kbase + off, 16, 1024, kSwizzle128B),
                     smem_desc(sbase + kOffQ + off, 16, 1024, kSwizzle128B), idq, ks > 0 ? 1u : 0u);
        }
        tc_commit(barp(BAR_SFULL0 + sb));
        if (tq == 0) DSA_TRACE_AT(p, 8);
    };
    // Phase the QK of tile tq may start: its ring slot is full and its S buffer is free.
    auto qk_ready = [&](uint32_t tq) {
        const int slot = static_cast<int>(tq % nslot);
        const bool full = mbar_try_wait(barp(BAR_FULL0 + slot), (tq / nslot) & 1);
        return full && (tq < 2 || mbar_try_wait(barp(BAR_SEMPTY0 + (tq & 1)), ((tq >> 1) - 1) & 1));
    };

    for (int i = 0; i < nseg; ++i) {
        const Segment s = cta_segment(p.part, blockIdx.x, i);
        const Tiles tl = segment_tokens(p, s);
        if (tl.n <= 0) continue;
        if (!mbar_wait(barp(BAR_QFULL), qseg & 1, abort_flag)) fail(p, abort_flag, kStatusTimeout);
        if (qseg == 0) DSA_TRACE_AT(p, 6);
        const uint32_t tau0 = tau;
        // QK(t) and PV(t-1) are independent: issue whichever becomes ready first (with one
        // ring slot, QK(t) needs the slot PV(t-1) frees, so PV(t-1) goes first).
        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            bool qk_done = false, pv_done = (t == 0);
            if (nslot == 1 && !pv_done) {
                issue_pv(tau - 1, tau - 1 == tau0);
                pv_done = true;
            }
            const uint64_t t_start = globaltimer_ns();
            while (!qk_done || !pv_done) {
                if (!qk_done && qk_ready(tau)) {
                    if (tau < 8) DSA_TRACE_AT(p, 56 + tau);
                    issue_qk(tau);
                    if (t == tl.ntiles - 1) tc_commit(barp(BAR_QEMPTY));
                    qk_done = true;
                }
                if (!pv_done && mbar_try_wait(barp(BAR_PFULL), (tau - 1) & 1)) {
                    issue_pv(tau - 1, tau - 1 == tau0);
                    pv_done = true;
                }
                if ((!qk_done || !pv_done) && (*abort_flag || globaltimer_ns() - t_start > kWaitLimitNs)) {
                    fail(p, abort_flag, kStatusTimeout);
                    break;
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

// Writes a warp's 32 dims x 16 heads block (dims on lanes, v[k] = head h0+k, scaled by
// f[k]) to row-major global rows (row stride kLatent elements) through a 2 KB per-warp
// staging area, with 16-byte stores. T is bf16 (output) or f16 (partials). Heads at or
// beyond hvalid are not written.
template <typename T>
__device__ __forceinline__ void store_block(T* rows, int h0, int hvalid, int dim0, const float* v, const float* f,
                                            uint8_t* stage, int lane) {
    constexpr int kPer16 = 16 / static_cast<int>(sizeof(T));  // elements per 16-byte store
    constexpr int kLanesPerRow = 32 / kPer16;                 // lanes covering one head's 32 dims
    constexpr int kRowsPerPass = 32 / kLanesPerRow;           // heads per warp-wide store
    T* stg = reinterpret_cast<T*>(stage);                     // [16 heads][32 dims]
#pragma unroll
    for (int k = 0; k < 16; ++k) {
        const float x = v[k] * f[k];
        if constexpr (std::is_same<T, __half>::value) {
            stg[k * 32 + lane] = __float2half_rn(x);
        } else {
            stg[k * 32 + lane] = __float2bfloat16_rn(x);
        }
    }
    __syncwarp();
#pragma unroll
    for (int pass = 0; pass < 16 / kRowsPerPass; ++pass) {
        const int hk = pass * kRowsPerPass + lane / kLanesPerRow;
        const int c = (lane % kLanesPerRow) * kPer16;
        const uint4 val = *reinterpret_cast<const uint4*>(stg + hk * 32 + c);
        if (h0 + hk < hvalid)
            *reinterpret_cast<uint4*>(rows + static_cast<int64_t>(h0 + hk) * kLatent + dim0 + c) = val;
    }
    __syncwarp();
}

__device__ void run_softmax(const DecodeParams& p, uint8_t* smem, uint32_t sbase, uint32_t tmem,
                            volatile int* abort_flag, int nseg) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int sw = warp - kSoftmaxWarp0;      // 0..7
    const int q4 = warp & 3;                  // TMEM lane quarter of this warp
    const int hh = sw >> 2;                   // head half: heads 32*hh .. 32*hh+31
    const int h0 = hh * 32;
    const int token = q4 * 32 + lane;         // token row of the tile = TMEM lane
    const int st = sw * 32 + lane;            // 0..255
    float* red = reinterpret_cast<float*>(smem + kOffRed);   // [2][4][64]
    float* c_s = reinterpret_cast<float*>(smem + kOffCs);
    float* m_s = reinterpret_cast<float*>(smem + kOffM);     // [2][64]
    uint8_t* stage = smem + kOffP + sw * 2048;               // epilogue staging (2 KB per warp)
    auto barp = [&](int b) { return sbase + kOffBars + 8 * b; };
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    uint32_t tau = 0;

    for (int i = 0; i < nseg; ++i) {
        const Segment s = cta_segment(p.part, blockIdx.x, i);
        const Tiles tl = segment_tokens(p, s);
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
        if (st < kHeadsPerCta) c_s[st] = p.qscale[static_cast<int64_t>(s.unit) * kHeadsPerCta + st];
        named_bar_sync<kBarSoftmax, kSoftmaxThreads>();
        if (st == 0 && i == 0) DSA_TRACE_AT(p, 12);

        float l_part[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) l_part[k] = 0.0f;
        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            const int sb = tau & 1;
            warp_wait(p, barp(BAR_SFULL0 + sb), (tau >> 1) & 1, abort_flag);
            if (st == 0 && tau == 0) DSA_TRACE_AT(p, 13);
            if (st == 0 && tau < 8) DSA_TRACE_AT(p, 24 + tau);
            tc_fence_after();
            float x[32];
            {
                const uint32_t ta = tmem + lane_base + kTmemS + sb * 128 + h0;
                uint32_t a[32];
                tmem_ld_x32(ta, a);        // hi-term scores of heads h0..h0+31
#pragma unroll
                for (int k = 0; k < 32; ++k) x[k] = __uint_as_float(a[k]);
#pragma unroll
                for (int half = 0; half < 2; ++half) {  // lo-term scores, 16 columns at a time
                    uint32_t b[16];
                    tmem_ld_x16(ta + 64 + half * 16, b);
#pragma unroll
                    for (int k = 0; k < 16; ++k) x[half * 16 + k] += __uint_as_float(b[k]);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(barp(BAR_SEMPTY0 + sb));

            const bool valid = t * kTileTokens + token < tl.n;
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
                const float4 c = *reinterpret_cast<const float4*>(c_s + h0 + k);
                x[k] = valid ? x[k] * c.x : kNegInf;
                x[k + 1] = valid ? x[k + 1] * c.y : kNegInf;
                x[k + 2] = valid ? x[k + 2] * c.z : kNegInf;
                x[k + 3] = valid ? x[k + 3] * c.w : kNegInf;
            }
            // Column max over this warp's 32 tokens, then over the 4 lane quarters.
            float* rbuf = red + (tau & 1) * (4 * kHeadsPerCta);
            {
                float mine = kNegInf;
#pragma unroll
                for (int k = 0; k < 32; ++k) {
                    const float r = redux_max(x[k]);
                    mine = (lane == k) ? r : mine;
                }
                rbuf[q4 * kHeadsPerCta + h0 + lane] = mine;
            }
            half_bar_sync(hh);
            if (st == 0 && tau == 0) DSA_TRACE_AT(p, 14);
            // Lane k owns head h0+k: tile max over the 4 quarters, running max (parity (t-1)&1
            // in m_s, -inf before the first tile), new max and rescale factor alpha. The new max
            // goes to parity t&1 (all four warps of the half write the same values), read back
            // only after the next half barrier. Every lane then takes head k's values by
            // shuffle as it uses them.
            const int hk = h0 + lane;
            const float mt = fmaxf(fmaxf(rbuf[hk], rbuf[kHeadsPerCta + hk]),
                                   fmaxf(rbuf[2 * kHeadsPerCta + hk], rbuf[3 * kHeadsPerCta + hk]));
            const float mo = t > 0 ? m_s[((t + 1) & 1) * kHeadsPerCta + hk] : kNegInf;
            const float mn = fmaxf(mo, mt);
            const float a_mine = (mo == kNegInf) ? 0.0f : ex2_approx(mo - mn);
            m_s[(t & 1) * kHeadsPerCta + hk] = mn;
            const uint32_t grew = __ballot_sync(0xffffffffu, a_mine < 1.0f);
#pragma unroll
            for (int k = 0; k < 32; ++k) {
                const float m_k = __shfl_sync(0xffffffffu, mn, k);
                const float a_k = __shfl_sync(0xffffffffu, a_mine, k);
                const float pr = ex2_approx(x[k] - m_k);
                l_part[k] = l_part[k] * a_k + pr;
                x[k] = pr;
            }
            // P and O may only change once the previous P.V has finished reading them.
            if (t > 0) warp_wait(p, barp(BAR_PVDONE), (tau - 1) & 1, abort_flag);
#pragma unroll
            for (int hc = 0; hc < 2; ++hc) {
                uint32_t hw[4], lw[4];
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    float ph[4], pl[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float pp = x[hc * 16 + k * 4 + e] * kPScale;
                        ph[e] = hi_part(pp);
                        pl[e] = pp - ph[e];
                    }
                    hw[k] = pack_e4m3x4(ph[0], ph[1], ph[2], ph[3]);
                    lw[k] = pack_e4m3x4(pl[0], pl[1], pl[2], pl[3]);
                }
                const uint32_t off = (2 * hh + hc) * 2048 + token * 16;
                st_shared_v4(sbase + kOffP + off, hw[0], hw[1], hw[2], hw[3]);
                st_shared_v4(sbase + kOffP + kPTermBytes + off, lw[0], lw[1], lw[2], lw[3]);
            }
            if (t > 0 && grew != 0u) {
                // Rescale this half's O^T columns by alpha (1 for heads whose max held).
                float al[32];
#pragma unroll
                for (int k = 0; k < 32; ++k) al[k] = __shfl_sync(0xffffffffu, a_mine, k);
                tc_fence_after();
#pragma unroll 1
                for (int mc = 0; mc < 4; ++mc) {
                    const uint32_t ta = tmem + lane_base + kTmemO + mc * 64 + h0;
                    uint32_t v[32];
                    tmem_ld_x32(ta, v);
#pragma unroll
                    for (int k = 0; k < 32; ++k) v[k] = __float_as_uint(__uint_as_float(v[k]) * al[k]);
                    tmem_st_x32(ta, v);
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(barp(BAR_PFULL));
            if (st == 0 && tau == 0) DSA_TRACE_AT(p, 16);
            if (st == 0 && tau < 8) DSA_TRACE_AT(p, 32 + tau);
        }

        // ---- epilogue ----
        warp_wait(p, barp(BAR_PVDONE), (tau - 1) & 1, abort_flag);
        if (st == 0 && i == 0) DSA_TRACE_AT(p, 17);
        tc_fence_after();
        // Row sums: per head over the warp's 32 tokens (butterfly, result in every lane),
        // then over the 4 lane quarters through shared memory.
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            float v = l_part[k];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
            l_part[k] = v;
        }
        if (st == 0 && i == 0) DSA_TRACE_AT(p, 2);
        if (lane == 0) {
#pragma unroll
            for (int k = 0; k < 32; k += 4)
                *reinterpret_cast<float4*>(red + q4 * kHeadsPerCta + h0 + k) =
                    make_float4(l_part[k], l_part[k + 1], l_part[k + 2], l_part[k + 3]);
        }
        half_bar_sync(hh);
        // Lane k: head h0+k's row sum, output factor and (for a partial) log-sum-exp.
        const bool whole = s.part < 0;
        float f_mine;
        {
            const int hk = h0 + lane;
            const float l = (red[hk] + red[kHeadsPerCta + hk]) + (red[2 * kHeadsPerCta + hk] + red[3 * kHeadsPerCta + hk]);
            f_mine = (whole ? p.v_scale : 1.0f) / (kPScale * l);
            if (!whole && q4 == 0)
                p.part_lse[s.part * kHeadsPerCta + hk] = m_s[((tl.ntiles - 1) & 1) * kHeadsPerCta + hk] + __log2f(l);
        }
        float f[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) f[k] = __shfl_sync(0xffffffffu, f_mine, k);
        if (st == 0 && i == 0) DSA_TRACE_AT(p, 15);
#pragma unroll 1
        for (int mc = 0; mc < 4; ++mc) {
            uint32_t v[32];
            tmem_ld_x32(tmem + lane_base + kTmemO + mc * 64 + h0, v);
            float o[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] = __uint_as_float(v[k]);
            const int dim0 = mc * 128 + q4 * 32;
            if (whole) {
                __nv_bfloat16* rows = reinterpret_cast<__nv_bfloat16*>(p.out) + head0 * kLatent;
                store_block(rows, h0, hvalid, dim0, o, f, stage, lane);
                store_block(rows, h0 + 16, hvalid, dim0, o + 16, f + 16, stage, lane);
            } else {
                __half* rows = reinterpret_cast<__half*>(p.part_o) + static_cast<int64_t>(s.part) * kHeadsPerCta * kLatent;
                store_block(rows, h0, kHeadsPerCta, dim0, o, f, stage, lane);
                store_block(rows, h0 + 16, kHeadsPerCta, dim0, o + 16, f + 16, stage, lane);
            }
            if (st == 0 && i == 0 && mc == 0) DSA_TRACE_AT(p, 23);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(barp(BAR_OEMPTY));
        if (st == 0 && i == 0) DSA_TRACE_AT(p, 18);
        // The staging area is the P buffer, and c_s / red are reused: the next segment
        // starts only after every softmax warp is done here.
        named_bar_sync<kBarSoftmax, kSoftmaxThreads>();
    }
    if (st == 0) DSA_TRACE_AT(p, 19);
}

__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);
    if (tid == 0) DSA_TRACE_AT(p, 0);

    if (tid == 0) {
        const uint32_t b = sbase + kOffBars;
        // one cp.async arrival and one plain arrival per gather thread
        mbar_init(b + 8 * BAR_FULL0, 2 * kProducerThreads);
        mbar_init(b + 8 * BAR_FULL1, 2 * kProducerThreads);
        mbar_init(b + 8 * BAR_EMPTY0, 1);
        mbar_init(b + 8 * BAR_EMPTY1, 1);
        mbar_init(b + 8 * BAR_SFULL0, 1);
        mbar_init(b + 8 * BAR_SFULL1, 1);
        mbar_init(b + 8 * BAR_SEMPTY0, kSoftmaxWarps);
        mbar_init(b + 8 * BAR_SEMPTY1, kSoftmaxWarps);
        mbar_init(b + 8 * BAR_PFULL, kSoftmaxWarps);
        mbar_init(b + 8 * BAR_PVDONE, 1);
        mbar_init(b + 8 * BAR_QFULL, 1);
        mbar_init(b + 8 * BAR_QEMPTY, 1);
        mbar_init(b + 8 * BAR_OEMPTY, kSoftmaxWarps);
        mbar_init(b + 8 * BAR_DRAIN, 1);
        mbar_init(b + 8 * BAR_DONE, kSoftmaxWarps);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(sbase + kOffTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffTmemSlot);
    // Everything above overlaps the prologue; its results are read only after this.
    griddep_wait();
    if (tid == 0) DSA_TRACE_AT(p, 1);

    int64_t first_unit;
    const int nseg = cta_segments(p.part, blockIdx.x, &first_unit);

    if (warp < kProducerWarps) {
        run_producer(p, sbase, abort_flag, nseg);
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            run_mma(p, sbase, tmem, abort_flag, nseg);
            // Wait (bounded, regardless of abort) until every issued MMA has completed and
            // the softmax warps have finished reading TMEM.
            const uint32_t db = sbase + kOffBars + 8 * BAR_DRAIN;
            tc_commit(db);
            uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(db, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
            DSA_TRACE_AT(p, 11);
            const uint32_t done = sbase + kOffBars + 8 * BAR_DONE;
            t0 = globaltimer_ns();
            while (!mbar_try_wait(done, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else {
        run_softmax(p, smem, sbase, tmem, abort_flag, nseg);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(sbase + kOffBars + 8 * BAR_DONE);
    }
    tc_fence_before();
    __syncthreads();
    if (tid == 0) DSA_TRACE_AT(p, 20);
    if (tid == kSoftmaxWarp0 * 32) DSA_TRACE_AT(p, 21);
    if (tid == kMmaWarp * 32 + 1) DSA_TRACE_AT(p, 22);
    griddep_launch_dependents();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t decode_kernel_setup() {
    cudaError_t e = cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(decode_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
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
    return cudaLaunchKernelEx(&cfg, decode_kernel, p);
}

}  // namespace dsa
