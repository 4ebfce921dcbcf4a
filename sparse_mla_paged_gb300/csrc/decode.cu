// The selected-index NoPE MLA paged decode kernel (attend.rs, decode_attention).
//
// One CTA per SM, persistent over a static slot-space partition (see common.cuh). Work
// unit = (decode row, group of 64 query heads). For each tile of 128 resolved tokens:
//
//   gather   warps 0-1   cp.async 16-byte copies of each token's 512-byte E4M3 latent row
//                        (byte offsets resolved by the prologue; the next tile's offsets
//                        are prefetched while waiting for a free slot) into a 2-slot ring,
//                        written in the 128-byte-swizzled K-major operand layout.
//   QK^T     warp 2      tcgen05.mma kind::f8f6f4, M = 128 tokens, N = 128 (64 heads x
//                        {hi, lo} query terms), K = 512: S^T -> TMEM (double buffered).
//   softmax  warps 3-10  two warps per TMEM lane quarter, each thread one token and 32
//                        heads: s = hi + lo, per-head scale, column max over the 128 tokens
//                        (redux.sync.max per warp + a 4-way exchange), online rescale,
//                        P' = 256*exp2(x - m) stored as two E4M3 terms (hi = top 4 bits,
//                        lo = rest); the row sums stay per thread until the epilogue.
//   P.V      warp 2      O^T[512 dims x 64 heads] += V^T * P'^T in TMEM: the same ring slot
//                        read as an MN-major operand (K and V are the same bytes).
//   epilogue warps 3-10  O / (256 l) * v_scale -> BF16 output, or (O/l, lse) partials,
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

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kProducerWarps = 2;
constexpr int kMmaWarp = 2;
constexpr int kSoftmaxWarp0 = 3;
constexpr int kSoftmaxWarps = 8;
constexpr int kThreads = (kSoftmaxWarp0 + kSoftmaxWarps) * 32;  // 352
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
constexpr int kOffBars = kOffCs + kHeadsPerCta * 4;
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
        // this lane's two tokens of a tile: warp*64 + lane and warp*64 + 32 + lane
        const int tok0 = warp * 64 + lane, tok1 = tok0 + 32;
        long long nx0 = tok0 < tl.n ? offs[tok0] : -1;
        long long nx1 = tok1 < tl.n ? offs[tok1] : -1;
        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            const long long o0 = nx0, o1 = nx1;
            const int32_t base = (t + 1) * kTileTokens;
            if (t + 1 < tl.ntiles) {  // prefetch the next tile's offsets before waiting
                nx0 = base + tok0 < tl.n ? offs[base + tok0] : -1;
                nx1 = base + tok1 < tl.n ? offs[base + tok1] : -1;
            }
            const bool in0 = t * kTileTokens + tok0 < tl.n, in1 = t * kTileTokens + tok1 < tl.n;
            if ((in0 && o0 < 0) || (in1 && o1 < 0)) atomicCAS(p.status, 0, kStatusBounds);
            const int slot = static_cast<int>(tau % nslot);
            const uint32_t use = tau / nslot;
            if (tau >= static_cast<uint32_t>(nslot))
                warp_wait(p, sbase + kOffBars + 8 * (BAR_EMPTY0 + slot), (use - 1) & 1, abort_flag);
            const uint32_t kdst = sbase + kOffRing + slot * kKvTileBytes;
            const uint32_t vdst = p.kv_same ? kdst : sbase + kOffRing + kKvTileBytes;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const long long mine = half ? o1 : o0;
#pragma unroll 4
                for (int j = 0; j < 32; ++j) {
                    const long long o = __shfl_sync(0xffffffffu, mine, j);
                    const int tk = warp * 64 + half * 32 + j;
                    const uint32_t d = chunk + tk * 128 + (((lane & 7) ^ (tk & 7)) << 4);
                    if (o >= 0) {
                        cp_async_16(kdst + d, p.k_cache + o + lane * 16);
                        if (!p.kv_same) cp_async_16(vdst + d, p.v_cache + o + lane * 16);
                    } else {
                        st_shared_v4(kdst + d, 0u, 0u, 0u, 0u);
                        if (!p.kv_same) st_shared_v4(vdst + d, 0u, 0u, 0u, 0u);
                    }
                }
            }
            const uint32_t fb = sbase + kOffBars + 8 * (BAR_FULL0 + slot);
            cp_async_arrive_noinc(fb);
            mbar_arrive(fb);
            if (tid == 0 && tau == 0) DSA_TRACE_AT(p, 4);
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

    for (int i = 0; i < nseg; ++i) {
        const Segment s = cta_segment(p.part, blockIdx.x, i);
        const Tiles tl = segment_tokens(p, s);
        if (tl.n <= 0) continue;
        if (!mbar_wait(barp(BAR_QFULL), qseg & 1, abort_flag)) fail(p, abort_flag, kStatusTimeout);
        if (qseg == 0) DSA_TRACE_AT(p, 6);
        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            if (nslot == 1 && t > 0) issue_pv(tau - 1, t == 1);
            const int slot = static_cast<int>(tau % nslot);
            const uint32_t use = tau / nslot;
            if (!mbar_wait(barp(BAR_FULL0 + slot), use & 1, abort_flag)) fail(p, abort_flag, kStatusTimeout);
            if (tau == 0) DSA_TRACE_AT(p, 7);
            if (tau < 8) DSA_TRACE_AT(p, 56 + tau);
            const int sb = tau & 1;
            if (tau >= 2 && !mbar_wait(barp(BAR_SEMPTY0 + sb), ((tau >> 1) - 1) & 1, abort_flag))
                fail(p, abort_flag, kStatusTimeout);
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
            if (tau == 0) DSA_TRACE_AT(p, 8);
            if (t == tl.ntiles - 1) tc_commit(barp(BAR_QEMPTY));
            if (nslot == 2 && t > 0) issue_pv(tau - 1, t == 1);
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
// staging area, with 16-byte stores. T is float (partials) or bf16 (output). Heads at or
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
        if constexpr (sizeof(T) == 4) {
            stg[k * 32 + lane] = x;
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
                float4* po = reinterpret_cast<float4*>(p.part_o + static_cast<int64_t>(s.part) * kHeadsPerCta * kLatent);
                for (int e = st; e < kHeadsPerCta * kLatent / 4; e += kSoftmaxThreads) po[e] = make_float4(0, 0, 0, 0);
                if (st < kHeadsPerCta) p.part_lse[s.part * kHeadsPerCta + st] = kNegInf;
            }
            continue;
        }
        if (st < kHeadsPerCta) c_s[st] = p.qscale[static_cast<int64_t>(s.unit) * kHeadsPerCta + st];
        named_bar_sync<kBarSoftmax, kSoftmaxThreads>();
        if (st == 0 && i == 0) DSA_TRACE_AT(p, 12);

        float m_run[32], l_part[32];
#pragma unroll
        for (int k = 0; k < 32; ++k) {
            m_run[k] = kNegInf;
            l_part[k] = 0.0f;
        }
        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            const int sb = tau & 1;
            warp_wait(p, barp(BAR_SFULL0 + sb), (tau >> 1) & 1, abort_flag);
            if (st == 0 && tau == 0) DSA_TRACE_AT(p, 13);
            if (st == 0 && tau < 16) DSA_TRACE_AT(p, 24 + tau);
            tc_fence_after();
            float x[32];
            {
                const uint32_t ta = tmem + lane_base + kTmemS + sb * 128 + h0;
                uint32_t a[32];
                tmem_ld_x32(ta, a);        // hi-term scores of heads h0..h0+31
#pragma unroll
                for (int k = 0; k < 32; ++k) x[k] = __uint_as_float(a[k]);
                tmem_ld_x32(ta + 64, a);   // lo-term scores
#pragma unroll
                for (int k = 0; k < 32; ++k) x[k] += __uint_as_float(a[k]);
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
            uint32_t grew = 0;
            float al[32];
#pragma unroll
            for (int k = 0; k < 32; k += 4) {
                const float4 r0 = *reinterpret_cast<const float4*>(rbuf + 0 * kHeadsPerCta + h0 + k);
                const float4 r1 = *reinterpret_cast<const float4*>(rbuf + 1 * kHeadsPerCta + h0 + k);
                const float4 r2 = *reinterpret_cast<const float4*>(rbuf + 2 * kHeadsPerCta + h0 + k);
                const float4 r3 = *reinterpret_cast<const float4*>(rbuf + 3 * kHeadsPerCta + h0 + k);
                const float mt[4] = {fmaxf(fmaxf(r0.x, r1.x), fmaxf(r2.x, r3.x)),
                                     fmaxf(fmaxf(r0.y, r1.y), fmaxf(r2.y, r3.y)),
                                     fmaxf(fmaxf(r0.z, r1.z), fmaxf(r2.z, r3.z)),
                                     fmaxf(fmaxf(r0.w, r1.w), fmaxf(r2.w, r3.w))};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float mo = m_run[k + e];
                    const float mn = fmaxf(mo, mt[e]);
                    const float a = (mo == kNegInf) ? 0.0f : ex2_approx(mo - mn);
                    grew |= (a < 1.0f ? 1u : 0u) << (k + e);
                    al[k + e] = a;
                    m_run[k + e] = mn;
                    const float pr = ex2_approx(x[k + e] - mn);
                    l_part[k + e] = l_part[k + e] * a + pr;
                    x[k + e] = pr;
                }
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
            if (st == 0 && tau < 16) DSA_TRACE_AT(p, 40 + tau);
        }

        // ---- epilogue ----
        warp_wait(p, barp(BAR_PVDONE), (tau - 1) & 1, abort_flag);
        if (st == 0 && i == 0) DSA_TRACE_AT(p, 17);
        tc_fence_after();
        // Row sums: this thread's token over its 32 heads -> per head over the warp (lane k
        // ends with head h0+k) -> over the 4 quarters.
        {
            float v[32];
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = l_part[k];
#define DSA_SUM_STEP(W, OFF)                                                    \
    {                                                                           \
        const bool upper = (lane & (OFF)) != 0;                                 \
        _Pragma("unroll") for (int k = 0; k < (W); ++k) {                       \
            const float send = upper ? v[k] : v[k + (W)];                       \
            const float keep = upper ? v[k + (W)] : v[k];                       \
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, (OFF));            \
        }                                                                       \
    }
            DSA_SUM_STEP(16, 16)
            DSA_SUM_STEP(8, 8)
            DSA_SUM_STEP(4, 4)
            DSA_SUM_STEP(2, 2)
            DSA_SUM_STEP(1, 1)
#undef DSA_SUM_STEP
            red[q4 * kHeadsPerCta + h0 + lane] = v[0];   // parity-0 half of the scratch
        }
        half_bar_sync(hh);
        float f[32];
        const bool whole = s.part < 0;
#pragma unroll
        for (int k = 0; k < 32; k += 4) {
            const float4 r0 = *reinterpret_cast<const float4*>(red + 0 * kHeadsPerCta + h0 + k);
            const float4 r1 = *reinterpret_cast<const float4*>(red + 1 * kHeadsPerCta + h0 + k);
            const float4 r2 = *reinterpret_cast<const float4*>(red + 2 * kHeadsPerCta + h0 + k);
            const float4 r3 = *reinterpret_cast<const float4*>(red + 3 * kHeadsPerCta + h0 + k);
            const float l[4] = {(r0.x + r1.x) + (r2.x + r3.x), (r0.y + r1.y) + (r2.y + r3.y),
                                (r0.z + r1.z) + (r2.z + r3.z), (r0.w + r1.w) + (r2.w + r3.w)};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                f[k + e] = (whole ? p.v_scale : 1.0f) / (kPScale * l[e]);
                if (!whole && q4 == 0 && lane == 0)
                    p.part_lse[s.part * kHeadsPerCta + h0 + k + e] = m_run[k + e] + __log2f(l[e]);
            }
        }
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
                float* rows = p.part_o + static_cast<int64_t>(s.part) * kHeadsPerCta * kLatent;
                store_block(rows, h0, kHeadsPerCta, dim0, o, f, stage, lane);
                store_block(rows, h0 + 16, kHeadsPerCta, dim0, o + 16, f + 16, stage, lane);
            }
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
