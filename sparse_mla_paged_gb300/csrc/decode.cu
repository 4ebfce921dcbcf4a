// The selected-index NoPE MLA paged decode kernel (attend.rs, decode_attention).
//
// One CTA per SM (persistent over a static slot-space partition, see common.cuh). Work
// unit = (decode row, group of 64 query heads). For each tile of 128 resolved tokens:
//
//   gather   warps 0-3   cp.async 16-byte copies of each token's 512-byte E4M3 latent
//                        row (block-table resolved) into a 2-slot ring, written in the
//                        128-byte-swizzled K-major operand layout.
//   QK^T     warp 8      tcgen05.mma kind::f8f6f4, M = 128 tokens, N = 128 (64 heads x
//                        {hi, lo} query terms), K = 512: S^T -> TMEM (double buffered).
//   softmax  warps 4-7   one thread per token (TMEM lane): s = hi + lo, per-head scale,
//                        column max / sum across the 128 tokens by a transposing warp
//                        reduction, online max / rescale, P' = 256*exp2(x - m) written
//                        to shared memory as two E4M3 terms (hi = top 4 bits, lo = rest).
//   P.V      warp 8      O^T[512 dims x 64 heads] += V^T * P'^T in TMEM: the same ring
//                        slot read as an MN-major operand (K and V are the same bytes).
//   epilogue warps 4-7   O / (256 l) * v_scale -> BF16 output, or (O/l, lse) partials.
//
// The contraction is exact in its inputs: keys and values are the cached E4M3 codes
// themselves (k_scale and v_scale are applied outside the MMA), queries are split into
// two E4M3 terms that reproduce the BF16 value (see prologue.cu), probabilities into two
// terms that carry about 8 significant bits. Accumulation is FP32 in TMEM.
//
// Shared memory 217 KB, TMEM 512 columns: O^T at 0..255 (chunk c of 128 dims at 64c),
// S^T buffers at 256 and 384.
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 288;
constexpr int kProducerWarps = 4;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kMmaWarp = 8;
constexpr int kProducerThreads = kProducerWarps * 32;

constexpr int kOffRing = 0;
constexpr int kOffQ = 2 * kKvTileBytes;
constexpr int kOffPHi = kOffQ + kQImageBytes;
constexpr int kOffPLo = kOffPHi + kTileTokens * kHeadsPerCta;
constexpr int kOffRedMax = kOffPLo + kTileTokens * kHeadsPerCta;
constexpr int kOffRedSum = kOffRedMax + 4 * kHeadsPerCta * 4;
constexpr int kOffM = kOffRedSum + 4 * kHeadsPerCta * 4;
constexpr int kOffL = kOffM + kHeadsPerCta * 4;
constexpr int kOffAlpha = kOffL + kHeadsPerCta * 4;
constexpr int kOffCs = kOffAlpha + kHeadsPerCta * 4;
constexpr int kOffMask = kOffCs + kHeadsPerCta * 4;
constexpr int kOffBars = kOffMask + 16;
enum {
    BAR_FULL0, BAR_FULL1, BAR_EMPTY0, BAR_EMPTY1, BAR_SFULL0, BAR_SFULL1, BAR_SEMPTY0, BAR_SEMPTY1,
    BAR_PFULL, BAR_PVDONE, BAR_QFULL, BAR_QEMPTY, BAR_OEMPTY, BAR_DRAIN, kNumBars
};
constexpr int kOffTmemSlot = kOffBars + kNumBars * 8;
constexpr int kOffAbort = kOffTmemSlot + 4;
constexpr int kSmemUsed = kOffAbort + 4;
constexpr int kSmemBytes = kSmemUsed + 1024;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 0;
constexpr uint32_t kTmemS = 256;

constexpr float kNegInf = -__builtin_huge_valf();

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

// Column reduction over the warp's 32 lanes for 64 values per lane. On return v[0] and
// v[1] hold the reduction of heads 2*lane and 2*lane+1 (62 shuffles instead of 320).
template <bool kMax>
__device__ __forceinline__ void transpose_reduce(float (&v)[64], int lane) {
#define DSA_TR_STEP(W, OFF)                                                       \
    {                                                                             \
        const bool upper = (lane & (OFF)) != 0;                                   \
        _Pragma("unroll") for (int i = 0; i < (W); ++i) {                         \
            const float send = upper ? v[i] : v[i + (W)];                         \
            const float keep = upper ? v[i + (W)] : v[i];                         \
            const float got = __shfl_xor_sync(0xffffffffu, send, (OFF));          \
            v[i] = kMax ? fmaxf(keep, got) : keep + got;                          \
        }                                                                         \
    }
    DSA_TR_STEP(32, 16)
    DSA_TR_STEP(16, 8)
    DSA_TR_STEP(8, 4)
    DSA_TR_STEP(4, 2)
    DSA_TR_STEP(2, 1)
#undef DSA_TR_STEP
}

__device__ __forceinline__ uint32_t pack_e4m3x4(float a, float b, float c, float d) {
    return f32x2_to_e4m3x2(a, b) | (f32x2_to_e4m3x2(c, d) << 16);
}

__device__ __forceinline__ float hi_part(float x) {
    return __uint_as_float(__float_as_uint(x) & 0xFFF00000u);
}

// ------------------------------------------------------------------------------------
// gather warps
// ------------------------------------------------------------------------------------
__device__ void run_producer(const DecodeParams& p, uint32_t sbase, volatile int* abort_flag, int nseg) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nslot = p.kv_same ? 2 : 1;
    const int64_t W = p.part.width;
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
        }
        ++qseg;
        const int32_t* ids = p.ids + static_cast<int64_t>(s.row) * W + tl.t0;
        const int32_t seq = s.row / p.rows_per_seq;
        const int32_t* bt = p.block_tables + static_cast<int64_t>(seq) * p.max_blocks_per_seq;
        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            const int slot = static_cast<int>(tau % nslot);
            const uint32_t use = tau / nslot;
            if (tau >= static_cast<uint32_t>(nslot))
                warp_wait(p, sbase + kOffBars + 8 * (BAR_EMPTY0 + slot), (use - 1) & 1, abort_flag);
            const int tok = warp * 32 + lane;
            const int32_t idx = t * kTileTokens + tok;
            long long off = -1;
            if (idx < tl.n) {
                const int32_t id = ids[idx];
                const int32_t blk = p.block_shift >= 0 ? (id >> p.block_shift) : id / p.block_size;
                const int32_t inblk = id - blk * p.block_size;
                if (p.max_blocks_per_seq > 0 && blk >= p.max_blocks_per_seq) {
                    atomicCAS(p.status, 0, kStatusBounds);
                } else {
                    const int32_t page = bt[blk];
                    if (page < 0)
                        atomicCAS(p.status, 0, kStatusBounds);
                    else
                        off = static_cast<long long>(page) * p.cache_stride + static_cast<long long>(inblk) * kLatent;
                }
            }
            const uint32_t kdst = sbase + kOffRing + slot * kKvTileBytes;
            const uint32_t vdst = p.kv_same ? kdst : sbase + kOffRing + kKvTileBytes;
            const uint32_t chunk = ((lane >> 3) * kKBlockBytes);
#pragma unroll 4
            for (int j = 0; j < 32; ++j) {
                const long long o = __shfl_sync(0xffffffffu, off, j);
                const int tk = warp * 32 + j;
                const uint32_t d = chunk + tk * 128 + ((((lane & 7) ^ (tk & 7))) << 4);
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
        }
    }
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
                const uint64_t bh = smem_desc(sbase + kOffPHi + ks * 512, 128, 2048, kSwizzleNone);
                const uint64_t bl = smem_desc(sbase + kOffPLo + ks * 512, 128, 2048, kSwizzleNone);
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
        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            if (nslot == 1 && t > 0) issue_pv(tau - 1, t == 1);
            const int slot = static_cast<int>(tau % nslot);
            const uint32_t use = tau / nslot;
            if (!mbar_wait(barp(BAR_FULL0 + slot), use & 1, abort_flag)) fail(p, abort_flag, kStatusTimeout);
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
            if (t == tl.ntiles - 1) tc_commit(barp(BAR_QEMPTY));
            if (nslot == 2 && t > 0) issue_pv(tau - 1, t == 1);
        }
        issue_pv(tau - 1, tl.ntiles == 1);
        ++qseg;
    }
}

// ------------------------------------------------------------------------------------
// softmax / epilogue warps
// ------------------------------------------------------------------------------------
__device__ void run_softmax(const DecodeParams& p, uint8_t* smem, uint32_t sbase, uint32_t tmem,
                            volatile int* abort_flag, int nseg) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int st = tid - kSoftmaxWarp0 * 32;  // token row of the tile / TMEM lane
    const int q4 = warp - kSoftmaxWarp0;      // TMEM lane quarter
    float* red_max = reinterpret_cast<float*>(smem + kOffRedMax);
    float* red_sum = reinterpret_cast<float*>(smem + kOffRedSum);
    float* m_s = reinterpret_cast<float*>(smem + kOffM);
    float* l_s = reinterpret_cast<float*>(smem + kOffL);
    float* a_s = reinterpret_cast<float*>(smem + kOffAlpha);
    float* c_s = reinterpret_cast<float*>(smem + kOffCs);
    uint32_t* mask_s = reinterpret_cast<uint32_t*>(smem + kOffMask);
    auto barp = [&](int b) { return sbase + kOffBars + 8 * b; };
    const uint32_t lane_base = static_cast<uint32_t>(q4 * 32) << 16;
    uint32_t tau = 0;

    for (int i = 0; i < nseg; ++i) {
        const Segment s = cta_segment(p.part, blockIdx.x, i);
        const Tiles tl = segment_tokens(p, s);
        const int hvalid = min(kHeadsPerCta, p.heads - s.group * kHeadsPerCta);
        const int64_t out_head0 = static_cast<int64_t>(s.row) * p.heads + s.group * kHeadsPerCta;
        if (tl.n <= 0) {
            // Empty selection: the output is zero; a partial carries weight zero.
            if (s.part < 0) {
                for (int e = st; e < hvalid * kLatent; e += 128) p.out[out_head0 * kLatent + e] = 0;
            } else {
                float* po = p.part_o + static_cast<int64_t>(s.part) * kHeadsPerCta * kLatent;
                for (int e = st; e < kHeadsPerCta * kLatent; e += 128) po[e] = 0.0f;
                if (st < kHeadsPerCta) p.part_lse[s.part * kHeadsPerCta + st] = kNegInf;
            }
            continue;
        }
        if (st < kHeadsPerCta) {
            m_s[st] = kNegInf;
            l_s[st] = 0.0f;
            c_s[st] = p.qscale[static_cast<int64_t>(s.unit) * kHeadsPerCta + st];
        }
        named_bar_sync(1, 128);
        for (int t = 0; t < tl.ntiles; ++t, ++tau) {
            const int sb = tau & 1;
            warp_wait(p, barp(BAR_SFULL0 + sb), (tau >> 1) & 1, abort_flag);
            tc_fence_after();
            float x[64];
            {
                const uint32_t ta = tmem + lane_base + kTmemS + sb * 128;
                uint32_t a[32], b[32];
                tmem_ld_x32(ta, a);
                tmem_ld_x32(ta + 64, b);
#pragma unroll
                for (int k = 0; k < 32; ++k) x[k] = __uint_as_float(a[k]) + __uint_as_float(b[k]);
                tmem_ld_x32(ta + 32, a);
                tmem_ld_x32(ta + 96, b);
#pragma unroll
                for (int k = 0; k < 32; ++k) x[32 + k] = __uint_as_float(a[k]) + __uint_as_float(b[k]);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(barp(BAR_SEMPTY0 + sb));

            const bool valid = t * kTileTokens + st < tl.n;
#pragma unroll
            for (int h = 0; h < 64; h += 4) {
                const float4 c = *reinterpret_cast<const float4*>(c_s + h);
                x[h] = valid ? x[h] * c.x : kNegInf;
                x[h + 1] = valid ? x[h + 1] * c.y : kNegInf;
                x[h + 2] = valid ? x[h + 2] * c.z : kNegInf;
                x[h + 3] = valid ? x[h + 3] * c.w : kNegInf;
            }
            {
                float v[64];
#pragma unroll
                for (int h = 0; h < 64; ++h) v[h] = x[h];
                transpose_reduce<true>(v, lane);
                *reinterpret_cast<float2*>(red_max + q4 * 64 + 2 * lane) = make_float2(v[0], v[1]);
            }
            named_bar_sync(1, 128);
            if (st < kHeadsPerCta) {
                const float mt = fmaxf(fmaxf(red_max[st], red_max[64 + st]), fmaxf(red_max[128 + st], red_max[192 + st]));
                const float mo = m_s[st];
                const float mn = fmaxf(mo, mt);
                const float al = (mo == kNegInf) ? 0.0f : ex2_approx(mo - mn);
                m_s[st] = mn;
                a_s[st] = al;
                const uint32_t bal = __ballot_sync(0xffffffffu, t > 0 && al < 1.0f);
                if (lane == 0) mask_s[q4] = bal;
            }
            named_bar_sync(1, 128);
#pragma unroll
            for (int h = 0; h < 64; h += 4) {
                const float4 m = *reinterpret_cast<const float4*>(m_s + h);
                x[h] = ex2_approx(x[h] - m.x);
                x[h + 1] = ex2_approx(x[h + 1] - m.y);
                x[h + 2] = ex2_approx(x[h + 2] - m.z);
                x[h + 3] = ex2_approx(x[h + 3] - m.w);
            }
            {
                float v[64];
#pragma unroll
                for (int h = 0; h < 64; ++h) v[h] = x[h];
                transpose_reduce<false>(v, lane);
                *reinterpret_cast<float2*>(red_sum + q4 * 64 + 2 * lane) = make_float2(v[0], v[1]);
            }
            named_bar_sync(1, 128);
            if (st < kHeadsPerCta)
                l_s[st] = l_s[st] * a_s[st] + ((red_sum[st] + red_sum[64 + st]) + (red_sum[128 + st] + red_sum[192 + st]));

            // P and O may only change once the previous P.V has finished reading them.
            if (t > 0) warp_wait(p, barp(BAR_PVDONE), (tau - 1) & 1, abort_flag);
#pragma unroll
            for (int hc = 0; hc < 4; ++hc) {
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
                st_shared_v4(sbase + kOffPHi + hc * 2048 + st * 16, hw[0], hw[1], hw[2], hw[3]);
                st_shared_v4(sbase + kOffPLo + hc * 2048 + st * 16, lw[0], lw[1], lw[2], lw[3]);
            }
            if (t > 0) {
                tc_fence_after();
                uint64_t msk = static_cast<uint64_t>(mask_s[0]) | (static_cast<uint64_t>(mask_s[1]) << 32);
                while (msk) {
                    const int h = __ffsll(static_cast<long long>(msk)) - 1;
                    msk &= msk - 1;
                    const float al = a_s[h];
#pragma unroll
                    for (int mc = 0; mc < 4; ++mc) {
                        const uint32_t ta = tmem + lane_base + kTmemO + mc * 64 + h;
                        const float o = __uint_as_float(tmem_ld_x1(ta));
                        tmem_st_x1(ta, __float_as_uint(o * al));
                    }
                }
                tmem_wait_st();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(barp(BAR_PFULL));
        }

        // ---- epilogue ----
        warp_wait(p, barp(BAR_PVDONE), (tau - 1) & 1, abort_flag);
        tc_fence_after();
        named_bar_sync(1, 128);
        if (st < kHeadsPerCta) {
            const float l = l_s[st];
            // complete: v_scale / (256 l); partial: 1 / (256 l) and the log-sum-exp
            a_s[st] = (s.part < 0 ? p.v_scale : 1.0f) / (kPScale * l);
            if (s.part >= 0) p.part_lse[s.part * kHeadsPerCta + st] = m_s[st] + __log2f(l);
        }
        named_bar_sync(1, 128);
#pragma unroll 1
        for (int mc = 0; mc < 4; ++mc) {
            const int d = mc * 128 + q4 * 32 + lane;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t v[32];
                tmem_ld_x32(tmem + lane_base + kTmemO + mc * 64 + half * 32, v);
                if (s.part < 0) {
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int h = half * 32 + k;
                        if (h < hvalid) {
                            const float o = __uint_as_float(v[k]) * a_s[h];
                            p.out[(out_head0 + h) * kLatent + d] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
                        }
                    }
                } else {
                    float* po = p.part_o + static_cast<int64_t>(s.part) * kHeadsPerCta * kLatent;
#pragma unroll
                    for (int k = 0; k < 32; ++k) {
                        const int h = half * 32 + k;
                        po[h * kLatent + d] = __uint_as_float(v[k]) * a_s[h];
                    }
                }
            }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(barp(BAR_OEMPTY));
        named_bar_sync(1, 128);
    }
}

__global__ void __launch_bounds__(kThreads, 1) decode_kernel(const DecodeParams p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffAbort);

    if (tid == 0) {
        const uint32_t b = sbase + kOffBars;
        mbar_init(b + 8 * BAR_FULL0, 2 * kProducerThreads);
        mbar_init(b + 8 * BAR_FULL1, 2 * kProducerThreads);
        mbar_init(b + 8 * BAR_EMPTY0, 1);
        mbar_init(b + 8 * BAR_EMPTY1, 1);
        mbar_init(b + 8 * BAR_SFULL0, 1);
        mbar_init(b + 8 * BAR_SFULL1, 1);
        mbar_init(b + 8 * BAR_SEMPTY0, 4);
        mbar_init(b + 8 * BAR_SEMPTY1, 4);
        mbar_init(b + 8 * BAR_PFULL, 4);
        mbar_init(b + 8 * BAR_PVDONE, 1);
        mbar_init(b + 8 * BAR_QFULL, 1);
        mbar_init(b + 8 * BAR_QEMPTY, 1);
        mbar_init(b + 8 * BAR_OEMPTY, 4);
        mbar_init(b + 8 * BAR_DRAIN, 1);
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

    int64_t first_unit;
    const int nseg = cta_segments(p.part, blockIdx.x, &first_unit);

    if (warp < kProducerWarps) {
        run_producer(p, sbase, abort_flag, nseg);
    } else if (warp < kMmaWarp) {
        run_softmax(p, smem, sbase, tmem, abort_flag, nseg);
    } else if (lane == 0) {
        run_mma(p, sbase, tmem, abort_flag, nseg);
        // Wait (bounded, regardless of abort) until every issued MMA has completed.
        const uint32_t db = sbase + kOffBars + 8 * BAR_DRAIN;
        tc_commit(db);
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(db, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
        }
    }
    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kTmemCols);
    }
}

}  // namespace

cudaError_t decode_kernel_setup() {
    return cudaFuncSetAttribute(decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
}

cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
    decode_kernel<<<p.part.ctas, kThreads, kSmemBytes, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dsa
