// Log-sum-exp combine of per-CTA partials for work units split across CTAs.
//
// A partial k of unit (row, head group) holds O_k = (sum_j 2^(x_j - m_k) V_j) / l_k in
// E4M3 code units, stored as f16 laid out [16 blocks of 32 dims][8 head groups][32 dims]
// [8 heads] (a block's 64 heads x 32 dims are 4 contiguous KB), and
// lse_k = m_k + log2(l_k), x being the score in log2 units. The softmax over the union of
// the pieces is out = v_scale * sum_k 2^(lse_k - LSE) O_k with LSE = log2 sum_k 2^lse_k; a
// piece with no tokens has lse = -inf and weight 0, and a unit whose pieces are all empty
// is 0. Units owned by one CTA were written directly by the decode kernel and are skipped.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kCombineWarps = kCombineThreads / 32;  // one per group of 8 heads
constexpr int kCombineDims = 32;                      // dims per block: the lanes of a warp
constexpr int kWeightChunk = 16;                      // pieces whose weights sit in shared memory at once
constexpr float kNegInfC = -__builtin_huge_valf();
static_assert(kCombineWarps * 8 == kHeadsPerCta, "a warp per 8-head group");

// The partition's arithmetic (cta_begin, cta_of_slot of common.cuh), in 32-bit unsigned
// arithmetic when every product fits (exact either way; a 64-bit division is a long
// software sequence, and each block of this kernel does several before its first load).
template <bool kNarrow>
__device__ __forceinline__ int64_t div_c(int64_t a, int64_t b) {
    if constexpr (kNarrow) return static_cast<int64_t>(static_cast<uint32_t>(a) / static_cast<uint32_t>(b));
    else return a / b;
}
template <bool kNarrow>
__device__ __forceinline__ int64_t begin_c(const Partition& part, int64_t c) {
    return div_c<kNarrow>(c * part.total_slots, part.ctas);
}
template <bool kNarrow>
__device__ __forceinline__ int64_t cta_of_c(const Partition& part, int64_t x) {
    return div_c<kNarrow>((x + 1) * part.ctas - 1, part.total_slots);
}

// Partial slot of unit u in CTA c, or -1 when CTA c has no slots at all.
template <bool kNarrow>
__device__ __forceinline__ int32_t piece_slot(const Partition& part, int64_t u, int64_t c) {
    const int64_t b = begin_c<kNarrow>(part, c);
    if (b >= begin_c<kNarrow>(part, c + 1)) return -1;
    return static_cast<int32_t>(2 * c + (u == div_c<kNarrow>(b, part.width) ? 0 : 1));
}

// v_scale * 2^(lse - m) / sum for one piece of one head, given f = v_scale / sum (0 for an
// empty piece, or a head whose pieces are all empty).
__device__ __forceinline__ float piece_weight(float lse, float m, float f) {
    return lse != kNegInfC ? f * exp2f(lse - m) : 0.0f;
}

// Block (u, db): dims 32*db .. 32*db + 31 of unit u, all 64 heads. Warp w takes heads
// 8w .. 8w + 7 and lane l dim 32*db + l, so the block reads 4 contiguous KB of each partial
// and each warp load 512 bytes; the output tile is transposed through shared memory. Lanes 0..7 of a warp form the
// pieces' weights of its 8 heads into the warp's own shared-memory rows (warp-level sync).
// kFast > 0 (the host's bound on pieces per unit): the pieces' partial slots are found
// before the grid-dependency wait (they depend on the partition only), then every thread
// loads its 16-byte slice of every piece at once while the weight lanes load the lse
// values: one round trip. kFast = 0: any number of pieces, kWeightChunk at a time, one
// round trip per chunk with a running maximum.
template <int kFast, bool kNarrow>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p) {
    // After a long decode the next call's first kernel may launch now (it waits for this
    // grid to complete); otherwise it launches when this grid exits.
    if (p.early_dependents) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ int32_t slot_s[kCombineThreads];
    __shared__ float w_s[kCombineWarps][kWeightChunk][8];
    __shared__ __align__(16) float a_s[kCombineWarps][8];  // per-head factors of the generic path
    __shared__ __align__(16) __nv_bfloat16 out_s[kHeadsPerCta][kCombineDims];  // the block's output tile
    const int64_t u = blockIdx.x;
    const int t = threadIdx.x, warp = t >> 5, lane = t & 31;
    const int dim = blockIdx.y * kCombineDims + lane;
    const int32_t r = static_cast<int32_t>(div_c<kNarrow>(u, p.part.groups));
    const int32_t g = static_cast<int32_t>(u - static_cast<int64_t>(r) * p.part.groups);
    const int64_t W = p.part.width;
    const int64_t c_lo = cta_of_c<kNarrow>(p.part, u * W);
    const int64_t c_hi = cta_of_c<kNarrow>(p.part, (u + 1) * W - 1);
    const int64_t npieces = c_hi + 1 - c_lo;
    if (npieces == 1) return;  // written whole by the decode kernel (uniform over the block)
    const __half* po = reinterpret_cast<const __half*>(p.part_o);
    auto slice = [&](int32_t slot) {  // heads 8*warp .. +8 of this lane's dim in partial `slot`
        return *reinterpret_cast<const uint4*>(
            po + static_cast<int64_t>(slot) * kHeadsPerCta * kLatent +
            ((static_cast<int64_t>(blockIdx.y) * kCombineWarps + warp) * kCombineDims + lane) * 8);
    };
    auto lse_of = [&](int32_t slot) {  // lse of head 8*warp + lane (lanes 0..7)
        return p.part_lse[static_cast<int64_t>(slot) * kHeadsPerCta + warp * 8 + lane];
    };
    float acc[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
    auto fold = [&](const uint4& raw, int k) {
        const __half2* hv = reinterpret_cast<const __half2*>(&raw);
        const float4 wa = *reinterpret_cast<const float4*>(&w_s[warp][k][0]);
        const float4 wb = *reinterpret_cast<const float4*>(&w_s[warp][k][4]);
        const float w[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float2 f = __half22float2(hv[e]);
            acc[2 * e] += w[2 * e] * f.x;
            acc[2 * e + 1] += w[2 * e + 1] * f.y;
        }
    };

    if (kFast > 0 && npieces <= kFast) {
        const int n = static_cast<int>(npieces);
        if (t < n) slot_s[t] = piece_slot<kNarrow>(p.part, u, c_lo + t);
        __syncthreads();
        // Launched as a programmatic dependent of the decode kernel: wait for its partials.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        constexpr int kN = kFast > 0 ? kFast : 1;
        uint4 raw[kN];
#pragma unroll
        for (int k = 0; k < kN; ++k) {
            raw[k] = make_uint4(0, 0, 0, 0);
            if (k < n && slot_s[k] >= 0) raw[k] = slice(slot_s[k]);  // a CTA without slots has no piece
        }
        if (lane < 8) {
            float lse[kN];
            float m = kNegInfC;
#pragma unroll
            for (int k = 0; k < kN; ++k) {
                lse[k] = (k < n && slot_s[k] >= 0) ? lse_of(slot_s[k]) : kNegInfC;
                m = fmaxf(m, lse[k]);
            }
            float sum = 0.0f;
            if (m != kNegInfC) {
#pragma unroll
                for (int k = 0; k < kN; ++k) sum += exp2f(lse[k] - m);  // 0 for an empty piece
            }
            const float f = sum > 0.0f ? p.v_scale / sum : 0.0f;
#pragma unroll
            for (int k = 0; k < kN; ++k)
                if (k < n) w_s[warp][k][lane] = piece_weight(lse[k], m, f);
        }
        __syncwarp();
#pragma unroll
        for (int k = 0; k < kN; ++k)
            if (k < n) fold(raw[k], k);
    } else if constexpr (kFast > 0) {
        // More pieces than the variant's bound (the host never launches it so): the plain
        // loop, piece by piece.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        // Maximum and sum over every piece, per head (lanes 0..7 of each warp).
        float m = kNegInfC, sum = 0.0f;
        if (lane < 8) {
            for (int64_t k = 0; k < npieces; ++k) {
                const int32_t slot = piece_slot<kNarrow>(p.part, u, c_lo + k);
                if (slot >= 0) m = fmaxf(m, lse_of(slot));
            }
            if (m != kNegInfC)
                for (int64_t k = 0; k < npieces; ++k) {
                    const int32_t slot = piece_slot<kNarrow>(p.part, u, c_lo + k);
                    if (slot >= 0) sum += exp2f(lse_of(slot) - m);
                }
        }
        const float f = sum > 0.0f ? p.v_scale / sum : 0.0f;
        for (int64_t k0 = 0; k0 < npieces; k0 += kWeightChunk) {
            const int n = static_cast<int>(min(npieces - k0, static_cast<int64_t>(kWeightChunk)));
            __syncthreads();  // the previous chunk's slots and weights are no longer read
            if (t < n) slot_s[t] = piece_slot<kNarrow>(p.part, u, c_lo + k0 + t);
            __syncthreads();
            if (lane < 8)
                for (int k = 0; k < n; ++k)
                    w_s[warp][k][lane] = slot_s[k] >= 0 ? piece_weight(lse_of(slot_s[k]), m, f) : 0.0f;
            __syncwarp();
            for (int k = 0; k < n; ++k)
                if (slot_s[k] >= 0) fold(slice(slot_s[k]), k);
        }
    } else {
        asm volatile("griddepcontrol.wait;" ::: "memory");
        // Any number of pieces, kWeightChunk at a time, in one pass: each chunk's slices and
        // log-sum-exps are all requested at once (one round trip per chunk), and the fold
        // keeps a running maximum per head (lanes 0..7 of each warp), rescaling what it has
        // accumulated when the maximum rises; the sum of the weights divides at the end.
        float m_run = kNegInfC, s_run = 0.0f;
        for (int64_t k0 = 0; k0 < npieces; k0 += kWeightChunk) {
            const int n = static_cast<int>(min(npieces - k0, static_cast<int64_t>(kWeightChunk)));
            __syncthreads();  // the previous chunk's slots and weights are no longer read
            if (t < n) slot_s[t] = piece_slot<kNarrow>(p.part, u, c_lo + k0 + t);
            __syncthreads();
            uint4 raw[kWeightChunk];
#pragma unroll
            for (int k = 0; k < kWeightChunk; ++k) {
                raw[k] = make_uint4(0, 0, 0, 0);
                if (k < n && slot_s[k] >= 0) raw[k] = slice(slot_s[k]);
            }
            if (lane < 8) {
                float lse[kWeightChunk];
                float cm = kNegInfC;
#pragma unroll
                for (int k = 0; k < kWeightChunk; ++k) {
                    lse[k] = (k < n && slot_s[k] >= 0) ? lse_of(slot_s[k]) : kNegInfC;
                    cm = fmaxf(cm, lse[k]);
                }
                const float m_new = fmaxf(m_run, cm);
                const float a = m_run != kNegInfC ? exp2f(m_run - m_new) : 0.0f;
                s_run *= a;
#pragma unroll
                for (int k = 0; k < kWeightChunk; ++k) {
                    const float w = piece_weight(lse[k], m_new, 1.0f);
                    s_run += w;
                    w_s[warp][k][lane] = w;
                }
                a_s[warp][lane] = a;
                m_run = m_new;
            }
            __syncwarp();
            const float4 aa = *reinterpret_cast<const float4*>(&a_s[warp][0]);
            const float4 ab = *reinterpret_cast<const float4*>(&a_s[warp][4]);
            const float av[8] = {aa.x, aa.y, aa.z, aa.w, ab.x, ab.y, ab.z, ab.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] *= av[e];
#pragma unroll
            for (int k = 0; k < kWeightChunk; ++k)
                if (k < n) fold(raw[k], k);
        }
        __syncwarp();
        if (lane < 8) a_s[warp][lane] = s_run > 0.0f ? p.v_scale / s_run : 0.0f;
        __syncwarp();
        const float4 fa = *reinterpret_cast<const float4*>(&a_s[warp][0]);
        const float4 fb = *reinterpret_cast<const float4*>(&a_s[warp][4]);
        const float fv[8] = {fa.x, fa.y, fa.z, fa.w, fb.x, fb.y, fb.z, fb.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] *= fv[e];
    }
    // The block's output tile [64 heads][32 dims] goes through shared memory, so that each
    // thread writes 16 bytes (8 dims of one head) of the BF16 output rows.
#pragma unroll
    for (int e = 0; e < 8; ++e) out_s[warp * 8 + e][lane] = __float2bfloat16_rn(acc[e]);
    __syncthreads();
    const int hl = t / 4, c = (t % 4) * 8;
    if (hl < p.heads - g * kHeadsPerCta)
        *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(p.out) +
                                  (static_cast<int64_t>(r) * p.heads + g * kHeadsPerCta + hl) * kLatent +
                                  blockIdx.y * kCombineDims + c) = *reinterpret_cast<const uint4*>(&out_s[hl][c]);
}

}  // namespace

cudaError_t combine_kernel_setup() {
    const void* fns[] = {reinterpret_cast<const void*>(combine_kernel<0, false>),
                         reinterpret_cast<const void*>(combine_kernel<4, false>),
                         reinterpret_cast<const void*>(combine_kernel<16, false>),
                         reinterpret_cast<const void*>(combine_kernel<0, true>),
                         reinterpret_cast<const void*>(combine_kernel<4, true>),
                         reinterpret_cast<const void*>(combine_kernel<16, true>)};
    for (const void* f : fns) {
        cudaFuncAttributes attr;
        cudaError_t e = cudaFuncGetAttributes(&attr, f);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(f, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_combine(const CombineParams& p, int units, int max_pieces, cudaStream_t stream) {
    if (units <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units, kLatent / kCombineDims);
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (p.part.narrow) {
        if (max_pieces <= 4) return cudaLaunchKernelEx(&cfg, combine_kernel<4, true>, p);
        if (max_pieces <= 16) return cudaLaunchKernelEx(&cfg, combine_kernel<16, true>, p);
        return cudaLaunchKernelEx(&cfg, combine_kernel<0, true>, p);
    }
    if (max_pieces <= 4) return cudaLaunchKernelEx(&cfg, combine_kernel<4, false>, p);
    if (max_pieces <= 16) return cudaLaunchKernelEx(&cfg, combine_kernel<16, false>, p);
    return cudaLaunchKernelEx(&cfg, combine_kernel<0, false>, p);
}

}  // namespace dsa
