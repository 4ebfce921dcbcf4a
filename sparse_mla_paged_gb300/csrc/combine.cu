// Log-sum-exp combine of per-CTA partials for work units split across CTAs.
//
// A partial k of unit (row, head group) holds O_k = (sum_j 2^(x_j - m_k) V_j) / l_k in
// E4M3 code units (stored as f16) and lse_k = m_k + log2(l_k), x being the score in log2 units. The
// softmax over the union of the pieces is out = v_scale * sum_k 2^(lse_k - LSE) O_k with
// LSE = log2 sum_k 2^lse_k; a piece with no tokens has lse = -inf and weight 0, and a
// unit whose pieces are all empty is 0. Units owned by one CTA were written directly by
// the decode kernel and are skipped here.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kCombineThreads = 256;
constexpr int kCombineHeads = kCombineThreads / 64;  // heads per block; 64 threads x 8 dims per head
constexpr int kPieceBatch = 8;                        // partial loads in flight per thread
constexpr float kNegInfC = -__builtin_huge_valf();

// Partial slot of unit u in CTA c, or -1 when CTA c has no slots at all.
__device__ __forceinline__ int32_t piece_slot(const Partition& part, int64_t u, int64_t c) {
    const int64_t b = cta_begin(part, c);
    if (b >= cta_begin(part, c + 1)) return -1;
    return static_cast<int32_t>(2 * c + (u == b / part.width ? 0 : 1));
}

// Softmax-weighted sum of a head's pieces; writes v_scale * acc / wsum as BF16.
__device__ __forceinline__ void store_head(const CombineParams& p, int32_t r, int32_t h, int dim0, const float (&acc)[8],
                                           float wsum) {
    if (h >= p.heads) return;
    const float f = wsum > 0.0f ? p.v_scale / wsum : 0.0f;
    uint4 packed;
    uint32_t* pw = reinterpret_cast<uint32_t*>(&packed);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * k] * f, acc[2 * k + 1] * f);
        pw[k] = *reinterpret_cast<uint32_t*>(&b);
    }
    *reinterpret_cast<uint4*>(p.out + (static_cast<int64_t>(r) * p.heads + h) * kLatent + dim0) = packed;
}

// Block (u, hb): heads hb*4 .. hb*4+3 of unit u; thread t: head hb*4 + t/64, dims 8*(t%64) ..
// +8. kFastPieces > 0 (the host's bound on pieces per unit): the pieces' partial slots are
// found before the grid-dependency wait (they depend on the partition only), then every
// thread loads its head's lse values and 16-byte slices of all pieces at once and folds
// them in registers. kFastPieces = 0: the block stages up to 256 pieces' slots and lse
// values per round in shared memory and folds them into a running softmax, kPieceBatch
// loads at a time. The variants differ in registers, hence in blocks per SM.
template <int kFastPieces>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p) {
    // After a long decode the next call's first kernel may launch now (it waits for this
    // grid to complete); otherwise it launches when this grid exits.
    if (p.early_dependents) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    __shared__ int32_t slot_s[kCombineThreads];
    __shared__ float lse_s[kCombineHeads][kCombineThreads];
    const int64_t u = blockIdx.x;
    const int hh = threadIdx.x >> 6;
    const int hl = blockIdx.y * kCombineHeads + hh;
    const int dim0 = (threadIdx.x & 63) * 8;
    const int32_t r = static_cast<int32_t>(u / p.part.groups), g = static_cast<int32_t>(u % p.part.groups);
    const int32_t h = g * kHeadsPerCta + hl;
    const int64_t W = p.part.width;
    const int64_t c_lo = cta_of_slot(p.part, u * W);
    const int64_t c_hi = cta_of_slot(p.part, (u + 1) * W - 1);
    const int64_t npieces = c_hi + 1 - c_lo;
    if (npieces == 1) return;  // written whole by the decode kernel (uniform over the block)

    if (kFastPieces > 0 && npieces <= kFastPieces) {
        if (static_cast<int64_t>(threadIdx.x) < npieces) slot_s[threadIdx.x] = piece_slot(p.part, u, c_lo + threadIdx.x);
        __syncthreads();
        // Launched as a programmatic dependent of the decode kernel: wait for its partials.
        asm volatile("griddepcontrol.wait;" ::: "memory");
        const int n = static_cast<int>(npieces);
        constexpr int kN = kFastPieces > 0 ? kFastPieces : 1;
        float lse[kN];
        uint4 raw[kN];
#pragma unroll
        for (int e = 0; e < kN; ++e) {
            lse[e] = kNegInfC;
            raw[e] = make_uint4(0, 0, 0, 0);
            if (e < n && slot_s[e] >= 0) {  // a CTA without slots has no piece
                const int64_t slot = slot_s[e];
                lse[e] = p.part_lse[slot * kHeadsPerCta + hl];
                raw[e] = *reinterpret_cast<const uint4*>(p.part_o + (slot * kHeadsPerCta + hl) * kLatent + dim0);
            }
        }
        float m = kNegInfC;
#pragma unroll
        for (int e = 0; e < kN; ++e) m = fmaxf(m, lse[e]);
        float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
        float wsum = 0.0f;
        if (m != kNegInfC) {
#pragma unroll
            for (int e = 0; e < kN; ++e) {
                const float w = exp2f(lse[e] - m);  // 0 for an empty piece (lse = -inf)
                wsum += w;
                const __half2* hv = reinterpret_cast<const __half2*>(&raw[e]);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = __half22float2(hv[k]);
                    acc[2 * k] += w * f.x;
                    acc[2 * k + 1] += w * f.y;
                }
            }
        }
        store_head(p, r, h, dim0, acc, wsum);
        return;
    }

    asm volatile("griddepcontrol.wait;" ::: "memory");
    float mx = kNegInfC, wsum = 0.0f;
    float acc[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) acc[k] = 0.0f;
    for (int64_t c0 = c_lo; c0 <= c_hi; c0 += kCombineThreads) {
        const int n = static_cast<int>(min(c_hi + 1 - c0, static_cast<int64_t>(kCombineThreads)));
        __syncthreads();  // the previous round's smem is no longer read
        if (static_cast<int>(threadIdx.x) < n) {
            const int32_t slot = piece_slot(p.part, u, c0 + threadIdx.x);
            slot_s[threadIdx.x] = slot;
#pragma unroll
            for (int k = 0; k < kCombineHeads; ++k)
                lse_s[k][threadIdx.x] =
                    slot >= 0 ? p.part_lse[static_cast<int64_t>(slot) * kHeadsPerCta + blockIdx.y * kCombineHeads + k]
                              : kNegInfC;
        }
        __syncthreads();
        float m = mx;
        for (int e = 0; e < n; ++e) m = fmaxf(m, lse_s[hh][e]);
        if (m == kNegInfC) continue;
        if (m > mx) {  // rescale what was folded so far
            const float a = mx == kNegInfC ? 0.0f : exp2f(mx - m);
            wsum *= a;
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] *= a;
            mx = m;
        }
        for (int e0 = 0; e0 < n; e0 += kPieceBatch) {
            uint4 raw[kPieceBatch];
            float w[kPieceBatch];
#pragma unroll
            for (int e = 0; e < kPieceBatch; ++e) {
                const int k = e0 + e;
                w[e] = k < n ? exp2f(lse_s[hh][k] - mx) : 0.0f;
                raw[e] = make_uint4(0, 0, 0, 0);
                if (w[e] != 0.0f)
                    raw[e] = *reinterpret_cast<const uint4*>(
                        p.part_o + (static_cast<int64_t>(slot_s[k]) * kHeadsPerCta + hl) * kLatent + dim0);
            }
#pragma unroll
            for (int e = 0; e < kPieceBatch; ++e) {
                wsum += w[e];
                const __half2* hv = reinterpret_cast<const __half2*>(&raw[e]);
#pragma unroll
                for (int k = 0; k < 4; ++k) {
                    const float2 f = __half22float2(hv[k]);
                    acc[2 * k] += w[e] * f.x;
                    acc[2 * k + 1] += w[e] * f.y;
                }
            }
        }
    }
    store_head(p, r, h, dim0, acc, wsum);
}

}  // namespace

cudaError_t combine_kernel_setup() {
    const void* fns[] = {reinterpret_cast<const void*>(combine_kernel<0>),
                         reinterpret_cast<const void*>(combine_kernel<4>),
                         reinterpret_cast<const void*>(combine_kernel<16>)};
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
    cfg.gridDim = dim3(units, kHeadsPerCta / kCombineHeads);
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (max_pieces <= 4) return cudaLaunchKernelEx(&cfg, combine_kernel<4>, p);
    if (max_pieces <= 16) return cudaLaunchKernelEx(&cfg, combine_kernel<16>, p);
    return cudaLaunchKernelEx(&cfg, combine_kernel<0>, p);
}

}  // namespace dsa
