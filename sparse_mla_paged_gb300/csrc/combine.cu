// Log-sum-exp combine of per-CTA partials for work units split across CTAs.
//
// A partial k of unit (row, head group) holds O_k = (sum_j 2^(x_j - m_k) V_j) / l_k in
// E4M3 code units and lse_k = m_k + log2(l_k), x being the score in log2 units. The
// softmax over the union of the pieces is out = v_scale * sum_k 2^(lse_k - LSE) O_k with
// LSE = log2 sum_k 2^lse_k; a piece with no tokens has lse = -inf and weight 0, and a
// unit whose pieces are all empty is 0. Units owned by one CTA were written directly by
// the decode kernel and are skipped here.
#include <cuda_bf16.h>

#include "common.cuh"

namespace dsa {
namespace {

constexpr int kCombineThreads = 128;  // 4 latent dims per thread
constexpr int kMaxPieces = 64;        // pieces buffered in shared memory per pass

__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p) {
    // Launched as a programmatic dependent of the decode kernel: wait for its partials.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const int64_t u = blockIdx.x;
    const int hl = blockIdx.y;
    const int32_t r = static_cast<int32_t>(u / p.part.groups), g = static_cast<int32_t>(u % p.part.groups);
    const int32_t h = g * kHeadsPerCta + hl;
    if (h >= p.heads) return;
    const int64_t W = p.part.width;
    const int64_t c_lo = cta_of_slot(p.part, u * W);
    const int64_t c_hi = cta_of_slot(p.part, (u + 1) * W - 1);
    if (c_lo == c_hi) return;

    __shared__ float lse_s[kMaxPieces];
    __shared__ int32_t slot_s[kMaxPieces];
    // Pass 1: the maximum lse over the pieces.
    float mx = -__int_as_float(0x7f800000);
    for (int64_t c = c_lo; c <= c_hi; ++c) {
        if (cta_begin(p.part, c) >= cta_begin(p.part, c + 1)) continue;  // CTA with no slots
        const int32_t first = static_cast<int32_t>(cta_begin(p.part, c) / W);
        const int32_t slot = static_cast<int32_t>(2 * c + (u == first ? 0 : 1));
        mx = fmaxf(mx, p.part_lse[static_cast<int64_t>(slot) * kHeadsPerCta + hl]);
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.0f;
    if (mx != -__int_as_float(0x7f800000)) {
        for (int64_t c0 = c_lo; c0 <= c_hi; c0 += kMaxPieces) {
            const int64_t c1 = min(c_hi + 1, c0 + kMaxPieces);
            __syncthreads();
            for (int64_t c = c0 + threadIdx.x; c < c1; c += kCombineThreads) {
                const int k = static_cast<int>(c - c0);
                if (cta_begin(p.part, c) >= cta_begin(p.part, c + 1)) {
                    slot_s[k] = -1;
                    lse_s[k] = 0.f;
                    continue;
                }
                const int32_t first = static_cast<int32_t>(cta_begin(p.part, c) / W);
                const int32_t slot = static_cast<int32_t>(2 * c + (u == first ? 0 : 1));
                slot_s[k] = slot;
                lse_s[k] = p.part_lse[static_cast<int64_t>(slot) * kHeadsPerCta + hl];
            }
            __syncthreads();
            for (int k = 0; k < static_cast<int>(c1 - c0); ++k) {
                if (slot_s[k] < 0) continue;
                const float w = exp2f(lse_s[k] - mx);
                wsum += w;
                if (w == 0.0f) continue;
                const float4 o = reinterpret_cast<const float4*>(
                    p.part_o + (static_cast<int64_t>(slot_s[k]) * kHeadsPerCta + hl) * kLatent)[threadIdx.x];
                acc.x += w * o.x;
                acc.y += w * o.y;
                acc.z += w * o.z;
                acc.w += w * o.w;
            }
        }
    }
    const float f = wsum > 0.0f ? p.v_scale / wsum : 0.0f;
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * f, acc.y * f);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * f, acc.w * f);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    reinterpret_cast<uint2*>(p.out + (static_cast<int64_t>(r) * p.heads + h) * kLatent)[threadIdx.x] = packed;
}

}  // namespace

cudaError_t combine_kernel_setup() {
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, combine_kernel);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(combine_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

cudaError_t launch_combine(const CombineParams& p, int units, cudaStream_t stream) {
    if (units <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units, kHeadsPerCta);
    cfg.blockDim = dim3(kCombineThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, combine_kernel, p);
}

}  // namespace dsa
