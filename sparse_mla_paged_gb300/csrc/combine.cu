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

constexpr int kCombineThreads = 128;  // 4 latent dims per thread; also pieces per chunk
constexpr float kNegInfC = -__builtin_huge_valf();

// Partial slot of unit u in CTA c, or -1 when CTA c has no slots at all.
__device__ __forceinline__ int32_t piece_slot(const Partition& part, int64_t u, int64_t c) {
    const int64_t b = cta_begin(part, c);
    if (b >= cta_begin(part, c + 1)) return -1;
    return static_cast<int32_t>(2 * c + (u == b / part.width ? 0 : 1));
}

__device__ __forceinline__ float block_max(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    const float m = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
    __syncthreads();
    return m;
}

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

    __shared__ float red[4];
    __shared__ float w_s[kCombineThreads];
    __shared__ int32_t slot_s[kCombineThreads];
    // Pass 1: the largest log-sum-exp over the pieces.
    float mx = kNegInfC;
    for (int64_t c0 = c_lo; c0 <= c_hi; c0 += kCombineThreads) {
        const int64_t c = c0 + threadIdx.x;
        float lse = kNegInfC;
        if (c <= c_hi) {
            const int32_t slot = piece_slot(p.part, u, c);
            if (slot >= 0) lse = p.part_lse[static_cast<int64_t>(slot) * kHeadsPerCta + hl];
        }
        mx = fmaxf(mx, block_max(lse, red));
    }
    // Pass 2: out = v_scale * sum_k 2^(lse_k - mx) O_k / sum_k 2^(lse_k - mx).
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.0f;
    if (mx != kNegInfC) {
        for (int64_t c0 = c_lo; c0 <= c_hi; c0 += kCombineThreads) {
            const int n = static_cast<int>(min(c_hi + 1 - c0, static_cast<int64_t>(kCombineThreads)));
            if (threadIdx.x < n) {
                const int32_t slot = piece_slot(p.part, u, c0 + threadIdx.x);
                float w = 0.0f;
                if (slot >= 0) w = exp2f(p.part_lse[static_cast<int64_t>(slot) * kHeadsPerCta + hl] - mx);
                slot_s[threadIdx.x] = slot;
                w_s[threadIdx.x] = w;
            }
            __syncthreads();
            for (int k0 = 0; k0 < n; k0 += 8) {
                float4 o[8];
                float w[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    const int k = k0 + e;
                    w[e] = k < n ? w_s[k] : 0.0f;
                    if (w[e] != 0.0f) {
                        const uint2 raw = reinterpret_cast<const uint2*>(
                            p.part_o + (static_cast<int64_t>(slot_s[k]) * kHeadsPerCta + hl) * kLatent)[threadIdx.x];
                        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
                        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
                        o[e] = make_float4(a.x, a.y, b.x, b.y);
                    } else {
                        o[e] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    wsum += w[e];
                    acc.x += w[e] * o[e].x;
                    acc.y += w[e] * o[e].y;
                    acc.z += w[e] * o[e].z;
                    acc.w += w[e] * o[e].w;
                }
            }
            __syncthreads();
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
