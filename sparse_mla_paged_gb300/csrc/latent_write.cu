// The cache writer (decode_k.rs, decode_k: the latent_write launch): for each new token,
//   y[c] = x[c] / sqrt(mean_c x^2 + eps) * w[c] * (1/kv_scale),
// stored as E4M3 (round to nearest even, saturating to +-448) in the token's 512-byte
// row at (slot / block_size)*cache_stride_bytes + (slot % block_size)*512, where the
// decode reads it; slot = physical*block_size + pos % block_size. The pages launch one
// block of kv_lora_rank threads per token and do not show its body; the RMSNorm-then-scale
// order above is the plain reading.
//
// One warp per token, eight tokens per 256-thread block, 16 consecutive dims per lane:
// two 16-byte loads of kv_a and of the weight, a warp-wide sum of squares in FP32 (no
// shared memory, no block barrier), one 16-byte store of sixteen codes, so a warp writes
// its token's 512-byte row in one coalesced store.
#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kWriteWarps = 8;
constexpr int kDimsPerLane = kLatent / 32;  // 16

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ void unpack8(const uint4 v, float* f) {
    f[0] = bf16_lo(v.x); f[1] = bf16_hi(v.x); f[2] = bf16_lo(v.y); f[3] = bf16_hi(v.y);
    f[4] = bf16_lo(v.z); f[5] = bf16_hi(v.z); f[6] = bf16_lo(v.w); f[7] = bf16_hi(v.w);
}

__global__ void __launch_bounds__(kWriteWarps * 32) latent_write_kernel(const LatentWriteParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kWriteWarps + (threadIdx.x >> 5);
    if (r >= p.rows) return;
    const long long slot = p.slots[r];
    if (slot < 0) return;  // the whole warp: nothing to write for this row
    const uint4* xs = reinterpret_cast<const uint4*>(p.kv_a + r * kLatent) + 2 * lane;
    const uint4* ws = reinterpret_cast<const uint4*>(p.weight) + 2 * lane;
    float x[kDimsPerLane], w[kDimsPerLane];
    unpack8(__ldg(xs), x);
    unpack8(__ldg(xs + 1), x + 8);
    unpack8(__ldg(ws), w);
    unpack8(__ldg(ws + 1), w + 8);
    float ss = 0.0f;
#pragma unroll
    for (int k = 0; k < kDimsPerLane; ++k) ss = fmaf(x[k], x[k], ss);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    const float inv_rms = rsqrtf(ss * (1.0f / kLatent) + p.eps);
    uint32_t codes[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int d = 4 * k;
        codes[k] = f32x2_to_e4m3x2(x[d] * inv_rms * w[d] * p.inv_scale, x[d + 1] * inv_rms * w[d + 1] * p.inv_scale) |
                   (f32x2_to_e4m3x2(x[d + 2] * inv_rms * w[d + 2] * p.inv_scale,
                                    x[d + 3] * inv_rms * w[d + 3] * p.inv_scale)
                    << 16);
    }
    const int64_t row = (slot / p.block_size) * p.cache_stride + (slot % p.block_size) * kLatent;
    reinterpret_cast<uint4*>(p.cache + row)[lane] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
}

}  // namespace

cudaError_t launch_latent_write(const LatentWriteParams& p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    latent_write_kernel<<<(p.rows + kWriteWarps - 1) / kWriteWarps, kWriteWarps * 32, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dsa
