// The cache writer (decode_k.rs, decode_k: the latent_write launch): for each new token,
//   y[c] = x[c] / sqrt(mean_c x^2 + eps) * w[c] * (1/kv_scale),
// stored as E4M3 (round to nearest even, saturating to +-448) in the token's 512-byte
// row at (slot / block_size)*cache_stride_bytes + (slot % block_size)*512, where the
// decode reads it; slot = physical*block_size + pos % block_size. The pages launch one
// block of kv_lora_rank threads per token and do not show its body; the RMSNorm-then-scale
// order above is the plain reading.
//
// One block of 128 threads per token, 4 dims per thread: 8-byte loads of kv_a and of the
// weight, a block-wide sum of squares in FP32, one 4-byte store of four codes.
#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kWriteThreads = kLatent / 4;  // 128

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__global__ void __launch_bounds__(kWriteThreads) latent_write_kernel(const LatentWriteParams p) {
    __shared__ float part[kWriteThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t r = blockIdx.x;
    const long long slot = p.slots[r];
    if (slot < 0) return;  // the whole block: nothing to write for this row
    const uint2 xr = reinterpret_cast<const uint2*>(p.kv_a + r * kLatent)[tid];
    const uint2 wr = reinterpret_cast<const uint2*>(p.weight)[tid];
    const float x[4] = {bf16_lo(xr.x), bf16_hi(xr.x), bf16_lo(xr.y), bf16_hi(xr.y)};
    const float w[4] = {bf16_lo(wr.x), bf16_hi(wr.x), bf16_lo(wr.y), bf16_hi(wr.y)};
    float ss = (x[0] * x[0] + x[1] * x[1]) + (x[2] * x[2] + x[3] * x[3]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (lane == 0) part[warp] = ss;
    __syncthreads();
    const float total = (part[0] + part[1]) + (part[2] + part[3]);
    const float inv_rms = rsqrtf(total * (1.0f / kLatent) + p.eps);
    float y[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) y[k] = x[k] * inv_rms * w[k] * p.inv_scale;
    const uint32_t codes = f32x2_to_e4m3x2(y[0], y[1]) | (f32x2_to_e4m3x2(y[2], y[3]) << 16);
    const int64_t row = (slot / p.block_size) * p.cache_stride + (slot % p.block_size) * kLatent;
    *reinterpret_cast<uint32_t*>(p.cache + row + 4 * tid) = codes;
}

}  // namespace

cudaError_t launch_latent_write(const LatentWriteParams& p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    latent_write_kernel<<<p.rows, kWriteThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dsa
