// Load-time transforms of absorbed MLA (build.rs: absorb_q, absorb_o). Each is one
// strided-batched GEMM over the heads on the tensor cores through cuBLAS (a plain library
// contraction; nothing around it to fuse): BF16 weights as stored in the checkpoint, FP32
// accumulation, FP32 or BF16 (round to nearest even) output.
//
//   q_absorb[h*kvl + c][k] = sum_{r < nope} kv_b[h*(nope+vd) + r][c] * q_b[h*nope + r][k]
//   o_absorb[i][h*kvl + c] = sum_{r < vd} o_proj[i][h*vd + r] * kv_b[h*(nope+vd) + nope + r][c]
//
// All matrices are row-major. In cuBLAS's column-major terms, head h of absorb_q is
// C[ql x kvl] = Q_h[ql x nope] * K_h^T with K_h the [kvl x nope] column-major view of the
// head's K rows of kv_b, and head h of absorb_o is C[kvl x hidden] = V_h[kvl x vd] * O_h[vd x
// hidden], V_h the column-major view of the head's V rows and O_h the head's columns of
// o_proj; the heads' C blocks interleave (leading dimension heads*kvl) without overlapping.
#include <cublas_v2.h>

#include <climits>
#include <mutex>
#include <vector>

#include "common.cuh"

namespace {

std::mutex g_blas_mu;
std::vector<cublasHandle_t> g_handles;  // one per device, created on first use

int32_t from_blas(cublasStatus_t s) {
    if (s == CUBLAS_STATUS_SUCCESS) return DSA_OK;
    if (s == CUBLAS_STATUS_NOT_SUPPORTED || s == CUBLAS_STATUS_ARCH_MISMATCH) return DSA_ERR_UNSUPPORTED;
    if (s == CUBLAS_STATUS_INVALID_VALUE) return DSA_ERR_INVALID_ARGUMENT;
    return DSA_ERR_CUDA;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Runs f(handle) with the current device's handle bound to `stream`, under the lock (a
// cuBLAS handle is not safe to share between threads).
template <class F>
int32_t with_handle(void* stream, F&& f) {
    int32_t st = dsa::check_device();
    if (st != DSA_OK) return st;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_blas_mu);
    if (static_cast<int>(g_handles.size()) <= dev) g_handles.resize(dev + 1, nullptr);
    if (g_handles[dev] == nullptr) {
        cublasHandle_t h = nullptr;
        if (cublasCreate(&h) != CUBLAS_STATUS_SUCCESS) return DSA_ERR_CUDA;
        g_handles[dev] = h;
    }
    cublasHandle_t h = g_handles[dev];
    st = from_blas(cublasSetStream(h, static_cast<cudaStream_t>(stream)));
    if (st != DSA_OK) return st;
    return from_blas(f(h));
}

int32_t check_sizes(const void* a, const void* kv_b, void* out, int32_t heads, int32_t nope, int32_t vd,
                    int32_t kvl, int32_t other, int32_t out_dtype) {
    if (!a || !kv_b || !out || heads < 1 || nope < 1 || vd < 1 || kvl < 1 || other < 1) return DSA_ERR_INVALID_ARGUMENT;
    if (out_dtype != 0 && out_dtype != 1) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned(a, 2) || !aligned(kv_b, 2) || !aligned(out, out_dtype == 0 ? 4 : 2)) return DSA_ERR_INVALID_ARGUMENT;
    // cuBLAS takes dimensions and leading dimensions as int.
    const int64_t h = heads;
    if (h * (nope + vd) > INT_MAX || h * kvl > INT_MAX || h * vd > INT_MAX) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

}  // namespace

extern "C" {

int32_t dsa_absorb_q(const void* q_b, const void* kv_b, int32_t heads, int32_t nope, int32_t vd, int32_t kvl,
                     int32_t q_lora_rank, void* out, int32_t out_dtype, void* stream) {
    int32_t st = check_sizes(q_b, kv_b, out, heads, nope, vd, kvl, q_lora_rank, out_dtype);
    if (st != DSA_OK) return st;
    const int64_t ql = q_lora_rank;
    return with_handle(stream, [&](cublasHandle_t h) {
        const float one = 1.0f, zero = 0.0f;
        return cublasGemmStridedBatchedEx(
            h, CUBLAS_OP_N, CUBLAS_OP_T, static_cast<int>(ql), kvl, nope, &one,
            q_b, CUDA_R_16BF, static_cast<int>(ql), static_cast<long long>(nope) * ql,
            kv_b, CUDA_R_16BF, kvl, static_cast<long long>(nope + vd) * kvl, &zero,
            out, out_dtype == 0 ? CUDA_R_32F : CUDA_R_16BF, static_cast<int>(ql), static_cast<long long>(kvl) * ql,
            heads, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
    });
}

int32_t dsa_absorb_o(const void* o_proj, const void* kv_b, int32_t heads, int32_t nope, int32_t vd, int32_t kvl,
                     int32_t hidden, void* out, int32_t out_dtype, void* stream) {
    int32_t st = check_sizes(o_proj, kv_b, out, heads, nope, vd, kvl, hidden, out_dtype);
    if (st != DSA_OK) return st;
    const size_t esz = 2;  // BF16 kv_b
    const void* v_half = static_cast<const uint8_t*>(kv_b) + static_cast<size_t>(nope) * kvl * esz;
    return with_handle(stream, [&](cublasHandle_t h) {
        const float one = 1.0f, zero = 0.0f;
        return cublasGemmStridedBatchedEx(
            h, CUBLAS_OP_N, CUBLAS_OP_N, kvl, hidden, vd, &one,
            v_half, CUDA_R_16BF, kvl, static_cast<long long>(nope + vd) * kvl,
            o_proj, CUDA_R_16BF, heads * vd, static_cast<long long>(vd), &zero,
            out, out_dtype == 0 ? CUDA_R_32F : CUDA_R_16BF, heads * kvl, static_cast<long long>(kvl),
            heads, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
    });
}

}  // extern "C"
