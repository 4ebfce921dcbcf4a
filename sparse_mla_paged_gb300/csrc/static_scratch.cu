// dsa_mla_decode_static: the decode with its scratch in a fixed, file-scope device array.
//
// Some callers cannot allocate device memory when they call the decode: for example code
// running inside a framework that owns every byte of device memory through its own pool,
// or a latency-critical serving path where cudaMalloc's device-wide synchronisation is not
// acceptable, and that also does not want to size and keep a workspace of its own. This
// entry point gives them the decode without any allocation: its scratch (the resolved
// ids, their byte offsets, the query operand images, the per-CTA partials and the status
// word) lives in g_scratch below, which every GPU that loads the library holds until the
// process exits. Calls never call cudaMalloc, cudaFree or any allocating routine.
//
// Host code cannot use g_scratch's name as an address (on the host it is only a stand-in
// for the symbol): the device address is looked up once per device with
// cudaGetSymbolAddress, on the first call made with that device current, and passed to
// the kernels. Because every call shares the one array, calls that overlap on the GPU
// (different streams, or different host threads) race on it and must be serialised by the
// caller. Each call rewrites every part of the array it later reads, and the status word
// is cleared at the start of every call, so nothing left by an earlier call leaks into a
// later one.
#include <mutex>
#include <vector>

#include "common.cuh"

namespace {

static __device__ __align__(256) uint8_t g_scratch[DSA_STATIC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
std::vector<void*> g_scratch_addr;  // device address of g_scratch, per device ordinal

// Device address of g_scratch on the current device (looked up on first use).
int32_t scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (static_cast<int>(g_scratch_addr.size()) <= dev) g_scratch_addr.resize(dev + 1, nullptr);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return DSA_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return DSA_OK;
}

}  // namespace

extern "C" int32_t dsa_mla_decode_static(const void* q, const void* k_cache, const void* v_cache,
                                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                                         const int32_t* seq_lens, const int32_t* sel_indices, int32_t sel_width,
                                         int32_t num_seqs, int32_t rows_per_seq, int32_t num_q_heads,
                                         int32_t block_size, int64_t cache_stride_bytes, float k_scale,
                                         float v_scale, float sm_scale, void* out, void* stream) {
    void* scratch = nullptr;
    const int32_t st = scratch_address(&scratch);
    if (st != DSA_OK) return st;
    // The workspace-taking path never allocates; a shape whose workspace exceeds the array
    // is rejected there with DSA_ERR_WORKSPACE before anything is enqueued.
    return dsa_mla_decode_ws(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, sel_indices,
                             sel_width, num_seqs, rows_per_seq, num_q_heads, block_size, cache_stride_bytes,
                             k_scale, v_scale, sm_scale, out, /*verify_rows=*/0, scratch, DSA_STATIC_SCRATCH_BYTES,
                             /*options=*/nullptr, stream);
}

// The status word of the latest static call is the first word of g_scratch; reading it
// back is a copy from the looked-up device address into the caller's variable.
extern "C" int32_t dsa_static_device_status(int32_t* status_out, void* stream) {
    if (!status_out) return DSA_ERR_INVALID_ARGUMENT;
    void* scratch = nullptr;
    const int32_t st = scratch_address(&scratch);
    if (st != DSA_OK) return st;
    return dsa_read_device_status(scratch, status_out, stream);
}
