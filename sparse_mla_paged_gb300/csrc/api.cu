// Host side of the C ABI declared in include/dsa_mla.h: argument checks, the work
// partition, workspace management and the launch sequence
//   prologue (index resolution + query split) -> decode -> combine (when needed),
// all enqueued on the caller's stream.
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"

using namespace dsa;

namespace {

struct DeviceState {
    bool checked = false;
    int32_t status = DSA_OK;  // result of the device check
    int sms = 0;
    size_t mem_bytes = 0;     // device memory size: bounds the rows a cache tensor map spans
    void* ws = nullptr;       // library-owned workspace
    size_t ws_bytes = 0;
};

std::mutex g_mu;
std::vector<DeviceState> g_devices;
#ifdef DSA_TRACE
unsigned long long* g_trace = nullptr;  // trace builds only: per-CTA decode timeline
#endif

struct Args {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    int32_t max_blocks_per_seq;
    const int32_t* seq_lens;
    const int32_t* sel;
    int32_t width, num_seqs, rows_per_seq, heads, block_size;
    int64_t stride;
    float k_scale, v_scale, sm_scale;
    void* out;
    int32_t verify_rows;
};

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int32_t check_args(const Args& a) {
    if (!a.q || !a.k_cache || !a.v_cache || !a.block_tables || !a.seq_lens || !a.sel || !a.out)
        return DSA_ERR_INVALID_ARGUMENT;
    if (a.num_seqs < 1 || a.rows_per_seq < 1 || a.heads < 1 || a.block_size < 1 || a.width < 1 ||
        a.max_blocks_per_seq < 0)
        return DSA_ERR_INVALID_ARGUMENT;
    if (a.stride < static_cast<int64_t>(a.block_size) * kLatent || a.stride % 16 != 0)
        return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned(a.q, 16) || !aligned(a.out, 16) || !aligned(a.k_cache, 16) || !aligned(a.v_cache, 16) ||
        !aligned(a.block_tables, 4) || !aligned(a.seq_lens, 4) || !aligned(a.sel, 4))
        return DSA_ERR_INVALID_ARGUMENT;
    if (a.verify_rows != 0 && a.verify_rows != 1) return DSA_ERR_INVALID_ARGUMENT;
    const int64_t rows = static_cast<int64_t>(a.num_seqs) * a.rows_per_seq;
    if (a.width > DSA_MAX_SEL_WIDTH) return DSA_ERR_UNSUPPORTED;
    if (rows > (1LL << 30) / a.width || rows * a.heads > (1LL << 31) / kLatent) return DSA_ERR_UNSUPPORTED;
    return DSA_OK;
}

int32_t from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return DSA_OK;
    if (e == cudaErrorNoKernelImageForDevice || e == cudaErrorInvalidDeviceFunction ||
        e == cudaErrorSharedObjectInitFailed)
        return DSA_ERR_NO_KERNEL;
    return DSA_ERR_CUDA;
}

// Checks the current device once (sm_103, kernels loadable) and returns its state.
int32_t current_device(DeviceState** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    if (static_cast<int>(g_devices.size()) <= dev) g_devices.resize(dev + 1);
    DeviceState& d = g_devices[dev];
    if (!d.checked) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return DSA_ERR_CUDA;
        d.sms = sms;
        size_t free_b = 0, total_b = 0;
        if (cudaMemGetInfo(&free_b, &total_b) != cudaSuccess) return DSA_ERR_CUDA;
        d.mem_bytes = total_b;
        if (major != 10 || minor != 3) {
            d.status = DSA_ERR_UNSUPPORTED;
        } else {
            d.status = from_cuda(decode_kernel_setup_64());
            if (d.status == DSA_OK) d.status = from_cuda(decode_kernel_setup_128());
            if (d.status == DSA_OK) d.status = from_cuda(prologue_kernel_setup());
            if (d.status == DSA_OK) d.status = from_cuda(combine_kernel_setup());
            if (d.status == DSA_OK) d.status = from_cuda(select_kernel_setup());
        }
        d.checked = true;
    }
    *out = &d;
    return d.status;
}

struct Plan {
    int64_t rows, groups, units;
    Partition part;
    bool any_split;
    bool small_tiles;  // 64-token tiles: at most two 128-slot tiles of work per CTA
    int max_pieces;    // most CTAs sharing one unit (selects the combine variant)
    WsLayout ws;
};

// Per-call choices (dsa_decode_options with its defaults filled in).
struct CallOptions {
    int32_t num_ctas = 0;
    int32_t tile_tokens = 0;
    int32_t gather_mode = 0;
    uint64_t wait_limit_ns = 0;
    cudaEvent_t ev0 = nullptr, ev1 = nullptr;
};

constexpr uint64_t kDefaultWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s

int32_t read_options(const dsa_decode_options* o, CallOptions* out) {
    CallOptions c;
    if (o) {
        if (o->num_ctas < 0) return DSA_ERR_INVALID_ARGUMENT;
        if (o->tile_tokens != 0 && o->tile_tokens != 64 && o->tile_tokens != 128) return DSA_ERR_INVALID_ARGUMENT;
        if (o->gather_mode < 0 || o->gather_mode > 2) return DSA_ERR_INVALID_ARGUMENT;
        if (o->reserved != 0) return DSA_ERR_INVALID_ARGUMENT;
        c.num_ctas = o->num_ctas;
        c.tile_tokens = o->tile_tokens;
        c.gather_mode = o->gather_mode;
        c.wait_limit_ns = o->wait_limit_ns;
        c.ev0 = static_cast<cudaEvent_t>(o->ev_begin);
        c.ev1 = static_cast<cudaEvent_t>(o->ev_end);
    }
    if (c.wait_limit_ns == 0) c.wait_limit_ns = kDefaultWaitLimitNs;
    *out = c;
    return DSA_OK;
}

// Default decode grid. At most one CTA per SM and at least kCtaMinSlots slots per CTA
// (c_max); within that, a grid aligned with the units is preferred: a CTA count that is a
// multiple of the unit count (every CTA's slots lie in one unit, each unit split into
// equal pieces) or divides it (every CTA takes whole units). Such a grid has no CTA that
// changes unit in mid-range and no unit that ends inside a CTA, which saves a unit change
// per CTA and, when each CTA takes whole units, the combine; measured on GB300 it beats an
// unaligned grid with up to a third more CTAs. The largest aligned count is taken when it
// is at least three quarters of c_max, else c_max.
int64_t default_grid(int64_t units, int64_t total_slots, int sms) {
    int64_t c_max = (total_slots + kCtaMinSlots - 1) / kCtaMinSlots;
    if (c_max > sms) c_max = sms;
    if (c_max < 1) c_max = 1;
    for (int64_t c = c_max; 4 * c >= 3 * c_max; --c)
        if (c % units == 0 || units % c == 0) return c;
    return c_max;
}

Plan make_plan(int64_t rows, int32_t heads, int32_t width, int32_t num_ctas, int sms, int32_t tile_tokens = 0) {
    Plan pl;
    pl.rows = rows;
    pl.groups = (heads + kHeadsPerCta - 1) / kHeadsPerCta;
    pl.units = rows * pl.groups;
    pl.part.total_slots = pl.units * width;
    pl.part.width = width;
    pl.part.groups = static_cast<int32_t>(pl.groups);
    int64_t c = num_ctas;
    if (c <= 0) c = default_grid(pl.units, pl.part.total_slots, sms);
    pl.part.ctas = static_cast<int32_t>(c);
    pl.part.narrow = pl.part.total_slots * (c + 1) < (int64_t{1} << 32) ? 1 : 0;
    pl.small_tiles = tile_tokens == 0 ? pl.part.total_slots <= 2 * kCtaMinSlots * c : tile_tokens == 64;
    pl.any_split = false;
    for (int64_t k = 1; k < c && !pl.any_split; ++k)
        if (cta_begin(pl.part, k) % width != 0) pl.any_split = true;
    pl.max_pieces = static_cast<int>(std::min<int64_t>(max_pieces_per_unit(pl.part), 1 << 20));
    pl.ws = ws_layout(rows, pl.groups, width, c);
    return pl;
}

// cuTensorMapEncodeTiled from the driver, looked up once.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            f = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    }();
    return fn;
}

// 2-D map of a dense cache: rows of 512 bytes (row = page*block_size + slot), enough rows
// to span the device's memory from the cache's base, read as boxes of 128 bytes x 1 row
// into the 128-byte-swizzled operand layout; rows past the map are zero-filled.
bool encode_cache_map(const void* base, size_t mem_bytes, CUtensorMap* m) {
    const auto fn = tensor_map_encoder();
    if (!fn) return false;
    const cuuint64_t rows = std::min<cuuint64_t>(mem_bytes / kLatent + 1, (1ull << 31) - 1);
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(kLatent), rows};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(kLatent)};
    const cuuint32_t box[2] = {128, 1};
    const cuuint32_t estride[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estride,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int32_t enqueue(const Args& a, const Plan& pl, uint8_t* ws, const CallOptions& opt, size_t mem_bytes,
                cudaStream_t stream) {
    const cudaEvent_t ev0 = opt.ev0, ev1 = opt.ev1;
    PrologueParams pp{};
    pp.sel = a.sel;
    pp.seq_lens = a.seq_lens;
    pp.q = static_cast<const uint16_t*>(a.q);
    pp.block_tables = a.block_tables;
    pp.offs = reinterpret_cast<long long*>(ws + pl.ws.offs);
    pp.cache_stride = a.stride;
    pp.block_size = a.block_size;
    pp.block_shift = -1;
    for (int s = 0; s < 31; ++s)
        if ((1 << s) == a.block_size) pp.block_shift = s;
    pp.max_blocks_per_seq = a.max_blocks_per_seq;
    pp.ids = nullptr;
    pp.cnt = reinterpret_cast<int32_t*>(ws + pl.ws.cnt);
    pp.qimg = ws + pl.ws.qimg;
    pp.qscale = reinterpret_cast<float*>(ws + pl.ws.qscale);
    pp.status = reinterpret_cast<int*>(ws + pl.ws.status);
    pp.rows = static_cast<int32_t>(pl.rows);
    pp.width = a.width;
    pp.heads = a.heads;
    pp.groups = static_cast<int32_t>(pl.groups);
    pp.rows_per_seq = a.rows_per_seq;
    pp.verify_rows = a.verify_rows;
    pp.score_scale = a.sm_scale * a.k_scale * 1.4426950408889634f;
    const bool early = pl.part.total_slots >= kEarlyDependentSlots * pl.part.ctas;
    int32_t st = from_cuda(launch_prologue(pp, static_cast<int>(pl.rows + pl.units), early, stream));
    if (st != DSA_OK) return st;

    DecodeParams dp{};
    dp.k_cache = static_cast<const uint8_t*>(a.k_cache);
    dp.v_cache = static_cast<const uint8_t*>(a.v_cache);
    dp.offs = pp.offs;
    dp.cnt = pp.cnt;
    dp.qimg = pp.qimg;
    dp.qscale = pp.qscale;
    dp.out = static_cast<uint16_t*>(a.out);
    dp.part_o = reinterpret_cast<uint16_t*>(ws + pl.ws.part_o);
    dp.part_lse = reinterpret_cast<float*>(ws + pl.ws.part_lse);
    dp.status = pp.status;
    dp.part = pl.part;
    dp.heads = a.heads;
    dp.kv_same = a.k_cache == a.v_cache ? 1 : 0;
    dp.v_scale = a.v_scale;
    dp.early_dependents = early ? 1 : 0;
    dp.wait_limit_ns = opt.wait_limit_ns;
    // Tensor-map gathers (on request) need rows of one uniform stride (dense pages) and
    // 128-byte aligned caches; anything else takes the per-thread copies.
    CUtensorMap kmap, vmap;
    std::memset(&kmap, 0, sizeof kmap);
    std::memset(&vmap, 0, sizeof vmap);
    dp.use_tma = 0;
    if (opt.gather_mode == 2 && a.stride == static_cast<int64_t>(a.block_size) * kLatent && aligned(a.k_cache, 128) &&
        aligned(a.v_cache, 128) && encode_cache_map(a.k_cache, mem_bytes, &kmap) &&
        (dp.kv_same || encode_cache_map(a.v_cache, mem_bytes, &vmap)))
        dp.use_tma = 1;
#ifdef DSA_TRACE
    dp.trace = g_trace;
#endif
    // Inside stream capture the records must be external, so that they become event-record
    // nodes of the graph; outside capture they are plain records.
    unsigned int ev_flags = cudaEventRecordDefault;
    if (ev0 || ev1) {
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return DSA_ERR_CUDA;
        if (cs == cudaStreamCaptureStatusActive) ev_flags = cudaEventRecordExternal;
    }
    if (ev0 && cudaEventRecordWithFlags(ev0, stream, ev_flags) != cudaSuccess) return DSA_ERR_CUDA;
    // With K and V in separate buffers a ring slot holds both tiles, so 128-token tiles would
    // leave a single slot and no pipelining: such calls take 64-token tiles (three slots)
    // unless the caller fixed the tile size (measured on ragged: 85 against 46 us per call).
    const bool small = pl.small_tiles || (opt.tile_tokens == 0 && !dp.kv_same);
    st = from_cuda(small ? launch_decode_64(dp, kmap, vmap, stream) : launch_decode_128(dp, kmap, vmap, stream));
    if (st != DSA_OK) return st;
    if (ev1 && cudaEventRecordWithFlags(ev1, stream, ev_flags) != cudaSuccess) return DSA_ERR_CUDA;

    if (pl.any_split) {
        CombineParams cp{};
        cp.part_o = dp.part_o;
        cp.part_lse = dp.part_lse;
        cp.out = dp.out;
        cp.part = pl.part;
        cp.heads = a.heads;
        cp.v_scale = a.v_scale;
        cp.early_dependents = dp.early_dependents;
        st = from_cuda(launch_combine(cp, static_cast<int>(pl.units), pl.max_pieces, stream));
    }
    return st;
}

int32_t run_ws(const Args& a, void* workspace, size_t workspace_bytes, const dsa_decode_options* options,
               cudaStream_t stream) {
    int32_t st = check_args(a);
    if (st != DSA_OK) return st;
    CallOptions opt;
    st = read_options(options, &opt);
    if (st != DSA_OK) return st;
    if (!workspace || !aligned(workspace, 256)) return DSA_ERR_INVALID_ARGUMENT;
    DeviceState* d = nullptr;
    st = current_device(&d);
    if (st != DSA_OK) return st;
    const Plan pl = make_plan(static_cast<int64_t>(a.num_seqs) * a.rows_per_seq, a.heads, a.width, opt.num_ctas,
                              d->sms, opt.tile_tokens);
    if (workspace_bytes < pl.ws.total) return DSA_ERR_WORKSPACE;
    return enqueue(a, pl, static_cast<uint8_t*>(workspace), opt, d->mem_bytes, stream);
}

int32_t run_lib(const Args& a, cudaStream_t stream) {
    int32_t st = check_args(a);
    if (st != DSA_OK) return st;
    DeviceState* d = nullptr;
    st = current_device(&d);
    if (st != DSA_OK) return st;
    const Plan pl = make_plan(static_cast<int64_t>(a.num_seqs) * a.rows_per_seq, a.heads, a.width, 0, d->sms);
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        if (d->ws_bytes < pl.ws.total) {
            cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
            if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return DSA_ERR_CUDA;
            if (cs != cudaStreamCaptureStatusNone) return DSA_ERR_WORKSPACE;
            if (d->ws) {
                if (cudaStreamSynchronize(stream) != cudaSuccess) return DSA_ERR_CUDA;
                cudaFree(d->ws);
                d->ws = nullptr;
                d->ws_bytes = 0;
            }
            const size_t want = pl.ws.total + pl.ws.total / 4;
            if (cudaMalloc(&d->ws, want) != cudaSuccess) return DSA_ERR_CUDA;
            if (cudaMemset(d->ws, 0, 256) != cudaSuccess) return DSA_ERR_CUDA;
            d->ws_bytes = want;
        }
        ws = d->ws;
    }
    CallOptions opt;
    read_options(nullptr, &opt);
    return enqueue(a, pl, static_cast<uint8_t*>(ws), opt, d->mem_bytes, stream);
}

Args make_args(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
               int32_t max_blocks_per_seq, const int32_t* seq_lens, const int32_t* sel, int32_t width,
               int32_t num_seqs, int32_t rows_per_seq, int32_t heads, int32_t block_size, int64_t stride,
               float k_scale, float v_scale, float sm_scale, void* out, int32_t verify_rows) {
    Args a;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.seq_lens = seq_lens;
    a.sel = sel;
    a.width = width;
    a.num_seqs = num_seqs;
    a.rows_per_seq = rows_per_seq;
    a.heads = heads;
    a.block_size = block_size;
    a.stride = stride;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.sm_scale = sm_scale;
    a.out = out;
    a.verify_rows = verify_rows;
    return a;
}

}  // namespace

// The device check shared with the other translation units (the absorb transforms).
int32_t dsa::check_device() {
    DeviceState* d = nullptr;
    return current_device(&d);
}

extern "C" {

#ifdef DSA_TRACE
void dsa_debug_set_trace(void* buffer) { g_trace = static_cast<unsigned long long*>(buffer); }
#endif

int32_t dsa_abi_version(void) { return 2; }

const char* dsa_status_string(int32_t status) {
    switch (status) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARGUMENT: return "invalid argument";
        case DSA_ERR_UNSUPPORTED: return "unsupported device or size";
        case DSA_ERR_WORKSPACE: return "workspace too small or growth during graph capture";
        case DSA_ERR_CUDA: return "CUDA runtime error";
        case DSA_ERR_NO_KERNEL: return "sm_103a kernel image missing for this device";
        case DSA_ERR_DEVICE_BOUNDS: return "device: page lookup outside the block table";
        case DSA_ERR_TIMEOUT: return "device: pipeline wait timed out";
        default: return "unknown status";
    }
}

int32_t dsa_mla_decode(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                       int32_t max_blocks_per_seq, const int32_t* seq_lens, const int32_t* sel_indices,
                       int32_t sel_width, int32_t num_seqs, int32_t rows_per_seq, int32_t num_q_heads,
                       int32_t block_size, int64_t cache_stride_bytes, float k_scale, float v_scale,
                       float sm_scale, void* out, void* stream) {
    return run_lib(make_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, sel_indices,
                             sel_width, num_seqs, rows_per_seq, num_q_heads, block_size, cache_stride_bytes,
                             k_scale, v_scale, sm_scale, out, 0),
                   static_cast<cudaStream_t>(stream));
}

int32_t dsa_mla_decode_k(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                         int32_t max_blocks_per_seq, const int32_t* seq_lens, const int32_t* sel_indices,
                         int32_t sel_width, int32_t num_seqs, int32_t k, int32_t num_q_heads, int32_t block_size,
                         int64_t cache_stride_bytes, float k_scale, float v_scale, float sm_scale, void* out,
                         void* stream) {
    return run_lib(make_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, sel_indices,
                             sel_width, num_seqs, k, num_q_heads, block_size, cache_stride_bytes, k_scale,
                             v_scale, sm_scale, out, 1),
                   static_cast<cudaStream_t>(stream));
}

size_t dsa_mla_decode_workspace_bytes(int32_t num_seqs, int32_t rows_per_seq, int32_t num_q_heads,
                                      int32_t sel_width, int32_t num_ctas) {
    if (num_seqs < 1 || rows_per_seq < 1 || num_q_heads < 1 || sel_width < 1 || num_ctas < 0) return 0;
    int sms = 0;
    if (num_ctas == 0) {
        DeviceState* d = nullptr;
        if (current_device(&d) != DSA_OK) return 0;
        sms = d->sms;
    }
    return make_plan(static_cast<int64_t>(num_seqs) * rows_per_seq, num_q_heads, sel_width, num_ctas, sms).ws.total;
}

int32_t dsa_mla_decode_grid(int32_t num_seqs, int32_t rows_per_seq, int32_t num_q_heads, int32_t sel_width,
                            int32_t num_ctas) {
    if (num_seqs < 1 || rows_per_seq < 1 || num_q_heads < 1 || sel_width < 1 || num_ctas < 0) return 0;
    int sms = 0;
    if (num_ctas == 0) {
        DeviceState* d = nullptr;
        if (current_device(&d) != DSA_OK) return 0;
        sms = d->sms;
    }
    return make_plan(static_cast<int64_t>(num_seqs) * rows_per_seq, num_q_heads, sel_width, num_ctas, sms).part.ctas;
}

int32_t dsa_mla_decode_ws(const void* q, const void* k_cache, const void* v_cache, const int32_t* block_tables,
                          int32_t max_blocks_per_seq, const int32_t* seq_lens, const int32_t* sel_indices,
                          int32_t sel_width, int32_t num_seqs, int32_t rows_per_seq, int32_t num_q_heads,
                          int32_t block_size, int64_t cache_stride_bytes, float k_scale, float v_scale,
                          float sm_scale, void* out, int32_t verify_rows, void* workspace, size_t workspace_bytes,
                          const dsa_decode_options* options, void* stream) {
    return run_ws(make_args(q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, sel_indices,
                            sel_width, num_seqs, rows_per_seq, num_q_heads, block_size, cache_stride_bytes,
                            k_scale, v_scale, sm_scale, out, verify_rows),
                  workspace, workspace_bytes, options, static_cast<cudaStream_t>(stream));
}

namespace {
struct HostStaging {
    size_t q, bt, sl, sel, out, total;
};
HostStaging host_staging(size_t base, int64_t rows, int32_t heads, int32_t width, int32_t table_rows,
                         int32_t mbps, int32_t num_seqs, int32_t verify_rows) {
    HostStaging h;
    size_t o = align256(base);
    h.q = o; o = align256(o + static_cast<size_t>(rows) * heads * kLatent * 2);
    h.bt = o; o = align256(o + static_cast<size_t>(table_rows) * (mbps > 0 ? mbps : 1) * 4);
    h.sl = o; o = align256(o + static_cast<size_t>(verify_rows ? num_seqs : rows) * 4);
    h.sel = o; o = align256(o + static_cast<size_t>(rows) * width * 4);
    h.out = o; o = align256(o + static_cast<size_t>(rows) * heads * kLatent * 2);
    h.total = o;
    return h;
}
}  // namespace

size_t dsa_mla_decode_host_workspace_bytes(int32_t num_seqs, int32_t rows_per_seq, int32_t num_q_heads,
                                           int32_t sel_width, int32_t table_rows, int32_t max_blocks_per_seq,
                                           int32_t verify_rows, int32_t num_ctas) {
    const size_t base = dsa_mla_decode_workspace_bytes(num_seqs, rows_per_seq, num_q_heads, sel_width, num_ctas);
    if (base == 0 || table_rows < 1 || max_blocks_per_seq < 0) return 0;
    return host_staging(base, static_cast<int64_t>(num_seqs) * rows_per_seq, num_q_heads, sel_width, table_rows,
                        max_blocks_per_seq, num_seqs, verify_rows)
        .total;
}

int32_t dsa_mla_decode_host(const void* q_host, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables_host, int32_t table_rows, int32_t max_blocks_per_seq,
                            const int32_t* seq_lens_host, const int32_t* sel_indices_host, int32_t sel_width,
                            int32_t num_seqs, int32_t rows_per_seq, int32_t num_q_heads, int32_t block_size,
                            int64_t cache_stride_bytes, float k_scale, float v_scale, float sm_scale,
                            void* out_host, int32_t verify_rows, void* workspace, size_t workspace_bytes,
                            int32_t num_ctas, void* stream) {
    if (!q_host || !block_tables_host || !seq_lens_host || !sel_indices_host || !out_host || table_rows < 1 ||
        !workspace || !aligned(workspace, 256))
        return DSA_ERR_INVALID_ARGUMENT;
    // Validate the shape with the device staging pointers standing in for the host ones.
    Args probe = make_args(workspace, k_cache, v_cache, reinterpret_cast<const int32_t*>(workspace),
                           max_blocks_per_seq, reinterpret_cast<const int32_t*>(workspace),
                           reinterpret_cast<const int32_t*>(workspace), sel_width, num_seqs, rows_per_seq,
                           num_q_heads, block_size, cache_stride_bytes, k_scale, v_scale, sm_scale, workspace,
                           verify_rows);
    int32_t st = check_args(probe);
    if (st != DSA_OK) return st;
    DeviceState* d = nullptr;
    st = current_device(&d);
    if (st != DSA_OK) return st;
    const int64_t rows = static_cast<int64_t>(num_seqs) * rows_per_seq;
    const Plan pl = make_plan(rows, num_q_heads, sel_width, num_ctas, d->sms);
    const HostStaging hs = host_staging(pl.ws.total, rows, num_q_heads, sel_width, table_rows, max_blocks_per_seq,
                                        num_seqs, verify_rows);
    if (workspace_bytes < hs.total) return DSA_ERR_WORKSPACE;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const size_t qb = static_cast<size_t>(rows) * num_q_heads * kLatent * 2;
    const size_t btb = static_cast<size_t>(table_rows) * (max_blocks_per_seq > 0 ? max_blocks_per_seq : 1) * 4;
    const size_t slb = static_cast<size_t>(verify_rows ? num_seqs : rows) * 4;
    const size_t selb = static_cast<size_t>(rows) * sel_width * 4;
    if (cudaMemcpyAsync(ws + hs.q, q_host, qb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(ws + hs.bt, block_tables_host, btb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(ws + hs.sl, seq_lens_host, slb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(ws + hs.sel, sel_indices_host, selb, cudaMemcpyHostToDevice, s) != cudaSuccess)
        return DSA_ERR_CUDA;
    Args a = make_args(ws + hs.q, k_cache, v_cache, reinterpret_cast<const int32_t*>(ws + hs.bt),
                       max_blocks_per_seq, reinterpret_cast<const int32_t*>(ws + hs.sl),
                       reinterpret_cast<const int32_t*>(ws + hs.sel), sel_width, num_seqs, rows_per_seq,
                       num_q_heads, block_size, cache_stride_bytes, k_scale, v_scale, sm_scale, ws + hs.out,
                       verify_rows);
    CallOptions opt;
    read_options(nullptr, &opt);
    st = enqueue(a, pl, ws, opt, d->mem_bytes, s);
    if (st != DSA_OK) return st;
    if (cudaMemcpyAsync(out_host, ws + hs.out, qb, cudaMemcpyDeviceToHost, s) != cudaSuccess) return DSA_ERR_CUDA;
    return DSA_OK;
}

int32_t dsa_resolve_indices(const int32_t* sel_indices, const int32_t* seq_lens, int32_t sel_width, int32_t rows,
                            int32_t* ids_out, int32_t* counts_out, void* stream) {
    if (!sel_indices || !seq_lens || !ids_out || !counts_out || sel_width < 1 || rows < 1)
        return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned(sel_indices, 4) || !aligned(seq_lens, 4) || !aligned(ids_out, 4) || !aligned(counts_out, 4))
        return DSA_ERR_INVALID_ARGUMENT;
    if (sel_width > DSA_MAX_SEL_WIDTH) return DSA_ERR_UNSUPPORTED;
    DeviceState* d = nullptr;
    int32_t st = current_device(&d);
    if (st != DSA_OK) return st;
    PrologueParams pp{};
    pp.sel = sel_indices;
    pp.seq_lens = seq_lens;
    pp.ids = ids_out;
    pp.cnt = counts_out;
    pp.rows = rows;
    pp.width = sel_width;
    pp.heads = 1;
    pp.groups = 1;
    pp.rows_per_seq = 1;
    return from_cuda(launch_prologue(pp, rows, false, static_cast<cudaStream_t>(stream)));
}

int32_t dsa_latent_write(const void* kv_a, const void* norm_weight, const int64_t* slots, int32_t rows,
                         float rms_eps, float kv_scale, int32_t block_size, int64_t cache_stride_bytes, void* cache,
                         void* stream) {
    if (!norm_weight || !cache || rows < 0 || block_size < 1) return DSA_ERR_INVALID_ARGUMENT;
    if (rows > 0 && (!kv_a || !slots)) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned(kv_a, 16) || !aligned(norm_weight, 16) || !aligned(slots, 8) || !aligned(cache, 16))
        return DSA_ERR_INVALID_ARGUMENT;
    if (cache_stride_bytes < static_cast<int64_t>(block_size) * kLatent || cache_stride_bytes % 16 != 0)
        return DSA_ERR_INVALID_ARGUMENT;
    if (!(rms_eps >= 0.0f) || !std::isfinite(rms_eps) || !std::isfinite(kv_scale) || kv_scale == 0.0f)
        return DSA_ERR_INVALID_ARGUMENT;
    if (rows == 0) return DSA_OK;
    DeviceState* d = nullptr;
    int32_t st = current_device(&d);
    if (st != DSA_OK) return st;
    LatentWriteParams p{};
    p.kv_a = static_cast<const uint16_t*>(kv_a);
    p.weight = static_cast<const uint16_t*>(norm_weight);
    p.slots = reinterpret_cast<const long long*>(slots);
    p.cache = static_cast<uint8_t*>(cache);
    p.cache_stride = cache_stride_bytes;
    p.rows = rows;
    p.block_size = block_size;
    p.eps = rms_eps;
    p.inv_scale = 1.0f / kv_scale;  // formed in single precision, as the pages' launcher does
    return from_cuda(launch_latent_write(p, static_cast<cudaStream_t>(stream)));
}

int32_t dsa_select_pools(const float* scores, const int32_t* q_pos, int32_t rows, int32_t n_pools, int32_t kpool,
                         int32_t topk, int32_t* ids_out, void* stream) {
    if (rows < 0 || n_pools < 0 || kpool < 1 || topk < 1) return DSA_ERR_INVALID_ARGUMENT;
    if (rows > 0 && (!q_pos || !ids_out || (n_pools > 0 && !scores))) return DSA_ERR_INVALID_ARGUMENT;
    if (!aligned(scores, 4) || !aligned(q_pos, 4) || !aligned(ids_out, 4)) return DSA_ERR_INVALID_ARGUMENT;
    if (static_cast<int64_t>(n_pools) * kpool > INT32_MAX || static_cast<int64_t>(topk) * kpool > INT32_MAX)
        return DSA_ERR_UNSUPPORTED;
    if (rows == 0) return DSA_OK;
    DeviceState* d = nullptr;
    int32_t st = current_device(&d);
    if (st != DSA_OK) return st;
    SelectParams p{};
    p.scores = scores;
    p.q_pos = q_pos;
    p.ids = ids_out;
    p.rows = rows;
    p.n_pools = n_pools;
    p.kpool = kpool;
    p.topk = topk;
    return from_cuda(launch_select(p, static_cast<cudaStream_t>(stream)));
}

int32_t dsa_read_device_status(const void* workspace, int32_t* status_out, void* stream) {
    if (!workspace || !status_out) return DSA_ERR_INVALID_ARGUMENT;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaStreamSynchronize(s) != cudaSuccess)
        return DSA_ERR_CUDA;
    *status_out = v;
    return DSA_OK;
}

int32_t dsa_last_device_status(int32_t* status_out, void* stream) {
    if (!status_out) return DSA_ERR_INVALID_ARGUMENT;
    DeviceState* d = nullptr;
    int32_t st = current_device(&d);
    if (st != DSA_OK) return st;
    void* ws = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        ws = d->ws;
    }
    if (!ws) {
        *status_out = DSA_OK;
        return DSA_OK;
    }
    return dsa_read_device_status(ws, status_out, stream);
}

}  // extern "C"
