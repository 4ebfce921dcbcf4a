// Shared definitions of the decode library: tile geometry, kernel parameter blocks,
// workspace layout and the static work partition. Host and device code both use the
// partition helpers, so the decode kernel and the combine kernel agree on it exactly.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "dsa_mla.h"

namespace dsa {

constexpr int kLatent = 512;           // kv_lora_rank: the whole cache token (NoPE)
constexpr int kCtaMinSlots = 128;      // default grid: at least this many slots per CTA
// From this many slots per decode CTA on, the decode and combine kernels let the next
// kernel on the stream launch early (measured: a gain on long decodes, a loss on short).
constexpr int64_t kEarlyDependentSlots = 2048;
constexpr int kHeadsPerCta = 64;       // query heads per work unit
// Query operand image of one unit: 128 rows of 512 E4M3 codes, row 32*q + 2*k + t holding
// term t (0 = hi, 1 = lo) of head 16*q + k, dims in natural order.
constexpr int kQImageBytes = 2 * kHeadsPerCta * kLatent;  // 64 KB
constexpr int kBitmapWords = 8192;     // resolve bitmap: seq_len up to 262144 tokens
constexpr int kResolveThreads = 256;

// Probabilities are carried as P' = 2^(x - m + kPBias) (x, m in log2 units) split into two
// E4M3 terms. A head's reference m is reset to its tile max plus kRescaleSlack when the
// tile max exceeds m by more than kRescaleMargin (so P' stays below
// 2^(kPBias + kRescaleMargin) < 448, the E4M3 maximum) and also when the tile max falls
// more than kRescaleDrop below m (so a tile far under an earlier maximum gets its own
// exponent window instead of sinking into E4M3's subnormal range and below it). A
// downward reset never takes m more than kRescaleFloor below the highest reference of the
// head, which keeps the rescaled FP32 accumulator far from overflow.
constexpr float kPBias = 7.0f;
constexpr float kRescaleMargin = 1.75f;
constexpr float kRescaleSlack = 1.0f;
constexpr float kRescaleDrop = 8.0f;
constexpr float kRescaleFloor = 64.0f;

// Device status codes mirror dsa_status.
constexpr int kStatusBounds = DSA_ERR_DEVICE_BOUNDS;
constexpr int kStatusTimeout = DSA_ERR_TIMEOUT;

// ------------------------------------------------------------------------------------
// Workspace layout (all offsets 256-byte aligned).
// ------------------------------------------------------------------------------------
struct WsLayout {
    size_t status, offs, cnt, qimg, qscale, part_o, part_lse, total;
};

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

__host__ __device__ inline WsLayout ws_layout(int64_t rows, int64_t groups, int64_t width, int64_t ctas) {
    WsLayout L;
    size_t o = 0;
    L.status = o; o += 256;
    L.offs = o; o = align256(o + static_cast<size_t>(rows * width) * 8);
    L.cnt = o; o = align256(o + static_cast<size_t>(rows) * 4);
    L.qimg = o; o = align256(o + static_cast<size_t>(rows * groups) * kQImageBytes);
    L.qscale = o; o = align256(o + static_cast<size_t>(rows * groups) * kHeadsPerCta * 4);
    L.part_o = o; o = align256(o + static_cast<size_t>(2 * ctas) * kHeadsPerCta * kLatent * 2);
    L.part_lse = o; o = align256(o + static_cast<size_t>(2 * ctas) * kHeadsPerCta * 4);
    L.total = o;
    return L;
}

// ------------------------------------------------------------------------------------
// Static work partition.
//
// A work unit is (row r, head group g) with sel_width "slots"; units are ordered
// u = r*groups + g. The concatenated slot space [0, T), T = units*sel_width, is cut into
// num_ctas contiguous ranges [c*T/C, (c+1)*T/C). A unit's slot range [s0, s1) maps to
// positions [min(s0, U), min(s1, U)) of that row's resolved list (U = resolved count), so
// ranges of neighbouring CTAs abut exactly whatever U is, and a CTA can request its
// first tokens before it knows U. A unit covered by one CTA is written
// straight to the output; a unit shared by several CTAs leaves per-CTA partials (slot
// 2c for the CTA's first unit, 2c+1 for its last) that the combine kernel merges.
// ------------------------------------------------------------------------------------
struct Partition {
    int64_t total_slots;  // T
    int32_t width;        // W
    int32_t ctas;         // C
    int32_t groups;       // G
    int32_t narrow;       // T*(C+1) < 2^32: the combine kernel divides in 32 bits
};

__host__ __device__ inline int64_t cta_begin(const Partition& p, int64_t c) {
    return c * p.total_slots / p.ctas;
}
// The CTA whose range holds slot x (the last one starting at or before x).
__host__ __device__ inline int64_t cta_of_slot(const Partition& p, int64_t x) {
    return ((x + 1) * p.ctas - 1) / p.total_slots;
}

struct Segment {
    int32_t unit, row, group;
    int64_t s0, s1;     // slot range within the unit
    int32_t part;       // partial slot, -1 when this CTA owns the whole unit
};

// Number of segments (units touched) of CTA c.
__host__ __device__ inline int32_t cta_segments(const Partition& p, int64_t c, int64_t* first_unit) {
    const int64_t b = cta_begin(p, c), e = cta_begin(p, c + 1);
    *first_unit = b / p.width;
    if (e <= b) return 0;
    return static_cast<int32_t>((e - 1) / p.width - b / p.width + 1);
}

__host__ __device__ inline Segment cta_segment(const Partition& p, int64_t c, int32_t i) {
    const int64_t b = cta_begin(p, c), e = cta_begin(p, c + 1);
    const int64_t u = b / p.width + i;
    Segment s;
    s.unit = static_cast<int32_t>(u);
    s.row = static_cast<int32_t>(u / p.groups);
    s.group = static_cast<int32_t>(u % p.groups);
    const int64_t ub = u * p.width;
    s.s0 = (b > ub ? b : ub) - ub;
    s.s1 = (e < ub + p.width ? e : ub + p.width) - ub;
    const bool whole = (s.s0 == 0 && s.s1 == p.width);
    s.part = whole ? -1 : static_cast<int32_t>(2 * c + (i == 0 ? 0 : 1));
    return s;
}

// Largest number of CTA ranges that one unit meets (CTAs with an empty range inside the
// unit included, as the combine kernel walks them): pieces(u) = cta_of_slot(u*W + W - 1) -
// cta_of_slot(u*W) + 1. A unit met by two or more ranges holds the start of one of them,
// so the maximum is taken over the units where CTAs start, or over all units when there
// are fewer units than CTAs.
inline int64_t max_pieces_per_unit(const Partition& p) {
    const int64_t units = p.total_slots / p.width;
    auto pieces = [&](int64_t u) { return cta_of_slot(p, u * p.width + p.width - 1) - cta_of_slot(p, u * p.width) + 1; };
    int64_t mp = 1;
    if (units <= p.ctas) {
        for (int64_t u = 0; u < units; ++u) mp = pieces(u) > mp ? pieces(u) : mp;
    } else {
        for (int64_t c = 0; c < p.ctas; ++c) {
            const int64_t k = pieces(cta_begin(p, c) / p.width);
            mp = k > mp ? k : mp;
        }
    }
    return mp;
}

// ------------------------------------------------------------------------------------
// Kernel parameter blocks.
// ------------------------------------------------------------------------------------
struct PrologueParams {
    const int32_t* sel;        // [R, W]
    const int32_t* seq_lens;   // [R] or [num_seqs] (verify rows)
    const uint16_t* q;         // bf16 bits [R, H, 512]; null: resolve only
    const int32_t* block_tables;  // null: ids only, no byte offsets
    int32_t* ids;              // [R, W], or null: the decode needs only offs and cnt
    long long* offs;           // [R, W] cache byte offset of each resolved token (-1: bad page)
    int32_t* cnt;              // [R]
    uint8_t* qimg;             // [R*G, 64 KB]
    float* qscale;             // [R*G, 64]
    int* status;               // reset by block 0 (may be null)
    int64_t cache_stride;
    int32_t rows, width, heads, groups, rows_per_seq, verify_rows;
    int32_t block_size, block_shift, max_blocks_per_seq;
    float score_scale;         // sm_scale * k_scale * log2(e)
};

struct DecodeParams {
    const uint8_t* k_cache;
    const uint8_t* v_cache;
    const long long* offs;
    const int32_t* cnt;
    const uint8_t* qimg;
    const float* qscale;
    uint16_t* out;             // bf16 bits [R, H, 512]
    uint16_t* part_o;          // f16 bits [2C, 64, 512]: O / l of a piece, E4M3 code units
    float* part_lse;           // [2C, 64]
    int* status;
    Partition part;
    int32_t heads;
    int32_t kv_same;
    float v_scale;
    int32_t early_dependents;  // let the next kernel launch once every CTA has started
    uint64_t wait_limit_ns;    // time limit of each pipeline wait (DSA_ERR_TIMEOUT past it)
    int32_t use_tma;           // gather by tensor map (dense pages), else per-thread copies
    unsigned long long* trace;  // per-CTA timeline, used only by -DDSA_TRACE builds
};

struct CombineParams {
    const uint16_t* part_o;
    const float* part_lse;
    uint16_t* out;
    Partition part;
    int32_t heads;
    float v_scale;
    int32_t early_dependents;  // let the next kernel launch as soon as every block has started
};

struct LatentWriteParams {
    const uint16_t* kv_a;      // bf16 bits [rows, 512]
    const uint16_t* weight;    // bf16 bits [512]: the kv_a RMSNorm weight
    const long long* slots;    // [rows]; a negative slot writes nothing
    uint8_t* cache;            // E4M3 pool
    int64_t cache_stride;      // bytes per page
    int32_t rows, block_size;
    float eps;                 // rms_eps
    float inv_scale;           // 1/kv_scale
};

struct SelectParams {
    const float* scores;       // [rows, n_pools] pooled indexer scores
    const int32_t* q_pos;      // [rows] position of each query row
    int32_t* ids;              // [rows, topk * kpool] token ids, -1 padded
    int32_t rows, n_pools, kpool, topk;
};

// Launchers (each defined next to its kernel).
// The decode and combine kernels are launched as programmatic dependents of the kernel
// before them on the stream (they start their set-up early and wait on the grid
// dependency before reading its results).
// programmatic: launch as a programmatic dependent of the kernel before it (done after long
// decodes, whose decode and combine kernels let their dependents launch early).
cudaError_t launch_prologue(const PrologueParams& p, int blocks, bool programmatic, cudaStream_t stream);
// The decode kernel exists for tiles of 64 and of 128 tokens (decode.cu compiled twice);
// 64-token tiles pipeline better when a CTA has little work, 128-token tiles use the
// tensor core better when it has much.
// kmap / vmap: 2-D tensor maps of the K and V caches ([rows of 512 bytes], box 128 x 1,
// 128-byte swizzle), read only when p.use_tma is set.
cudaError_t launch_decode_64(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                             cudaStream_t stream);
cudaError_t launch_decode_128(const DecodeParams& p, const CUtensorMap& kmap, const CUtensorMap& vmap,
                              cudaStream_t stream);
// max_pieces: the most CTAs sharing one unit (max_pieces_per_unit; selects the variant).
cudaError_t launch_combine(const CombineParams& p, int units, int max_pieces, cudaStream_t stream);
cudaError_t launch_latent_write(const LatentWriteParams& p, cudaStream_t stream);
int32_t check_device();  // DSA_OK when the current device is an sm_103 with the kernels loaded
cudaError_t select_kernel_setup();
cudaError_t launch_select(const SelectParams& p, cudaStream_t stream);
cudaError_t decode_kernel_setup_64();
cudaError_t decode_kernel_setup_128();
cudaError_t prologue_kernel_setup();
cudaError_t combine_kernel_setup();

}  // namespace dsa
