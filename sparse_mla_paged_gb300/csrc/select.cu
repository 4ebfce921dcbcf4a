// The selector that makes the decode's input rows (attend.rs module doc: [q_rows, width]
// token ids with -1 holes; decode_k.rs decode_k: index_topk pools per row, row r taking
// only pools that end at or before its position q_pos[r]). Pool p covers positions
// p*kpool .. p*kpool + kpool - 1, so the eligible pools of a row are the prefix
// p < (q_pos + 1) / kpool. The index_topk eligible pools of highest score are taken (equal
// scores: the lower pool; NaN lowest) and listed in ascending position, kpool ids each,
// then -1 up to index_topk*kpool entries. The selector's body is not on the pages; this is
// the reading the oracle states too.
//
// One block of 512 threads per row. The row's scores become order-preserving 32-bit keys;
// three radix digits (11, 11 and 10 bits of the key) find the index_topk-th largest key T
// and how many pools with key T are still to be taken.
// * Rows of at most 40960 pools (select_staged_kernel): the keys are staged once in shared
//   memory while the first digit's histogram is built. Thread t then owns pools 32t ..
//   32t + 31 (per round of 32768 pools) and works on 32-bit masks of them: each warp lists
//   its pools in T's first-digit bin (a few hundred in all for spread scores) in a region
//   of its own, and counts the other two digits over that list (over its threads' own
//   pools when the list overflowed). A last pass marks the pools above T and equal to T;
//   one block scan of both counts ranks the equal ones (the lowest-numbered are kept up to
//   the count still needed) and gives each thread its output position, and the taken pools
//   are written in ascending order. Block barriers are the cost after staging, so block
//   scans and histograms are double-buffered: nine barriers follow the staging.
// * Longer rows (select_kernel): the three digit passes re-read the scores from global
//   memory; each warp then owns a contiguous segment of pools, counts its keys above and
//   equal to T, one scan over the warps gives every warp its output offset, and a second
//   sweep writes the taken pools' ids in order with ballot prefix counts.
#include "common.cuh"

namespace dsa {
namespace {

constexpr int kSelectThreads = 1024;
constexpr int kSelectWarps = kSelectThreads / 32;
constexpr int kBins = 2048;
constexpr int kBinsPerThread = kBins / kSelectThreads;
constexpr int kStageMaxPools = 40960;  // 160 KB of staged keys

// Larger key = better rank. NaN is 0, below every number; -0 and +0 are one key;
// subnormals keep their order (integer tests only, so no flush to zero can merge them).
__device__ __forceinline__ uint32_t score_key(float s) {
    const uint32_t b = __float_as_uint(s), mag = b & 0x7FFFFFFFu;
    if (mag > 0x7F800000u) return 0u;
    if (mag == 0u) return 0x80000000u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

constexpr int kCandidates = 4096;       // threshold-bin candidates kept in shared memory
constexpr int kWarpCandidates = kCandidates / kSelectWarps;  // a private region per warp
constexpr int kLoadBatch = 8;           // 16-byte score loads in flight per thread

static_assert(kSelectWarps == 32, "a warp reads all warp totals, one per lane");

// Warp totals for block scans, double-buffered: scan k writes buffer k % 2, so one barrier
// per scan suffices (a buffer is written again only after the next scan's barrier, which
// every reader of it has passed).
struct ScanState {
    uint32_t (*buf)[kSelectWarps];
    int parity;
};

// Exclusive prefix sum over the block, in unsigned (wrapping) arithmetic; *total receives
// the block total. Every thread of the block must call it (one block barrier).
__device__ __forceinline__ uint32_t block_exclusive_scan(uint32_t v, ScanState& st, uint32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    uint32_t* sums = st.buf[st.parity];
    st.parity ^= 1;
    if (lane == 31) sums[warp] = x;
    __syncthreads();
    const uint32_t t = sums[lane];
    *total = __reduce_add_sync(0xffffffffu, t);
    return __reduce_add_sync(0xffffffffu, lane < warp ? t : 0u) + x - v;
}

// Radix step shared by both kernels: given the digit histogram, the thread whose bins
// (kBinsPerThread of them, counted from the top: thread 0 holds 2047 down) hold the
// crossing point where the count from above reaches need records the digit and the count
// still needed in it. Two block barriers.
__device__ __forceinline__ void find_crossing(const int32_t* hist, int32_t need, ScanState& st, uint32_t* sh_digit,
                                              int32_t* sh_need) {
    int32_t c[kBinsPerThread], s = 0;
#pragma unroll
    for (int k = 0; k < kBinsPerThread; ++k) {
        c[k] = hist[kBins - 1 - (kBinsPerThread * threadIdx.x + k)];
        s += c[k];
    }
    uint32_t total;
    const int32_t above = static_cast<int32_t>(block_exclusive_scan(static_cast<uint32_t>(s), st, &total));
    if (above < need && above + s >= need) {
        int32_t acc = above;
#pragma unroll
        for (int k = 0; k < kBinsPerThread; ++k) {
            if (acc + c[k] >= need) {
                *sh_digit = static_cast<uint32_t>(kBins - 1 - (kBinsPerThread * threadIdx.x + k));
                *sh_need = need - acc;
                break;
            }
            acc += c[k];
        }
    }
    __syncthreads();
}

// The 32 keys of pools [base, base + 32) from shared memory, in 16-byte pieces taken in an
// order rotated by the thread index (threads 128 bytes apart then hit different banks).
// Each piece is handed to f(bit, key4, valid4) with bit = the first pool's offset from base;
// a thread whose 32 pools are all eligible takes the path without per-key bounds.
template <typename F>
__device__ __forceinline__ void for_own_keys(const uint32_t* keys, int32_t base, int32_t n, F&& f) {
    if (base + 32 <= n) {
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int c = (k + threadIdx.x) & 7;
            f(4 * c, *reinterpret_cast<const uint4*>(keys + base + 4 * c), 4);
        }
        return;
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const int c = (k + threadIdx.x) & 7;
        const int32_t e0 = base + 4 * c;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        int valid = 0;
        if (e0 + 3 < n) {
            v = *reinterpret_cast<const uint4*>(keys + e0);
            valid = 4;
        } else if (e0 < n) {
            valid = n - e0;
            v.x = keys[e0];
            if (valid > 1) v.y = keys[e0 + 1];
            if (valid > 2) v.z = keys[e0 + 2];
        }
        f(4 * c, v, valid);
    }
}

__global__ void __launch_bounds__(kSelectThreads) select_staged_kernel(const SelectParams p) {
    extern __shared__ __align__(16) uint32_t keys[];  // [n_pools]
    __shared__ int32_t hist[2][kBins];                 // one digit counted while the other is cleared
    __shared__ uint32_t cand_key[kCandidates];
    __shared__ uint32_t scan_buf[2][kSelectWarps];
    __shared__ uint32_t sh_digit;
    __shared__ int32_t sh_need;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t r = blockIdx.x;
    const float* sc = p.scores + r * p.n_pools;
    int32_t* out = p.ids + r * static_cast<int64_t>(p.topk) * p.kpool;
    const int64_t q = p.q_pos[r];
    const int64_t by_pos = q < 0 ? 0 : (q + 1) / p.kpool;
    const int32_t n = static_cast<int32_t>(by_pos < p.n_pools ? by_pos : p.n_pools);  // eligible: pools [0, n)
    const int64_t width = static_cast<int64_t>(p.topk) * p.kpool;
    ScanState st{scan_buf, 0};

    if (n <= p.topk) {  // every eligible pool is taken
        for (int64_t e = tid; e < width; e += kSelectThreads) out[e] = e < static_cast<int64_t>(n) * p.kpool ? static_cast<int32_t>(e) : -1;
        return;
    }
    for (int b = tid; b < 2 * kBins; b += kSelectThreads) (&hist[0][0])[b] = 0;
    __syncthreads();

    // Stage the keys and count the first digit (bits 31..21), kLoadBatch loads in flight
    // per thread before any is used.
    const bool vec = (reinterpret_cast<uintptr_t>(sc) & 15u) == 0;
    const int32_t n4 = vec ? n / 4 : 0;
    const float4* sc4 = reinterpret_cast<const float4*>(sc);
#pragma unroll 1
    for (int32_t i0 = tid; i0 < n4; i0 += kLoadBatch * kSelectThreads) {
        float4 v[kLoadBatch];
#pragma unroll
        for (int k = 0; k < kLoadBatch; ++k) {
            const int32_t i = i0 + k * kSelectThreads;
            v[k] = i < n4 ? __ldg(sc4 + i) : make_float4(0.0f, 0.0f, 0.0f, 0.0f);
        }
#pragma unroll
        for (int k = 0; k < kLoadBatch; ++k) {
            const int32_t i = i0 + k * kSelectThreads;
            if (i < n4) {
                const uint4 kk = make_uint4(score_key(v[k].x), score_key(v[k].y), score_key(v[k].z), score_key(v[k].w));
                reinterpret_cast<uint4*>(keys)[i] = kk;
                atomicAdd(&hist[0][kk.x >> 21], 1);
                atomicAdd(&hist[0][kk.y >> 21], 1);
                atomicAdd(&hist[0][kk.z >> 21], 1);
                atomicAdd(&hist[0][kk.w >> 21], 1);
            }
        }
    }
    for (int32_t i = 4 * n4 + tid; i < n; i += kSelectThreads) {
        const uint32_t k = score_key(__ldg(sc + i));
        keys[i] = k;
        atomicAdd(&hist[0][k >> 21], 1);
    }
    __syncthreads();
    find_crossing(hist[0], p.topk, st, &sh_digit, &sh_need);
    const uint32_t bin_lo = sh_digit << 21;  // keys of the threshold bin: [bin_lo, bin_lo + 2^21)
    int32_t need = sh_need;
    for (int b = tid; b < kBins; b += kSelectThreads) hist[0][b] = 0;  // for the third digit

    // Candidates: the pools of the threshold bin. Thread t owns pools 32t .. 32t + 31 of
    // each round of kSelectThreads*32 pools; each warp lists its candidates in a region of
    // its own (warp scan of the per-thread counts, no atomics, no block barrier).
    const int32_t rounds = (n + kSelectThreads * 32 - 1) / (kSelectThreads * 32);
    int32_t my_cands = 0;  // this warp's, uniform over the warp
    for (int32_t rd = 0; rd < rounds; ++rd) {
        const int32_t base = rd * kSelectThreads * 32 + 32 * tid;
        uint32_t cmask = 0u;
        for_own_keys(keys, base, n, [&](int bit, uint4 v, int valid) {
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (e < valid && u[e] - bin_lo < (1u << 21)) cmask |= 1u << (bit + e);
        });
        const int32_t c = __popc(cmask);
        int32_t x = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int32_t y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        int32_t slot = my_cands + x - c;
        my_cands += __shfl_sync(0xffffffffu, x, 31);
        while (cmask != 0u) {
            const int b = __ffs(cmask) - 1;
            cmask &= cmask - 1u;
            if (slot < kWarpCandidates) cand_key[warp * kWarpCandidates + slot] = keys[base + b];
            ++slot;
        }
    }
    __syncwarp();  // the warp's list, written by its lanes, is read by other lanes below
    const bool listed = my_cands <= kWarpCandidates;  // per warp: else its own pools are re-read
    const uint32_t* my_list = cand_key + warp * kWarpCandidates;

    // The two last digits: each warp counts its own candidates (or, when its list
    // overflowed, the threshold-bin keys among its threads' own pools).
    uint32_t prefix = bin_lo, mask = 0x7FFu << 21;
#pragma unroll 1
    for (int pass = 0; pass < 2; ++pass) {
        const int shift = pass == 0 ? 10 : 0;
        const uint32_t digit = pass == 0 ? 0x7FFu : 0x3FFu;
        int32_t* h = hist[pass == 0 ? 1 : 0];
        if (listed) {
            for (int32_t j = lane; j < my_cands; j += 32) {
                const uint32_t u = my_list[j];
                if ((u & mask) == prefix) atomicAdd(&h[(u >> shift) & digit], 1);
            }
        } else {
            for (int32_t rd = 0; rd < rounds; ++rd)
                for_own_keys(keys, rd * kSelectThreads * 32 + 32 * tid, n, [&](int, uint4 v, int valid) {
                    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (e < valid && (u[e] & mask) == prefix) atomicAdd(&h[(u[e] >> shift) & digit], 1);
                });
        }
        __syncthreads();
        find_crossing(h, need, st, &sh_digit, &sh_need);
        prefix |= sh_digit << shift;
        need = sh_need;
        mask |= digit << shift;
    }
    const uint32_t T = prefix;  // the topk-th largest key; `need` pools with key T are taken

    // Emit in ascending pool order, round by round: every pool above T, and the
    // lowest-numbered pools equal to T up to `need`. One block scan of the packed counts
    // (equal << 16 | above; each total is at most 32768) gives both prefixes: the equal
    // pools kept before a thread are min(need left, equal pools before it).
    int32_t eq_seen = 0, out_base = 0;
    for (int32_t rd = 0; rd < rounds; ++rd) {
        const int32_t base = rd * kSelectThreads * 32 + 32 * tid;
        uint32_t gmask = 0u, emask = 0u;
        for_own_keys(keys, base, n, [&](int bit, uint4 v, int valid) {
            const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                if (e < valid && u[e] > T) gmask |= 1u << (bit + e);
                if (e < valid && u[e] == T) emask |= 1u << (bit + e);
            }
        });
        uint32_t packed_total;
        const uint32_t packed =
            block_exclusive_scan((static_cast<uint32_t>(__popc(emask)) << 16) | __popc(gmask), st, &packed_total);
        const int32_t left = max(0, need - eq_seen);  // equal pools still to take
        const int32_t eq_before = static_cast<int32_t>(packed >> 16);
        int32_t keep = min(__popc(emask), max(0, left - eq_before));
        while (keep-- > 0) {  // the lowest-numbered equal pools of this thread
            gmask |= emask & (0u - emask);
            emask &= emask - 1u;
        }
        int32_t pos = out_base + static_cast<int32_t>(packed & 0xFFFFu) + min(left, eq_before);
        while (gmask != 0u) {
            const int32_t pool = base + __ffs(gmask) - 1;
            gmask &= gmask - 1u;
            int32_t* o = out + static_cast<int64_t>(pos++) * p.kpool;
            for (int32_t c = 0; c < p.kpool; ++c) o[c] = pool * p.kpool + c;
        }
        const int32_t eq_total = static_cast<int32_t>(packed_total >> 16);
        eq_seen += eq_total;
        out_base += static_cast<int32_t>(packed_total & 0xFFFFu) + min(left, eq_total);
    }
}

// Rows longer than the staging limit: three digit passes over the scores in global memory,
// then warp-segment compaction (see the file comment).
__global__ void __launch_bounds__(kSelectThreads) select_kernel(const SelectParams p) {
    __shared__ int32_t hist[kBins];
    __shared__ uint32_t scan_buf[2][kSelectWarps];
    __shared__ int32_t seg_out[kSelectWarps], seg_eq_base[kSelectWarps];
    __shared__ uint32_t sh_digit;
    __shared__ int32_t sh_need;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t r = blockIdx.x;
    const float* sc = p.scores + r * p.n_pools;
    int32_t* out = p.ids + r * static_cast<int64_t>(p.topk) * p.kpool;
    const int64_t q = p.q_pos[r];
    const int64_t by_pos = q < 0 ? 0 : (q + 1) / p.kpool;
    const int32_t n = static_cast<int32_t>(by_pos < p.n_pools ? by_pos : p.n_pools);  // eligible: pools [0, n)
    const int64_t width = static_cast<int64_t>(p.topk) * p.kpool;
    ScanState st{scan_buf, 0};
    if (n <= p.topk) {  // every eligible pool is taken
        for (int64_t e = tid; e < width; e += kSelectThreads) out[e] = e < static_cast<int64_t>(n) * p.kpool ? static_cast<int32_t>(e) : -1;
        return;
    }

    // Threshold: T = the topk-th largest key, need = how many pools with key T to take.
    uint32_t prefix = 0u, mask = 0u;
    int32_t need = p.topk;
#pragma unroll 1
    for (int pass = 0; pass < 3; ++pass) {
        const int shift = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
        const uint32_t digit = pass == 2 ? 0x3FFu : 0x7FFu;
        for (int b = tid; b < kBins; b += kSelectThreads) hist[b] = 0;
        __syncthreads();
        for (int32_t i = tid; i < n; i += kSelectThreads) {
            const uint32_t u = score_key(__ldg(sc + i));
            if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & digit], 1);
        }
        __syncthreads();
        find_crossing(hist, need, st, &sh_digit, &sh_need);
        prefix |= sh_digit << shift;
        need = sh_need;
        mask |= digit << shift;
    }

    // Warp w owns pools [w*seg, min(n, (w+1)*seg)), seg a multiple of 32.
    const int32_t seg = ((n + kSelectWarps * 32 - 1) / (kSelectWarps * 32)) * 32;
    const int32_t lo = warp * seg, hi = min(n, lo + seg);
    const uint32_t lanes_below = (1u << lane) - 1u;
    int32_t gt = 0, eq = 0;
    for (int32_t i0 = lo; i0 < hi; i0 += 32) {
        const int32_t i = i0 + lane;
        const uint32_t u = i < hi ? score_key(__ldg(sc + i)) : 0u;
        gt += __popc(__ballot_sync(0xffffffffu, i < hi && u > prefix));
        eq += __popc(__ballot_sync(0xffffffffu, i < hi && u == prefix));
    }
    uint32_t eq_total, t_total;
    const int32_t e_base = static_cast<int32_t>(block_exclusive_scan(lane == 0 ? eq : 0, st, &eq_total));
    const int32_t t = gt + max(0, min(eq, need - e_base));
    const int32_t t_base = static_cast<int32_t>(block_exclusive_scan(lane == 0 ? t : 0, st, &t_total));
    if (lane == 0) {
        seg_out[warp] = t_base;
        seg_eq_base[warp] = e_base;
    }
    __syncthreads();
    int32_t pos = seg_out[warp];
    int32_t eq_seen = seg_eq_base[warp];
    for (int32_t i0 = lo; i0 < hi; i0 += 32) {
        const int32_t i = i0 + lane;
        const uint32_t u = i < hi ? score_key(__ldg(sc + i)) : 0u;
        const bool equal = i < hi && u == prefix;
        const uint32_t eq_mask = __ballot_sync(0xffffffffu, equal);
        const bool take = (i < hi && u > prefix) || (equal && eq_seen + __popc(eq_mask & lanes_below) < need);
        eq_seen += __popc(eq_mask);
        const uint32_t take_mask = __ballot_sync(0xffffffffu, take);
        if (take) {
            int32_t* o = out + static_cast<int64_t>(pos + __popc(take_mask & lanes_below)) * p.kpool;
            for (int32_t c = 0; c < p.kpool; ++c) o[c] = i * p.kpool + c;
        }
        pos += __popc(take_mask);
    }
}

}  // namespace

cudaError_t select_kernel_setup() {
    return cudaFuncSetAttribute(select_staged_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kStageMaxPools * 4);
}

cudaError_t launch_select(const SelectParams& p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    if (p.n_pools <= kStageMaxPools)
        select_staged_kernel<<<p.rows, kSelectThreads, p.n_pools * 4, stream>>>(p);
    else
        select_kernel<<<p.rows, kSelectThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace dsa
