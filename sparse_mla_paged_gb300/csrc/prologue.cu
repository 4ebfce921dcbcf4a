// Prologue of the decode: index resolution and query preparation, one launch.
//
// Blocks [0, rows) resolve one selection row each (attend.rs module doc: -1 holes,
// set membership with duplicates collapsed; decode_k.rs: row r only sees positions
// below its own seq_len): the distinct ids 0 <= id < L in ascending order, -1 padded,
// and (for the decode) each id's cache byte offset through the block table
// (decode_k.rs: physical = block_table[pos / block_size], slot = physical*block_size +
// pos % block_size), so the decode's gather needs one load per token.
//   * L <= 16 * 262144: a bitmap of 262144 bits in shared memory per window of that many
//     positions, windows in ascending order (one for L <= 262144); ids set with atomicOr
//     and written out by a block-wide prefix count, which yields them sorted.
//   * longer rows: bitonic sort of the row in shared memory, then a prefix count of
//     first occurrences.
// Blocks [rows, rows + rows*groups) turn one (row, 64-head group) of BF16 queries into
// the operand image the decode kernel loads into tensor memory: per head a power-of-two
// scale 2^e (|q|*2^e < 256) and two E4M3 terms hi + lo whose sum is q*2^e. hi keeps the
// top 4 significant bits (truncation), lo is the remainder; for |q*2^e| >= 2^-2 the
// split is exact, since a BF16 value has 8 significant bits. The image holds 128 rows of
// 512 codes (row 32q + 2k + t = term t of head 16q + k), stored chunk-major: the 16 bytes
// of chunk c of row r are at c*2048 + r*16.
#include "common.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kMaxSel = DSA_MAX_SEL_WIDTH;                        // resolved ids per row, at most
constexpr int kPrologueSmem = kBitmapWords * 4 + kMaxSel * 4;     // bitmap or keys, then the ids
static_assert(kQImageBytes <= kPrologueSmem, "a query block stages its image in the same shared memory");
constexpr int kBatch = 8;                                         // loads in flight per thread
constexpr int kMaxWindows = 16;  // bitmap windows per row (4M positions); longer rows are sorted

__device__ __forceinline__ int32_t row_seq_len(const PrologueParams& p, int32_t r) {
    int32_t L = p.verify_rows ? p.seq_lens[r / p.rows_per_seq] + (r % p.rows_per_seq) + 1 : p.seq_lens[r];
    return L < 0 ? 0 : L;
}

// Exclusive prefix sum over the block (kResolveThreads threads); also returns the total.
__device__ __forceinline__ int32_t block_exclusive_scan(int32_t v, int32_t* scratch, int32_t* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) scratch[warp] = x;
    __syncthreads();
    if (warp == 0) {
        int32_t w = lane < kResolveThreads / 32 ? scratch[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int32_t y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < kResolveThreads / 32) scratch[lane] = w;  // inclusive per-warp totals
    }
    __syncthreads();
    const int32_t before = (warp > 0 ? scratch[warp - 1] : 0) + x - v;
    *total = scratch[kResolveThreads / 32 - 1];
    __syncthreads();
    return before;
}

// sm: kBitmapWords words of scratch (bitmap or sort keys); ids_s: kMaxSel resolved ids.
__device__ void resolve_row(const PrologueParams& p, int32_t r, uint32_t* sm, int32_t* ids_s, int32_t* scratch) {
    const int tid = threadIdx.x;
    const int32_t W = p.width;
    const int32_t L = row_seq_len(p, r);
    const int32_t seq = r / p.rows_per_seq;
    const int32_t* sel = p.sel + static_cast<int64_t>(r) * W;
    int32_t* ids = p.ids ? p.ids + static_cast<int64_t>(r) * W : nullptr;
    long long* offs = p.block_tables ? p.offs + static_cast<int64_t>(r) * W : nullptr;
    int32_t total = 0;
    // The first batch of the selection row is requested together with the row's length
    // (before the branch on it), and arrives while the whole bitmap is cleared: clearing
    // all of it does not wait for the length (the sort path overwrites it anyway).
    int32_t idv[kBatch];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
        const int32_t j = tid + k * kResolveThreads;
        idv[k] = j < W ? sel[j] : -1;
    }
    uint4* sm4 = reinterpret_cast<uint4*>(sm);
#pragma unroll
    for (int k = 0; k < kBitmapWords / 4 / kResolveThreads; ++k)
        sm4[tid + k * kResolveThreads] = make_uint4(0u, 0u, 0u, 0u);
    // Rows up to kMaxWindows bitmaps long are resolved one window of kBitmapWords*32
    // positions at a time, in ascending order (one window for L <= 262144): mark the ids
    // that fall in the window, then count and extract them after the ids of the windows
    // before. The first window's ids come from the batch already loaded; a later window
    // reads the row again (from L2).
    const int32_t nwin = static_cast<int32_t>((static_cast<int64_t>(L) + kBitmapWords * 32 - 1) / (kBitmapWords * 32));
    if (nwin <= kMaxWindows) {
        for (int32_t win = 0; win < nwin; ++win) {
            const int32_t lo = win * (kBitmapWords * 32);
            const int32_t hi = min(L, lo + kBitmapWords * 32);
            const int32_t nwords = (hi - lo + 31) >> 5;
            if (win > 0) {
                __syncthreads();  // the previous window's extraction has read the bitmap
#pragma unroll
                for (int k = 0; k < kBitmapWords / 4 / kResolveThreads; ++k)
                    sm4[tid + k * kResolveThreads] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int32_t j = tid + k * kResolveThreads;
                    idv[k] = j < W ? sel[j] : -1;
                }
            }
            __syncthreads();
            for (int32_t j0 = tid;; j0 += kBatch * kResolveThreads) {
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int32_t id = idv[k];
                    if (id >= lo && id < hi) atomicOr(&sm[(id - lo) >> 5], 1u << ((id - lo) & 31));
                }
                const int32_t n0 = j0 + kBatch * kResolveThreads;
                if (n0 - tid >= W) break;
#pragma unroll
                for (int k = 0; k < kBatch; ++k) {
                    const int32_t j = n0 + k * kResolveThreads;
                    idv[k] = j < W ? sel[j] : -1;
                }
            }
            __syncthreads();
            // Each warp takes a contiguous range of words (a multiple of 32) and reads it 32
            // consecutive words at a time (one word per lane, free of bank conflicts): a count
            // pass, a block scan of the warp totals, then an extraction pass in which a warp
            // scan of the words' bit counts places every lane's ids.
            const int lane = tid & 31, warp = tid >> 5;
            const int32_t wpw = ((nwords + kResolveThreads - 1) / kResolveThreads) * 32;
            const int32_t wbeg = warp * wpw;
            const int32_t wend = min(wbeg + wpw, nwords);
            int32_t mine = 0;
#pragma unroll 4
            for (int32_t w = wbeg + lane; w < wend; w += 32) mine += __popc(sm[w]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
            int32_t wtotal = 0;
            int32_t pos = block_exclusive_scan(lane == 0 ? mine : 0, scratch, &wtotal);
            pos = __shfl_sync(0xffffffffu, pos, 0) + total;
            // Four steps of 32 words at a time: their warp scans are independent and interleave.
            constexpr int kSteps = 4;
            for (int32_t w0 = wbeg; w0 < wend; w0 += 32 * kSteps) {
                uint32_t bits[kSteps];
                int32_t c[kSteps], incl[kSteps];
#pragma unroll
                for (int j = 0; j < kSteps; ++j) {
                    const int32_t w = w0 + 32 * j + lane;
                    bits[j] = w < wend ? sm[w] : 0u;
                    c[j] = __popc(bits[j]);
                    incl[j] = c[j];
                }
#pragma unroll
                for (int o = 1; o < 32; o <<= 1)
#pragma unroll
                    for (int j = 0; j < kSteps; ++j) {
                        const int32_t y = __shfl_up_sync(0xffffffffu, incl[j], o);
                        if (lane >= o) incl[j] += y;
                    }
#pragma unroll
                for (int j = 0; j < kSteps; ++j) {
                    int32_t at = pos + incl[j] - c[j];
                    const int32_t w = w0 + 32 * j + lane;
                    while (bits[j]) {
                        const int b = __ffs(bits[j]) - 1;
                        ids_s[at++] = lo + w * 32 + b;
                        bits[j] &= bits[j] - 1;
                    }
                    pos += __shfl_sync(0xffffffffu, incl[j], 31);
                }
            }
            total += wtotal;
        }
    } else {
        __syncthreads();  // the clearing above is done before the keys overwrite it
        int32_t* keys = reinterpret_cast<int32_t*>(sm);
        int32_t n = 1;
        while (n < W) n <<= 1;
        for (int32_t j = tid; j < n; j += kResolveThreads) {
            int32_t id = j < W ? sel[j] : -1;
            keys[j] = (id >= 0 && id < L) ? id : INT32_MAX;
        }
        __syncthreads();
        for (int32_t k = 2; k <= n; k <<= 1) {
            for (int32_t j = k >> 1; j > 0; j >>= 1) {
                for (int32_t i = tid; i < n; i += kResolveThreads) {
                    const int32_t x = i ^ j;
                    if (x > i) {
                        const int32_t a = keys[i], b = keys[x];
                        const bool up = (i & k) == 0;
                        if ((a > b) == up) {
                            keys[i] = b;
                            keys[x] = a;
                        }
                    }
                }
                __syncthreads();
            }
        }
        const int32_t per = (W + kResolveThreads - 1) / kResolveThreads;
        const int32_t j0 = tid * per;
        const int32_t j1 = min(j0 + per, W);
        int32_t mine = 0;
        for (int32_t j = j0; j < j1; ++j)
            mine += (keys[j] != INT32_MAX && (j == 0 || keys[j] != keys[j - 1])) ? 1 : 0;
        int32_t pos = block_exclusive_scan(mine, scratch, &total);
        for (int32_t j = j0; j < j1; ++j)
            if (keys[j] != INT32_MAX && (j == 0 || keys[j] != keys[j - 1])) ids_s[pos++] = keys[j];
    }
    __syncthreads();
    // Coalesced write-out of the ids (-1 padded), then each id's byte offset with all of a
    // thread's block-table loads in flight at once.
    if (ids)
        for (int32_t j = tid; j < W; j += kResolveThreads) ids[j] = j < total ? ids_s[j] : -1;
    if (tid == 0) p.cnt[r] = total;
    if (!offs) return;
    for (int32_t j0 = tid; j0 < total; j0 += kBatch * kResolveThreads) {
        // Cache byte offset of each id through the block table (decode_k.rs: physical =
        // block_table[pos / block_size], slot = physical*block_size + pos % block_size),
        // -1 when the table has no valid page for it (the decode kernel reports that as a
        // device status). All of the batch's table loads are issued (predicated, with no
        // branch between them) before any of their results is used.
        int32_t id[kBatch], page[kBatch];
#pragma unroll
        for (int e = 0; e < kBatch; ++e) {
            const int32_t j = j0 + e * kResolveThreads;
            id[e] = j < total ? ids_s[j] : 0;
            const int32_t blk = p.block_shift >= 0 ? (id[e] >> p.block_shift) : id[e] / p.block_size;
            const bool ok = j < total && (p.max_blocks_per_seq <= 0 || blk < p.max_blocks_per_seq);
            page[e] = ok ? p.block_tables[static_cast<int64_t>(seq) * p.max_blocks_per_seq + blk] : -1;
        }
#pragma unroll
        for (int e = 0; e < kBatch; ++e) {
            const int32_t j = j0 + e * kResolveThreads;
            if (j < total) {
                const int32_t inblk = p.block_shift >= 0 ? (id[e] & (p.block_size - 1)) : id[e] % p.block_size;
                offs[j] = page[e] >= 0 ? static_cast<long long>(page[e]) * p.cache_stride +
                                             static_cast<long long>(inblk) * kLatent
                                       : -1ll;
            }
        }
    }
}

// One (row, group): 8 warps x 8 heads; lane l handles latent dims [16l, 16l+16). The
// image is assembled in shared memory (row r's chunk c at r*512 + (c ^ (r % 32))*16, so
// that both the row writes and the chunk reads below are free of bank conflicts) and then
// written out chunk-major with each warp storing 512 contiguous bytes.
__device__ void prepare_queries(const PrologueParams& p, int32_t unit, uint8_t* stage) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int32_t r = unit / p.groups, g = unit % p.groups;
    uint8_t* img = p.qimg + static_cast<int64_t>(unit) * kQImageBytes;
    constexpr int kHeadsPerWarp = kHeadsPerCta / (kResolveThreads / 32);  // 8
    // All of this warp's loads first (8 heads x 32 bytes per lane), then the arithmetic.
    uint4 raw[kHeadsPerWarp][2];
#pragma unroll
    for (int i = 0; i < kHeadsPerWarp; ++i) {
        const int32_t h = g * kHeadsPerCta + warp + i * (kResolveThreads / 32);
        if (h < p.heads) {
            const uint4* src = reinterpret_cast<const uint4*>(
                p.q + (static_cast<int64_t>(r) * p.heads + h) * kLatent + lane * 16);
            raw[i][0] = src[0];
            raw[i][1] = src[1];
        } else {
            raw[i][0] = raw[i][1] = make_uint4(0, 0, 0, 0);
        }
    }
#pragma unroll
    for (int i = 0; i < kHeadsPerWarp; ++i) {
        const int hl = warp + i * (kResolveThreads / 32);
        float x[16];
        const uint32_t w[8] = {raw[i][0].x, raw[i][0].y, raw[i][0].z, raw[i][0].w,
                               raw[i][1].x, raw[i][1].y, raw[i][1].z, raw[i][1].w};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            x[2 * k] = __uint_as_float(w[k] << 16);
            x[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
        float amax = 0.0f;
#pragma unroll
        for (int k = 0; k < 16; ++k) amax = fmaxf(amax, fabsf(x[k]));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        // e with amax * 2^e in [128, 256): amax = 1.m * 2^(E-127), so e = 134 - E.
        int e = 0;
        if (amax > 0.0f) {
            const int E = static_cast<int>((__float_as_uint(amax) >> 23) & 0xFF);
            e = 134 - E;
            e = e > 126 ? 126 : (e < -126 ? -126 : e);
        }
        const float sc = __uint_as_float(static_cast<uint32_t>(e + 127) << 23);
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            float vh[4], vl[4];
#pragma unroll
            for (int m = 0; m < 4; ++m) {
                const float v = x[4 * k + m] * sc;
                vh[m] = __uint_as_float(__float_as_uint(v) & 0xFFF00000u);
                vl[m] = v - vh[m];
            }
            hi[k] = f32x2_to_e4m3x2(vh[0], vh[1]) | (f32x2_to_e4m3x2(vh[2], vh[3]) << 16);
            lo[k] = f32x2_to_e4m3x2(vl[0], vl[1]) | (f32x2_to_e4m3x2(vl[2], vl[3]) << 16);
        }
        // Rows 2k and 2k+1 of quarter q hold the hi and lo terms of head 16q + k, so the
        // decode finds both terms of a head in neighbouring TMEM lanes. The image is stored
        // chunk-major ([32 chunks of 16 bytes][128 rows][16 bytes]): 32 consecutive rows of
        // one chunk are 512 contiguous bytes, which the decode reads one row per lane.
        const int rh = 32 * (hl >> 4) + 2 * (hl & 15);
        *reinterpret_cast<uint4*>(stage + rh * 512 + ((lane ^ (rh & 31)) << 4)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(stage + (rh + 1) * 512 + ((lane ^ ((rh + 1) & 31)) << 4)) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
        if (lane == 0)
            p.qscale[static_cast<int64_t>(unit) * kHeadsPerCta + hl] =
                p.score_scale * __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
    }
    __syncthreads();
    // 4096 16-byte pieces; piece k is chunk k / 128 of row k % 128.
    for (int k = threadIdx.x; k < kQImageBytes / 16; k += kResolveThreads) {
        const int c = k >> 7, r = k & 127;
        *reinterpret_cast<uint4*>(img + c * 2048 + r * 16) =
            *reinterpret_cast<const uint4*>(stage + r * 512 + ((c ^ (r & 31)) << 4));
    }
}

__global__ void __launch_bounds__(kResolveThreads) prologue_kernel(const PrologueParams p) {
    extern __shared__ __align__(16) uint32_t bitmap[];  // kBitmapWords words, then kMaxSel ids
    __shared__ int32_t scratch[kResolveThreads / 32];
    // When launched as a programmatic dependent of the kernel before it on the stream,
    // nothing is read or written before that kernel has completed.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // Let the decode kernel launch and run its set-up while this grid finishes; it waits
    // for this grid's completion before reading anything written here.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (blockIdx.x == 0 && threadIdx.x == 0 && p.status) atomicExch(p.status, 0);
    if (static_cast<int32_t>(blockIdx.x) < p.rows)
        resolve_row(p, blockIdx.x, bitmap, reinterpret_cast<int32_t*>(bitmap + kBitmapWords), scratch);
    else
        prepare_queries(p, blockIdx.x - p.rows, reinterpret_cast<uint8_t*>(bitmap));
}

}  // namespace

cudaError_t prologue_kernel_setup() {
    cudaFuncAttributes attr;
    cudaError_t e = cudaFuncGetAttributes(&attr, prologue_kernel);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(prologue_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPrologueSmem);
    if (e != cudaSuccess) return e;
    // Same shared-memory carveout as the decode kernel, so the SMs need no
    // reconfiguration between the two.
    return cudaFuncSetAttribute(prologue_kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

cudaError_t launch_prologue(const PrologueParams& p, int blocks, bool programmatic, cudaStream_t stream) {
    if (blocks <= 0) return cudaSuccess;
    if (!programmatic) {
        prologue_kernel<<<blocks, kResolveThreads, kPrologueSmem, stream>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(kResolveThreads);
    cfg.dynamicSmemBytes = kPrologueSmem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, prologue_kernel, p);
}

}  // namespace dsa
