/*
 * dsa_mla.h: C ABI of libdsa_mla, the GB300 (sm_103a) selected-index NoPE MLA paged
 * decode.
 *
 * Source pages (cited by title and item):
 *   [attend.rs]   spark_model/layers/glm5next_dsa/attend.rs
 *   [decode_k.rs] metrale_model_arch/glm5next_dsa/layer/decode_k.rs
 *   [build.rs]    spark_model/layers/glm5next_dsa/build.rs (the load-time absorb transforms)
 *
 * What is computed (attend.rs, module doc and decode_attention). For every decode row r
 * (sequence seq = r / rows_per_seq) and query head h:
 *   S_r       = distinct ids j of sel_indices[r, :] with 0 <= j < seq_len(r)
 *               (-1 and any other id outside [0, seq_len(r)) is a hole; duplicates
 *               count once: set membership, not a weighting)
 *   K_j = V_j = the 512-byte E4M3 latent row of token j, at byte
 *               block_tables[seq*max_blocks_per_seq + j/block_size]*cache_stride_bytes
 *               + (j % block_size)*512 of k_cache (resp. v_cache)
 *   out[r,h,:] = sum_{j in S_r} softmax_j(sm_scale * q[r,h,:].(k_scale*K_j)) (v_scale*V_j)
 *               and 0 when S_r is empty.
 * kv_lora_rank is fixed at 512 and there is one latent KV head with no rope section
 * (attend.rs, module doc on the NoPE layout; DsaDecodePaging::validate).
 *
 * Conventions for every entry point:
 *  - Device pointers are caller-owned CUDA device memory on the current device; the
 *    library never frees or keeps them. "stream" is a cudaStream_t passed as void*.
 *  - Calls enqueue work on the stream and return without synchronising, as the pages'
 *    launcher does (attend.rs, decode_attention), except where stated.
 *  - Arguments are checked on the host before anything is enqueued; an invalid call
 *    returns its status and writes nothing.
 *  - A missing or unloadable kernel is a hard error (DSA_ERR_NO_KERNEL), never a
 *    fallback to another path (attend.rs, Glm5NextDsaDecodeKernel::resolve).
 *  - Problems only visible on the device (a block-table entry that is negative or past
 *    max_blocks_per_seq, a pipeline wait that ran out of time) do not fault: the kernel
 *    skips the access and records the first such status in the workspace's status
 *    word, read back with dsa_read_device_status / dsa_last_device_status /
 *    dsa_static_device_status. The output of a call that recorded a device status is
 *    undefined.
 */
#ifndef DSA_MLA_H
#define DSA_MLA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dsa_status {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARGUMENT = 1, /* bad pointer, size, alignment or stride */
    DSA_ERR_UNSUPPORTED = 2,      /* device is not sm_103, or a size beyond the limits below */
    DSA_ERR_WORKSPACE = 3,        /* workspace too small, or growth needed during graph capture */
    DSA_ERR_CUDA = 4,             /* a CUDA runtime call or launch failed */
    DSA_ERR_NO_KERNEL = 5,        /* the sm_103a kernel image is missing for this device */
    DSA_ERR_DEVICE_BOUNDS = 6,    /* device-side: a page lookup fell outside the block table */
    DSA_ERR_TIMEOUT = 7           /* device-side: a pipeline wait exceeded its time limit */
} dsa_status;

/* Limits. sel_width may not exceed DSA_MAX_SEL_WIDTH. */
#define DSA_LATENT_DIM 512
#define DSA_MAX_SEL_WIDTH 8192

/* Version of this ABI (incremented on any incompatible change). */
int32_t dsa_abi_version(void);

/* Static description of a status code. Never NULL. */
const char* dsa_status_string(int32_t status);

/*
 * dsa_mla_decode: the selected-index decode (attend.rs, decode_attention).
 *
 *  q                  bf16 [R, num_q_heads, 512], R = num_seqs * rows_per_seq, rows ordered
 *                     seq*rows_per_seq + i; absorbed queries in latent space (attend.rs,
 *                     DsaDecodeInputs::q). 16-byte aligned.
 *  k_cache, v_cache   E4M3 paged latent cache; page p starts at byte p*cache_stride_bytes.
 *                     In NoPE MLA K and V are one buffer, passed twice (attend.rs,
 *                     DsaDecodeInputs); distinct buffers are also accepted and read
 *                     separately.
 *                     16-byte aligned, non-NULL.
 *  block_tables       int32 page ids; the table of sequence s starts at
 *                     block_tables + s*max_blocks_per_seq (max_blocks_per_seq = 0: every
 *                     sequence reads the one table at block_tables, decode_k.rs decode_k).
 *  max_blocks_per_seq block-table row stride in entries (>= 0). When > 0, a lookup past
 *                     it is a device-side DSA_ERR_DEVICE_BOUNDS.
 *  seq_lens           int32 [R]: row r only sees token positions < seq_lens[r].
 *  sel_indices        int32 [R, sel_width] selected token ids, -1 = hole.
 *  sel_width          1..DSA_MAX_SEL_WIDTH.
 *  num_seqs, rows_per_seq, num_q_heads  >= 1.
 *  block_size         tokens per page, >= 1.
 *  cache_stride_bytes bytes per page, >= block_size*512 and a multiple of 16
 *                     (block_size*512 for a dense pool: decode_k.rs, cache_stride_bytes).
 *  k_scale, v_scale   cache dequantisation scales (attend.rs, DsaDecodeInputs).
 *  sm_scale           score scale; the pages' launcher passes kv_lora_rank^-0.5, since
 *                     the scores are formed over the 512-wide latent (attend.rs,
 *                     decode_attention).
 *  out                bf16 [R, num_q_heads, 512], latent space. 16-byte aligned.
 *
 * Uses a library-owned workspace per device, grown on demand with cudaMalloc; growing
 * it while the stream is being captured into a graph returns DSA_ERR_WORKSPACE (use
 * dsa_mla_decode_ws with caller memory for capture).
 */
int32_t dsa_mla_decode(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                       const int32_t* seq_lens, const int32_t* sel_indices, int32_t sel_width,
                       int32_t num_seqs, int32_t rows_per_seq, int32_t num_q_heads,
                       int32_t block_size, int64_t cache_stride_bytes, float k_scale,
                       float v_scale, float sm_scale, void* out, void* stream);

/*
 * dsa_mla_decode_k: k consecutive verify rows per sequence (decode_k.rs, decode_k and
 * attend_rows). Arguments as dsa_mla_decode with rows_per_seq = k, except:
 *  seq_lens  int32 [num_seqs]: the sequence length seq_len before the k new tokens.
 *            Row i (0 <= i < k) of sequence s sits at position seq_len + i and sees
 *            positions < seq_lens[s] + i + 1: each row's visible length is its own
 *            position plus one (decode_k.rs, decode_k).
 * All k rows of a sequence share its block table.
 */
int32_t dsa_mla_decode_k(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, int32_t max_blocks_per_seq,
                         const int32_t* seq_lens, const int32_t* sel_indices, int32_t sel_width,
                         int32_t num_seqs, int32_t k, int32_t num_q_heads, int32_t block_size,
                         int64_t cache_stride_bytes, float k_scale, float v_scale,
                         float sm_scale, void* out, void* stream);

/*
 * Bytes of caller workspace dsa_mla_decode_ws needs for this shape. num_ctas is the
 * decode grid size to plan for (0 = the default for the current device, which needs a
 * CUDA device; returns 0 if none is available).
 */
size_t dsa_mla_decode_workspace_bytes(int32_t num_seqs, int32_t rows_per_seq,
                                      int32_t num_q_heads, int32_t sel_width, int32_t num_ctas);

/*
 * Decode grid size (CTAs) that a call of this shape runs with: num_ctas itself when it
 * is positive, else the default for the current device (0 if no CUDA device is
 * available or an argument is out of range). The default takes at most one CTA per SM
 * and at least 128 slots (selection positions of one 64-head group of one row) per CTA,
 * and prefers a count aligned with the units (rows x 64-head groups): a multiple of the
 * unit count or a divisor of it, when one is at least three quarters of that bound.
 */
int32_t dsa_mla_decode_grid(int32_t num_seqs, int32_t rows_per_seq, int32_t num_q_heads,
                            int32_t sel_width, int32_t num_ctas);

/*
 * Per-call options of dsa_mla_decode_ws (NULL = all defaults). Zero-initialise and set the
 * fields you need; zero means "default" in every field. The source pages have no
 * counterpart to these options: they choose between equivalent launch shapes or serve
 * measurement and testing, and never change what is computed beyond floating-point
 * rounding order.
 *  num_ctas       decode grid size; 0 = default (dsa_mla_decode_grid: at most the SM count).
 *                 Must match the num_ctas the workspace was sized for.
 *  tile_tokens    KV tokens per decode tile: 0 = automatic (64-token tiles when each
 *                 decode CTA has at most 256 selected slots of work or when k_cache and
 *                 v_cache are different buffers, 128 otherwise), 64 or 128 = that size.
 *                 Any other value is DSA_ERR_INVALID_ARGUMENT.
 *  gather_mode    how the decode fetches cache rows: 0 = default (per-thread 16-byte
 *                 copies), 1 = per-thread copies, 2 = tensor-map four-row gathers when
 *                 the pages are dense (cache_stride_bytes = block_size*512) and the caches
 *                 are 128-byte aligned, per-thread copies otherwise. The gathers give the
 *                 same results; on GB300 they measured slower than the copies. Any other
 *                 value is DSA_ERR_INVALID_ARGUMENT.
 *  wait_limit_ns  time limit of every pipeline wait inside the decode kernel; 0 = the
 *                 default of one second. A wait that runs out records DSA_ERR_TIMEOUT in
 *                 the status word, stops the kernel's pipeline and leaves the output
 *                 undefined; the kernel still drains its own copies and tensor-core work
 *                 before it exits. A small limit is only useful to exercise that path;
 *                 a limit below 500 ns makes every wait that is not already complete
 *                 when first checked give up at once.
 *  ev_begin, ev_end  optional cudaEvent_t (as void*) recorded on the stream immediately
 *                 before and after the main decode kernel (inside graph capture they
 *                 become event-record nodes).
 */
typedef struct dsa_decode_options {
    int32_t num_ctas;
    int32_t tile_tokens;
    int32_t gather_mode;
    int32_t reserved; /* must be 0 */
    uint64_t wait_limit_ns;
    void* ev_begin;
    void* ev_end;
} dsa_decode_options;

/*
 * dsa_mla_decode_ws: dsa_mla_decode / dsa_mla_decode_k with caller-owned workspace
 * (device memory, 256-byte aligned, >= dsa_mla_decode_workspace_bytes for the same
 * shape and num_ctas). Never allocates, so it can be captured into a CUDA graph.
 *  verify_rows   0: seq_lens is per row (dsa_mla_decode); 1: seq_lens is per sequence
 *                and rows follow the verify rule (dsa_mla_decode_k).
 *  options       per-call options (see dsa_decode_options), or NULL.
 * The first 256 bytes of the workspace hold the device status word of the latest call.
 */
int32_t dsa_mla_decode_ws(const void* q, const void* k_cache, const void* v_cache,
                          const int32_t* block_tables, int32_t max_blocks_per_seq,
                          const int32_t* seq_lens, const int32_t* sel_indices, int32_t sel_width,
                          int32_t num_seqs, int32_t rows_per_seq, int32_t num_q_heads,
                          int32_t block_size, int64_t cache_stride_bytes, float k_scale,
                          float v_scale, float sm_scale, void* out, int32_t verify_rows,
                          void* workspace, size_t workspace_bytes,
                          const dsa_decode_options* options, void* stream);

/*
 * dsa_mla_decode_host: the same decode with the per-step inputs and the output in HOST
 * memory (pinned for asynchronous copies). The caches stay device-resident. The call
 * copies q, block_tables (table_rows * max(max_blocks_per_seq,1) entries), seq_lens and
 * sel_indices into device staging inside `workspace`, runs the decode and copies out
 * back, all on `stream`; the output is valid after the stream synchronises.
 *  table_rows   rows of block_tables to copy (num_seqs, or 1 for a shared table).
 *  workspace    >= dsa_mla_decode_host_workspace_bytes(...).
 */
size_t dsa_mla_decode_host_workspace_bytes(int32_t num_seqs, int32_t rows_per_seq,
                                           int32_t num_q_heads, int32_t sel_width,
                                           int32_t table_rows, int32_t max_blocks_per_seq,
                                           int32_t verify_rows, int32_t num_ctas);
int32_t dsa_mla_decode_host(const void* q_host, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables_host, int32_t table_rows,
                            int32_t max_blocks_per_seq, const int32_t* seq_lens_host,
                            const int32_t* sel_indices_host, int32_t sel_width, int32_t num_seqs,
                            int32_t rows_per_seq, int32_t num_q_heads, int32_t block_size,
                            int64_t cache_stride_bytes, float k_scale, float v_scale,
                            float sm_scale, void* out_host, int32_t verify_rows,
                            void* workspace, size_t workspace_bytes, int32_t num_ctas,
                            void* stream);

/*
 * dsa_resolve_indices: the index resolution step on its own (attend.rs module doc: -1
 * holes, set membership with duplicates collapsed). For each row: the distinct ids
 * 0 <= id < seq_lens[r] in ascending order, then -1 padding to sel_width.
 *  ids_out     int32 [rows, sel_width]; counts_out int32 [rows].
 */
int32_t dsa_resolve_indices(const int32_t* sel_indices, const int32_t* seq_lens,
                            int32_t sel_width, int32_t rows, int32_t* ids_out,
                            int32_t* counts_out, void* stream);

/*
 * dsa_latent_write: the cache writer that produces the rows the decode reads (decode_k.rs,
 * decode_k: the latent_write launch, one per new token). For each row i with slots[i] >= 0:
 *   y[c] = kv_a[i,c] / sqrt(mean_c kv_a[i,c]^2 + rms_eps) * norm_weight[c] * (1/kv_scale)
 * is stored as E4M3 (round to nearest even, saturating to +-448) in the 512 bytes at
 *   cache + (slots[i] / block_size)*cache_stride_bytes + (slots[i] % block_size)*512,
 * slot = physical_page*block_size + position % block_size as the pages compute it. The
 * kernel body is not on the pages; this RMSNorm-then-scale order is the plain reading.
 * 1/kv_scale is formed in single precision, as the pages' launcher does.
 *  kv_a         bf16 [rows, 512], 16-byte aligned (the kv_a projection of the new tokens).
 *  norm_weight  bf16 [512], 16-byte aligned (the kv_a RMSNorm weight).
 *  slots        int64 [rows], 8-byte aligned; a negative slot writes nothing.
 *  rows >= 0 (kv_a and slots may be null when rows == 0); rms_eps >= 0; kv_scale finite
 *  and non-zero.
 *  block_size, cache_stride_bytes  as for dsa_mla_decode (stride >= block_size*512, a
 *               multiple of 16); cache 16-byte aligned.
 * The pool size is not an argument: a slot past the pool is the caller's error, as a
 * block-table entry past it is for the decode. Rows with the same slot race.
 */
int32_t dsa_latent_write(const void* kv_a, const void* norm_weight, const int64_t* slots,
                         int32_t rows, float rms_eps, float kv_scale, int32_t block_size,
                         int64_t cache_stride_bytes, void* cache, void* stream);

/*
 * dsa_select_pools: the selector that makes the decode's sel_indices rows (attend.rs
 * module doc: a [q_rows, width] row of token ids with -1 holes; decode_k.rs decode_k: the
 * index_topk pools of highest indexer score, row r taking only pools that end at or before
 * its position q_pos[r]). Pool p covers positions p*kpool .. p*kpool + kpool - 1 and is
 * eligible for row r when (p + 1)*kpool - 1 <= q_pos[r]. Per row, the topk eligible pools
 * of highest score are taken (equal scores: the lower pool; NaN ranks below every number;
 * -0 equals +0) and written in ascending position, kpool consecutive ids each, then -1 up
 * to topk*kpool entries. The selector's body is not on the pages; this is the reading taken.
 *  scores   float32 [rows, n_pools] pooled scores; q_pos int32 [rows]; ids_out int32
 *           [rows, topk*kpool]; all 4-byte aligned.
 *  rows, n_pools >= 0 (the arrays may be null when rows == 0, scores when n_pools == 0);
 *  kpool, topk >= 1; n_pools*kpool and topk*kpool below 2^31
 *  (DSA_ERR_UNSUPPORTED otherwise).
 */
int32_t dsa_select_pools(const float* scores, const int32_t* q_pos, int32_t rows,
                         int32_t n_pools, int32_t kpool, int32_t topk, int32_t* ids_out,
                         void* stream);

/*
 * dsa_absorb_q, dsa_absorb_o: the load-time transforms of absorbed MLA (build.rs,
 * absorb_q and absorb_o), the pair that puts the decode's queries and outputs in the
 * kv_lora_rank-dim latent space (NoPE: no rope section). All matrices row-major, BF16
 * weights as the checkpoint stores them, FP32 accumulation on the tensor cores (cuBLAS),
 * output FP32 (out_dtype 0) or BF16 rounded to nearest even (out_dtype 1):
 *   q_absorb[h*kvl + c][k] = sum_{r < nope} kv_b[h*(nope+vd) + r][c] * q_b[h*nope + r][k]
 *   o_absorb[i][h*kvl + c] = sum_{r < vd} o_proj[i][h*vd + r] * kv_b[h*(nope+vd) + nope + r][c]
 *  q_b     bf16 [heads*nope, q_lora_rank]   (the query up-projection, per head nope rows)
 *  kv_b    bf16 [heads*(nope+vd), kvl]      (per head: nope K rows, then vd V rows)
 *  o_proj  bf16 [hidden, heads*vd]          (the output projection)
 *  out     [heads*kvl, q_lora_rank] for absorb_q, [hidden, heads*kvl] for absorb_o;
 *          caller-owned device memory, 4-byte (FP32) or 2-byte (BF16) aligned.
 *  heads, nope, vd, kvl, q_lora_rank, hidden >= 1; heads*(nope+vd), heads*kvl and
 *  heads*vd below 2^31 (DSA_ERR_UNSUPPORTED otherwise). Inputs 2-byte aligned.
 * Enqueued on `stream`; returns DSA_ERR_CUDA when the library GEMM fails.
 */
int32_t dsa_absorb_q(const void* q_b, const void* kv_b, int32_t heads, int32_t nope, int32_t vd,
                     int32_t kvl, int32_t q_lora_rank, void* out, int32_t out_dtype, void* stream);
int32_t dsa_absorb_o(const void* o_proj, const void* kv_b, int32_t heads, int32_t nope, int32_t vd,
                     int32_t kvl, int32_t hidden, void* out, int32_t out_dtype, void* stream);

/*
 * dsa_mla_decode_static: dsa_mla_decode for callers that cannot allocate device memory at
 * call time (for instance code running under a framework that owns all device memory
 * through its own pool, or a latency-critical path that cannot accept cudaMalloc's
 * device-wide synchronisation) and that do not keep a workspace of their own. Arguments,
 * semantics and errors as dsa_mla_decode; it never calls cudaMalloc, cudaFree or any
 * allocating routine. Its scratch is a fixed device array of DSA_STATIC_SCRATCH_BYTES
 * (40 MiB) in the library, present on every GPU that loads the library until the process
 * exits; a shape whose workspace (dsa_mla_decode_workspace_bytes with num_ctas = 0) is
 * larger returns DSA_ERR_WORKSPACE and enqueues nothing.
 *  - The first call on a device looks up the array's device address (cudaGetSymbolAddress)
 *    with that device current; make that first call before any stream capture.
 *  - All calls share the one array: calls whose work overlaps on the GPU (other streams or
 *    threads) race on it and must be serialised by the caller.
 * The source pages have no counterpart to this entry point.
 */
#define DSA_STATIC_SCRATCH_BYTES (40u * 1024u * 1024u)
int32_t dsa_mla_decode_static(const void* q, const void* k_cache, const void* v_cache,
                              const int32_t* block_tables, int32_t max_blocks_per_seq,
                              const int32_t* seq_lens, const int32_t* sel_indices, int32_t sel_width,
                              int32_t num_seqs, int32_t rows_per_seq, int32_t num_q_heads,
                              int32_t block_size, int64_t cache_stride_bytes, float k_scale,
                              float v_scale, float sm_scale, void* out, void* stream);

/*
 * Device status of the latest call on a caller workspace (dsa_mla_decode_ws /
 * dsa_mla_decode_host), on the library workspace of the current device
 * (dsa_last_device_status), or on the fixed array of dsa_mla_decode_static
 * (dsa_static_device_status; like that entry point it allocates nothing). Each
 * synchronises the stream, writes the status to *status_out and returns DSA_OK, or
 * returns DSA_ERR_CUDA.
 */
int32_t dsa_read_device_status(const void* workspace, int32_t* status_out, void* stream);
int32_t dsa_last_device_status(int32_t* status_out, void* stream);
int32_t dsa_static_device_status(int32_t* status_out, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_MLA_H */
