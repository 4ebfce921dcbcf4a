/*
 * Oracle for the selected-index (DSA) NoPE MLA paged decode.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, obviously correct CPU
 * statement of what the decode computes. Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference arm may build, load or call it; the product
 * path never does. It shares no code, header, table or constant with the CUDA path.
 *
 * Arithmetic is IEEE double throughout. Every function names the passage of the
 * source pages it restates:
 *
 *   [attend.rs]   spark_model/layers/glm5next_dsa/attend.rs
 *   [decode_k.rs] metrale_model_arch/glm5next_dsa/layer/decode_k.rs
 *
 * Parity pins (how this oracle is checked against something other than itself) live
 * in tests/test_oracle_pins.py: a dense masked brute force written independently in
 * numpy, FP8 decode against torch.float8_e4m3fn and the OCP table values, closed
 * forms (single token, all holes, zero query, large scale), and invariants
 * (permutation, duplication, extra holes). The exact softmax values at full
 * configuration scale are pinned only through those properties.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define LATENT 512 /* kv_lora_rank: the whole cache token under NoPE ([attend.rs] module doc, "NoPE") */

/* ------------------------------------------------------------------------------------
 * Element decoding.
 * ---------------------------------------------------------------------------------- */

/* FP8 E4M3 ("fn" variant of the OCP 8-bit floating point specification): 1 sign bit,
 * 4 exponent bits with bias 7, 3 mantissa bits; exponent field 0 encodes subnormals
 * m/8 * 2^-6; exponent 15 with mantissa 7 is NaN; there is no infinity. The cache is
 * "FP8" in [attend.rs] (DsaDecodeInputs::k_cache); E4M3 is the reading taken. */
double oracle_e4m3_to_f64(uint8_t code) {
    int sign = (code >> 7) & 1;
    int exponent = (code >> 3) & 0xF;
    int mantissa = code & 0x7;
    double magnitude;
    if (exponent == 0xF && mantissa == 0x7) return NAN;
    if (exponent == 0)
        magnitude = ldexp((double)mantissa / 8.0, 1 - 7);
    else
        magnitude = ldexp(1.0 + (double)mantissa / 8.0, exponent - 7);
    return sign ? -magnitude : magnitude;
}

/* BF16: the upper 16 bits of an IEEE binary32 ([attend.rs] DsaDecodeInputs::q). */
double oracle_bf16_to_f64(uint16_t bits) {
    uint32_t word = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &word, sizeof f);
    return (double)f;
}

void oracle_e4m3_table(double* out256) {
    for (int c = 0; c < 256; ++c) out256[c] = oracle_e4m3_to_f64((uint8_t)c);
}

/* ------------------------------------------------------------------------------------
 * Index resolution.
 *
 * [attend.rs] module doc: a selection row is a list of token ids in which -1 is a hole,
 * and the reference mask is pure set membership with duplicates collapsed. Row r may
 * only see positions below its own seq_len ([decode_k.rs] decode_k: row r's seq_len
 * entry is pos + 1; bt_entries_needed: row r attends tokens below its seq_len). Reading
 * taken: any id < 0 or >= seq_lens[r] is a hole. The resolved set is written in
 * ascending order, padded with -1, so that it has one canonical form.
 * ---------------------------------------------------------------------------------- */

static int cmp_i32(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/* Resolves one row; returns the number of distinct valid ids written to ids_out[0..). */
static int32_t resolve_row(const int32_t* sel_row, int32_t sel_width, int32_t seq_len,
                           int32_t* ids_out) {
    int32_t n = 0;
    for (int32_t j = 0; j < sel_width; ++j) {
        int32_t id = sel_row[j];
        if (id >= 0 && id < seq_len) ids_out[n++] = id;
    }
    qsort(ids_out, (size_t)n, sizeof(int32_t), cmp_i32);
    int32_t u = 0;
    for (int32_t j = 0; j < n; ++j)
        if (u == 0 || ids_out[u - 1] != ids_out[j]) ids_out[u++] = ids_out[j];
    for (int32_t j = u; j < sel_width; ++j) ids_out[j] = -1;
    return u;
}

int32_t oracle_resolve_indices(const int32_t* sel_indices, const int32_t* seq_lens,
                               int32_t sel_width, int32_t rows, int32_t* ids_out,
                               int32_t* counts_out) {
    if (sel_width < 0 || rows < 0) return -1;
    for (int32_t r = 0; r < rows; ++r)
        counts_out[r] = resolve_row(sel_indices + (int64_t)r * sel_width, sel_width,
                                    seq_lens[r], ids_out + (int64_t)r * sel_width);
    return 0;
}

/* ------------------------------------------------------------------------------------
 * Decode.
 *
 * For decode row r of sequence seq = r / rows_per_seq and every query head h
 * ([attend.rs] decode_attention and DsaDecodeInputs):
 *   S      = resolved ids of row r (above)
 *   K_j[c] = k_scale * e4m3(k_cache[page(j)*cache_stride_bytes + (j % block_size)*512 + c])
 *   V_j[c] = v_scale * e4m3(v_cache[ same byte offset ])
 *   page(j) = block_tables[seq*max_blocks_per_seq + j / block_size]
 *            ([decode_k.rs] decode_k: physical = block_table[pos / block_size],
 *             slot = physical*block_size + pos % block_size; the page stride is
 *             block_size * kv_lora_rank bytes, passed as cache_stride_bytes)
 *   s_j    = sm_scale * sum_c q[r,h,c] * K_j[c]
 *   out[r,h,c] = sum_j exp(s_j - max s) V_j[c] / sum_j exp(s_j - max s),   0 if S is empty.
 * The row stride of block_tables is max_blocks_per_seq; 0 means every sequence reads
 * row 0 ([decode_k.rs] decode_k, "read with a row stride of 0").
 * ---------------------------------------------------------------------------------- */

typedef struct {
    const uint16_t* q;
    const uint8_t* k_cache;
    const uint8_t* v_cache;
    int64_t cache_bytes;
    const int32_t* block_tables;
    int32_t max_blocks_per_seq;
    const int32_t* seq_lens;
    int32_t sel_width;
    int32_t rows_per_seq;
    int32_t num_q_heads;
    int32_t block_size;
    int64_t cache_stride_bytes;
    double k_scale, v_scale, sm_scale;
    const int32_t* rows;      /* which decode rows to evaluate */
    int32_t n_rows;
    const int32_t* resolved;  /* [n_rows, sel_width] */
    const int32_t* counts;    /* [n_rows] */
    double* out;              /* [n_rows, num_q_heads, 512] */
    double e4m3[256];
    int32_t next_task;        /* shared work counter, guarded by lock */
    pthread_mutex_t lock;
    int32_t error;
} decode_job;

static int64_t token_byte_offset(const decode_job* J, int32_t seq, int32_t id, int* ok) {
    int64_t entry = (int64_t)seq * J->max_blocks_per_seq + id / J->block_size;
    int32_t page = J->block_tables[entry];
    int64_t off = (int64_t)page * J->cache_stride_bytes + (int64_t)(id % J->block_size) * LATENT;
    *ok = page >= 0 && off >= 0 && off + LATENT <= J->cache_bytes;
    return off;
}

/* One (row, head) task: the definition above, written out. */
static void decode_one(decode_job* J, int32_t task) {
    int32_t i = task / J->num_q_heads;
    int32_t h = task % J->num_q_heads;
    int32_t r = J->rows[i];
    int32_t seq = r / J->rows_per_seq;
    int32_t n = J->counts[i];
    const int32_t* S = J->resolved + (int64_t)i * J->sel_width;
    const uint16_t* qh = J->q + ((int64_t)r * J->num_q_heads + h) * LATENT;
    double* o = J->out + ((int64_t)i * J->num_q_heads + h) * LATENT;
    double qd[LATENT];
    for (int c = 0; c < LATENT; ++c) {
        qd[c] = oracle_bf16_to_f64(qh[c]);
        o[c] = 0.0;
    }
    if (n == 0) return; /* empty set: output is zero */

    double* s = (double*)malloc(sizeof(double) * (size_t)n);
    int64_t* off = (int64_t*)malloc(sizeof(int64_t) * (size_t)n);
    double m = -INFINITY;
    for (int32_t j = 0; j < n; ++j) {
        int ok;
        off[j] = token_byte_offset(J, seq, S[j], &ok);
        if (!ok) {
            pthread_mutex_lock(&J->lock);
            J->error = -2;
            pthread_mutex_unlock(&J->lock);
            free(s);
            free(off);
            return;
        }
        const uint8_t* krow = J->k_cache + off[j];
        double dot = 0.0;
        for (int c = 0; c < LATENT; ++c) dot += qd[c] * (J->k_scale * J->e4m3[krow[c]]);
        s[j] = J->sm_scale * dot;
        if (s[j] > m) m = s[j];
    }
    double z = 0.0;
    for (int32_t j = 0; j < n; ++j) {
        double w = exp(s[j] - m);
        z += w;
        const uint8_t* vrow = J->v_cache + off[j];
        for (int c = 0; c < LATENT; ++c) o[c] += w * (J->v_scale * J->e4m3[vrow[c]]);
    }
    for (int c = 0; c < LATENT; ++c) o[c] /= z;
    free(s);
    free(off);
}

static void* decode_worker(void* arg) {
    decode_job* J = (decode_job*)arg;
    int32_t total = J->n_rows * J->num_q_heads;
    for (;;) {
        pthread_mutex_lock(&J->lock);
        int32_t t = J->next_task++;
        pthread_mutex_unlock(&J->lock);
        if (t >= total) break;
        decode_one(J, t);
    }
    return NULL;
}

/* Returns 0 on success, -1 on a bad argument, -2 when a selected token resolves outside
 * the cache (a caller contract violation). threads <= 0 uses every online core. */
int32_t oracle_dsa_mla_decode(const uint16_t* q, const uint8_t* k_cache, const uint8_t* v_cache,
                              int64_t cache_bytes, const int32_t* block_tables,
                              int32_t max_blocks_per_seq, const int32_t* seq_lens,
                              const int32_t* sel_indices, int32_t sel_width, int32_t num_seqs,
                              int32_t rows_per_seq, int32_t num_q_heads, int32_t block_size,
                              int64_t cache_stride_bytes, double k_scale, double v_scale,
                              double sm_scale, const int32_t* rows, int32_t n_rows, double* out,
                              int32_t threads) {
    if (num_seqs < 1 || rows_per_seq < 1 || num_q_heads < 1 || block_size < 1 || sel_width < 1 ||
        max_blocks_per_seq < 0 || n_rows < 0)
        return -1;
    int32_t total_rows = num_seqs * rows_per_seq;
    for (int32_t i = 0; i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= total_rows) return -1;

    decode_job* J = (decode_job*)calloc(1, sizeof(decode_job));
    J->q = q;
    J->k_cache = k_cache;
    J->v_cache = v_cache;
    J->cache_bytes = cache_bytes;
    J->block_tables = block_tables;
    J->max_blocks_per_seq = max_blocks_per_seq;
    J->seq_lens = seq_lens;
    J->sel_width = sel_width;
    J->rows_per_seq = rows_per_seq;
    J->num_q_heads = num_q_heads;
    J->block_size = block_size;
    J->cache_stride_bytes = cache_stride_bytes;
    J->k_scale = k_scale;
    J->v_scale = v_scale;
    J->sm_scale = sm_scale;
    J->rows = rows;
    J->n_rows = n_rows;
    J->out = out;
    oracle_e4m3_table(J->e4m3);
    pthread_mutex_init(&J->lock, NULL);

    int32_t* resolved = (int32_t*)malloc(sizeof(int32_t) * (size_t)n_rows * (size_t)sel_width + 4);
    int32_t* counts = (int32_t*)malloc(sizeof(int32_t) * (size_t)n_rows + 4);
    for (int32_t i = 0; i < n_rows; ++i)
        counts[i] = resolve_row(sel_indices + (int64_t)rows[i] * sel_width, sel_width,
                                seq_lens[rows[i]], resolved + (int64_t)i * sel_width);
    J->resolved = resolved;
    J->counts = counts;

    if (threads <= 0) threads = (int32_t)sysconf(_SC_NPROCESSORS_ONLN);
    if (threads < 1) threads = 1;
    if (threads > n_rows * num_q_heads) threads = n_rows * num_q_heads;
    if (threads <= 1) {
        decode_worker(J);
    } else {
        pthread_t* tids = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)threads);
        for (int32_t t = 0; t < threads; ++t) pthread_create(&tids[t], NULL, decode_worker, J);
        for (int32_t t = 0; t < threads; ++t) pthread_join(tids[t], NULL);
        free(tids);
    }
    int32_t err = J->error;
    pthread_mutex_destroy(&J->lock);
    free(resolved);
    free(counts);
    free(J);
    return err;
}

int32_t oracle_online_cores(void) { return (int32_t)sysconf(_SC_NPROCESSORS_ONLN); }

/* ------------------------------------------------------------------------------------
 * Cache writer.
 *
 * [decode_k.rs] decode_k, the latent_write launch: for each new token the kernel is given
 * the row's kv_a (kv_lora_rank BF16 values), the kv_a RMSNorm weight (BF16), the cache
 * pool, the token's slot = physical*block_size + pos % block_size, rms_eps and
 * 1/kv_scale (a single-precision value computed on the host). The kernel body is not on
 * the pages. Reading taken: the plain RMSNorm followed by the cache scale,
 *   y[c] = x[c] / sqrt(mean_c x^2 + eps) * w[c] * (1/kv_scale),
 * stored as E4M3 (round to nearest even, saturating to +-448) at byte
 *   (slot / block_size)*cache_stride_bytes + (slot % block_size)*512 + c,
 * the layout the decode reads. A negative slot writes nothing.
 * ---------------------------------------------------------------------------------- */

/* E4M3 ("fn") code of v from the format's definition: magnitudes of 448 and above
 * saturate to 448 (0x7E); normal values have 3 mantissa bits after the implicit 1 and
 * exponents -6..8; below 2^-6 the subnormals m/8 * 2^-6. Ties round to the even code. */
uint8_t oracle_e4m3_encode(double v) {
    if (isnan(v)) return 0x7F;
    uint8_t sign = signbit(v) ? 0x80 : 0x00;
    double a = fabs(v);
    if (a >= 448.0) return sign | 0x7E;
    if (a < ldexp(1.0, -6)) {
        double m = nearbyint(ldexp(a, 9)); /* units of 2^-9, round half to even */
        if (m >= 8.0) return sign | 0x08;  /* rounded up to the smallest normal, 2^-6 */
        return sign | (uint8_t)m;
    }
    int k;
    double f = frexp(a, &k);                  /* a = f * 2^k, f in [0.5, 1) */
    int e = k - 1;                            /* a = (2f) * 2^e, 2f in [1, 2) */
    double m = nearbyint((2.0 * f - 1.0) * 8.0);
    if (m >= 8.0) {
        m = 0.0;
        e += 1;
    }
    return sign | (uint8_t)((e + 7) << 3) | (uint8_t)m;
}

/* Writes rows tokens; values_out (may be NULL) receives each element's value before the
 * E4M3 rounding, [rows, 512]. Returns 0, -1 on bad arguments, -2 when a slot's bytes fall
 * outside cache_bytes. */
int32_t oracle_latent_write(const uint16_t* kv_a, const uint16_t* weight, const int64_t* slots, int32_t rows,
                            double rms_eps, double inv_kv_scale, int32_t block_size,
                            int64_t cache_stride_bytes, uint8_t* cache, int64_t cache_bytes,
                            double* values_out) {
    if (rows < 0 || block_size < 1 || cache_stride_bytes < (int64_t)block_size * LATENT) return -1;
    for (int32_t r = 0; r < rows; ++r) {
        const int64_t slot = slots[r];
        if (slot < 0) continue;
        const uint16_t* x = kv_a + (int64_t)r * LATENT;
        double sumsq = 0.0;
        for (int c = 0; c < LATENT; ++c) {
            double xc = oracle_bf16_to_f64(x[c]);
            sumsq += xc * xc;
        }
        const double inv_rms = 1.0 / sqrt(sumsq / LATENT + rms_eps);
        const int64_t base = (slot / block_size) * cache_stride_bytes + (slot % block_size) * LATENT;
        if (base < 0 || base + LATENT > cache_bytes) return -2;
        for (int c = 0; c < LATENT; ++c) {
            double y = oracle_bf16_to_f64(x[c]) * inv_rms * oracle_bf16_to_f64(weight[c]) * inv_kv_scale;
            if (values_out) values_out[(int64_t)r * LATENT + c] = y;
            cache[base + c] = oracle_e4m3_encode(y);
        }
    }
    return 0;
}

/* ------------------------------------------------------------------------------------
 * Selector.
 *
 * [attend.rs] module doc: the decode consumes a [q_rows, out_width] i32 row of token ids
 * with -1 holes, produced by the selector; [attend.rs] DsaDecodePaging::validate: pools
 * are built over absolute positions, index_kpool positions each; [decode_k.rs] decode_k:
 * the selection takes index_topk pools, and row r only takes pools that end at or before
 * its position q_pos[r]. The selector's body is not on the pages. Reading taken: pool p
 * (positions p*kpool .. p*kpool + kpool - 1) is eligible for row r when
 * (p + 1)*kpool - 1 <= q_pos[r]; the index_topk eligible pools of highest score are taken
 * (equal scores: the lower pool first; NaN ranks below every number); the row lists the
 * taken pools in ascending position, each as its kpool consecutive ids, then -1 up to
 * index_topk*kpool entries.
 * ---------------------------------------------------------------------------------- */

typedef struct {
    float score;
    int32_t pool;
} pool_rank_t;

/* Orders by score descending (NaN last), then pool ascending. */
static int cmp_pool_rank(const void* a, const void* b) {
    const pool_rank_t* x = (const pool_rank_t*)a;
    const pool_rank_t* y = (const pool_rank_t*)b;
    int xn = isnan(x->score), yn = isnan(y->score);
    if (xn != yn) return xn - yn;
    if (!xn && x->score != y->score) return x->score > y->score ? -1 : 1;
    return (x->pool > y->pool) - (x->pool < y->pool);
}

int32_t oracle_select_pools(const float* scores, const int32_t* q_pos, int32_t rows, int32_t n_pools,
                            int32_t kpool, int32_t topk, int32_t* ids_out) {
    if (rows < 0 || n_pools < 0 || kpool < 1 || topk < 1) return -1;
    pool_rank_t* cand = (pool_rank_t*)malloc(sizeof(pool_rank_t) * (size_t)(n_pools > 0 ? n_pools : 1));
    int32_t* taken = (int32_t*)malloc(sizeof(int32_t) * (size_t)topk);
    for (int32_t r = 0; r < rows; ++r) {
        int32_t n = 0;
        for (int32_t p = 0; p < n_pools; ++p)
            if ((int64_t)(p + 1) * kpool - 1 <= (int64_t)q_pos[r]) {
                cand[n].score = scores[(int64_t)r * n_pools + p];
                cand[n].pool = p;
                ++n;
            }
        qsort(cand, (size_t)n, sizeof(pool_rank_t), cmp_pool_rank);
        int32_t m = n < topk ? n : topk;
        for (int32_t i = 0; i < m; ++i) taken[i] = cand[i].pool;
        qsort(taken, (size_t)m, sizeof(int32_t), cmp_i32);
        int32_t* out = ids_out + (int64_t)r * topk * kpool;
        int64_t o = 0;
        for (int32_t i = 0; i < m; ++i)
            for (int32_t t = 0; t < kpool; ++t) out[o++] = taken[i] * kpool + t;
        for (; o < (int64_t)topk * kpool; ++o) out[o] = -1;
    }
    free(cand);
    free(taken);
    return 0;
}

/* ------------------------------------------------------------------------------------
 * Load-time transforms of absorbed MLA.
 *
 * [build.rs] absorb_q: the query up-projection q_b is pre-multiplied by the K half of
 * kv_b, so that queries arrive in the kvl-dim latent space the decode dots against:
 *   q_absorb[h*kvl + c][k] = sum_{r < nope} kv_b[h*(nope+vd) + r][c] * q_b[h*nope + r][k]
 * with q_b [heads*nope, ql], kv_b [heads*(nope+vd), kvl], q_absorb [heads*kvl, ql].
 * [build.rs] absorb_o: the output projection is pre-multiplied by the V half of kv_b
 * (rows nope .. nope+vd-1 of each head's block), so that it reads the decode's latent
 * output:
 *   o_absorb[i][h*kvl + c] = sum_{r < vd} o_proj[i][h*vd + r] * kv_b[h*(nope+vd) + nope + r][c]
 * with o_proj [hidden, heads*vd], o_absorb [hidden, heads*kvl]. All matrices row-major;
 * NoPE (no rope section, [build.rs] absorb_q refuses one). Inputs are the checkpoint's
 * BF16 values; the sums are in double. Only output rows [row0, row0 + nrows) are written
 * (out points at row row0), so a large transform can be checked on sampled rows.
 * ---------------------------------------------------------------------------------- */

int32_t oracle_absorb_q(const uint16_t* q_b, const uint16_t* kv_b, int32_t heads, int32_t nope, int32_t vd,
                        int32_t kvl, int32_t ql, int64_t row0, int64_t nrows, double* out) {
    if (heads < 1 || nope < 1 || vd < 0 || kvl < 1 || ql < 1) return -1;
    if (row0 < 0 || nrows < 0 || row0 + nrows > (int64_t)heads * kvl) return -1;
    for (int64_t row = row0; row < row0 + nrows; ++row) {
        const int64_t h = row / kvl, c = row % kvl;
        for (int64_t k = 0; k < ql; ++k) {
            double sum = 0.0;
            for (int64_t r = 0; r < nope; ++r)
                sum += oracle_bf16_to_f64(kv_b[(h * (nope + vd) + r) * kvl + c]) *
                       oracle_bf16_to_f64(q_b[(h * nope + r) * ql + k]);
            out[(row - row0) * ql + k] = sum;
        }
    }
    return 0;
}

int32_t oracle_absorb_o(const uint16_t* o_proj, const uint16_t* kv_b, int32_t heads, int32_t nope, int32_t vd,
                        int32_t kvl, int32_t hidden, int64_t row0, int64_t nrows, double* out) {
    if (heads < 1 || nope < 0 || vd < 1 || kvl < 1 || hidden < 1) return -1;
    if (row0 < 0 || nrows < 0 || row0 + nrows > hidden) return -1;
    const int64_t in_w = (int64_t)heads * vd, out_w = (int64_t)heads * kvl;
    for (int64_t i = row0; i < row0 + nrows; ++i)
        for (int64_t h = 0; h < heads; ++h)
            for (int64_t c = 0; c < kvl; ++c) {
                double sum = 0.0;
                for (int64_t r = 0; r < vd; ++r)
                    sum += oracle_bf16_to_f64(o_proj[i * in_w + h * vd + r]) *
                           oracle_bf16_to_f64(kv_b[(h * (nope + vd) + nope + r) * kvl + c]);
                out[(i - row0) * out_w + h * kvl + c] = sum;
            }
    return 0;
}
