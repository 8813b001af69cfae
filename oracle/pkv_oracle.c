/*
 * Reference (oracle) implementation of one paged-KV decode step, in plain C
 * with fp64 arithmetic.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this library.  It shares no code,
 * header or table with the CUDA library; the two meet only through the seeded
 * inputs of the workload generator.
 *
 * What it computes, and the passage each step follows:
 *   - slot of a token: physical block from the block table at position/bs,
 *     times the block size, plus position mod bs ("vLLM Architecture and
 *     Installation", Example 3, paged KV cache block tables: the worked
 *     slots 13, 24 and 23);
 *   - append: each scheduled token's K and V row is written to its slot
 *     (same Example 3: the runner's slot mapping tells the attention kernel
 *     where new keys and values go);
 *   - decode attention: one query token per sequence reads the sequence's
 *     whole history through its block table (same Example 3) and forms
 *     softmax(scale * q.K^T) . V ("Batching and Scheduling", Example 1:
 *     every sequence reads its own, unshared KV cache each step).  Query head
 *     g reads KV head g / (Hq/Hkv) (grouped-query attention; the pages do not
 *     fix the mapping, contiguous groups are the plain reading).
 *
 * Pool layout (one layer): k_cache[NB][Hkv][bs][D], v_cache likewise.
 *
 * Attention is the plain definition: gather the sequence's K and V through
 * the table into contiguous fp64 arrays, then dense softmax attention with
 * the maximum subtracted before exp.
 *
 * FP8 KV cache ("vLLM Architecture and Installation", Example 6, startup
 * memory profiling and the number of KV blocks: with an FP8 KV cache each
 * value takes one byte instead of two, so blocks halve and the token
 * capacity doubles).  The pages name
 * the 8-bit format but not its layout or scaling; the plain reading taken
 * here is E4M3 (sign, 4-bit exponent with bias 7, 3-bit fraction, no
 * infinities, S.1111.111 is NaN, largest finite 448) with one fp32 scale per
 * layer for K and one for V: a stored byte b stands for scale * e4m3(b), and
 * a value x is stored as the code nearest to the fp32 quotient x / scale
 * (ties to the even code, magnitudes from 448 up saturating to 448).
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_E4M3 = 3 };

static size_t orc_elem_bytes(int dtype) {
    return dtype == ORC_F32 ? 4u : dtype == ORC_E4M3 ? 1u : 2u;
}

/* E4M3 -> double, from the format's definition: sign | 4-bit exponent
 * (bias 7) | 3-bit fraction; exponent 0 holds subnormals frac * 2^-9;
 * exponent 15 with fraction 7 is NaN (there is no infinity). */
static double orc_e4m3_to_double(uint8_t b) {
    int sign = (b >> 7) & 1;
    int expo = (b >> 3) & 0xf;
    int frac = b & 0x7;
    double v;
    if (expo == 15 && frac == 7)
        v = NAN;
    else if (expo == 0)
        v = ldexp((double)frac, -9);
    else
        v = ldexp((double)(8 + frac), expo - 10); /* 1.frac * 2^(e-7) */
    return sign ? -v : v;
}

/* Nearest E4M3 code of a binary32 value, by search over every finite code:
 * the code whose value is closest to x, the even code (fraction LSB 0) on a
 * tie, magnitudes at or above the largest finite value (448) saturate to it,
 * NaN gives 0x7F, the sign is kept (also for zero). */
uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7f;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a = fabs((double)x);
    if (a >= 448.0) return sign | 0x7e;
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7e; ++c) {
        double err = fabs(orc_e4m3_to_double((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return sign | (uint8_t)best;
}

/* Quantize n stored values of src_dtype with one scale: the fp32 quotient
 * x / scale, then the nearest code. */
void oracle_quantize_e4m3(int src_dtype, const void* src, int64_t n, float scale, uint8_t* out);

/* IEEE binary16 -> double, written from the format's definition:
 * sign | 5-bit exponent (bias 15) | 10-bit fraction. */
static double orc_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
    else if (expo == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), expo - 25); /* 1.frac * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 -> double: the top 16 bits of an IEEE binary32. */
static double orc_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double orc_load(const void* base, size_t idx, int dtype) {
    if (dtype == ORC_E4M3) return orc_e4m3_to_double(((const uint8_t*)base)[idx]);
    if (dtype == ORC_F32) {
        float f;
        memcpy(&f, (const char*)base + 4 * idx, 4);
        return (double)f;
    }
    uint16_t h;
    memcpy(&h, (const char*)base + 2 * idx, 2);
    return dtype == ORC_F16 ? orc_half_to_double(h) : orc_bf16_to_double(h);
}

/* Decode n stored values to double (exposed so tests can pin the decoders). */
void oracle_decode(int dtype, const void* src, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = orc_load(src, (size_t)i, dtype);
}

void oracle_quantize_e4m3(int src_dtype, const void* src, int64_t n, float scale, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) {
        float x = (float)orc_load(src, (size_t)i, src_dtype); /* exact: the source is <= 32 bits */
        float y = x / scale;                                   /* binary32 division */
        out[i] = oracle_e4m3_encode(y);
    }
}

/* Physical slot of logical position `pos` of sequence `s`. */
int64_t oracle_slot(const int32_t* block_tables, int max_blocks, int s, int pos, int block_size) {
    int64_t blk = block_tables[(int64_t)s * max_blocks + pos / block_size];
    return blk * block_size + pos % block_size;
}

/* Slot of each sequence's newest token (position ctx-1); -1 where ctx == 0. */
void oracle_slot_mapping(const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                         int num_seqs, int block_size, int32_t* slot_out) {
    for (int s = 0; s < num_seqs; ++s)
        slot_out[s] = context_lens[s] > 0
                          ? (int32_t)oracle_slot(block_tables, max_blocks, s, context_lens[s] - 1, block_size)
                          : -1;
}

/* Write token i's K and V rows ([n_tokens][Hkv][D]) into the pool at
 * slot_mapping[i]; negative slots are skipped.  Returns 0, or -1 (nothing
 * written past the first bad slot) if a slot lies outside the pool. */
int oracle_append(int dtype, int num_blocks, int block_size, int num_kv_heads, int head_dim,
                  void* k_cache, void* v_cache, int n_tokens, const void* k, const void* v,
                  const int32_t* slot_mapping) {
    size_t row = (size_t)head_dim * orc_elem_bytes(dtype);
    for (int i = 0; i < n_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) return -1;
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t dst = (size_t)(((blk * num_kv_heads + h) * block_size + off)) * row;
            size_t src = ((size_t)i * num_kv_heads + h) * row;
            memcpy((char*)k_cache + dst, (const char*)k + src, row);
            memcpy((char*)v_cache + dst, (const char*)v + src, row);
        }
    }
    return 0;
}

/* Append into an E4M3 pool: each K (V) row of src_dtype is quantized with
 * k_scale (v_scale) and its codes written to the row's slot, as
 * oracle_append does for plain rows. */
int oracle_append_e4m3(int src_dtype, int num_blocks, int block_size, int num_kv_heads, int head_dim,
                       uint8_t* k_cache, uint8_t* v_cache, int n_tokens, const void* k, const void* v,
                       const int32_t* slot_mapping, float k_scale, float v_scale) {
    size_t srow = (size_t)head_dim * orc_elem_bytes(src_dtype);
    for (int i = 0; i < n_tokens; ++i) {
        int64_t slot = slot_mapping[i];
        if (slot < 0) continue;
        if (slot >= (int64_t)num_blocks * block_size) return -1;
        int64_t blk = slot / block_size, off = slot % block_size;
        for (int h = 0; h < num_kv_heads; ++h) {
            size_t dst = (size_t)(((blk * num_kv_heads + h) * block_size + off)) * (size_t)head_dim;
            size_t src = ((size_t)i * num_kv_heads + h) * srow;
            oracle_quantize_e4m3(src_dtype, (const char*)k + src, head_dim, k_scale, k_cache + dst);
            oracle_quantize_e4m3(src_dtype, (const char*)v + src, head_dim, v_scale, v_cache + dst);
        }
    }
    return 0;
}

typedef struct {
    int q_dtype, kv_dtype;
    double k_scale, v_scale; /* a stored K (V) element stands for k_scale (v_scale) times its value */
    const void *q, *k_cache, *v_cache;
    const int32_t *tables, *ctx;
    int max_blocks, num_seqs, hq, hkv, d, bs, num_blocks;
    double scale;
    double* out;
    int64_t first, last; /* rows (s, g) handled by this worker */
    int status;
} orc_job;

static void* orc_attend_rows(void* arg) {
    orc_job* J = (orc_job*)arg;
    int G = J->hq / J->hkv, D = J->d;
    int64_t cap = 0;
    double *K = NULL, *V = NULL, *x = NULL, *qd = (double*)malloc(sizeof(double) * (size_t)D);
    for (int64_t r = J->first; r < J->last; ++r) {
        int s = (int)(r / J->hq), g = (int)(r % J->hq);
        int h = g / G;
        int n = J->ctx[s];
        double* o = J->out + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (n <= 0) continue;
        if (n > cap) {
            cap = n;
            K = (double*)realloc(K, sizeof(double) * (size_t)cap * D);
            V = (double*)realloc(V, sizeof(double) * (size_t)cap * D);
            x = (double*)realloc(x, sizeof(double) * (size_t)cap);
        }
        /* 1. gather this sequence's K and V through its block table */
        for (int t = 0; t < n; ++t) {
            int64_t blk = J->tables[(int64_t)s * J->max_blocks + t / J->bs];
            if (blk < 0 || blk >= J->num_blocks) { J->status = -1; blk = 0; }
            int64_t off = t % J->bs;
            size_t base = (size_t)(((blk * J->hkv + h) * J->bs + off)) * D;
            for (int d = 0; d < D; ++d) {
                K[(size_t)t * D + d] = J->k_scale * orc_load(J->k_cache, base + d, J->kv_dtype);
                V[(size_t)t * D + d] = J->v_scale * orc_load(J->v_cache, base + d, J->kv_dtype);
            }
        }
        for (int d = 0; d < D; ++d) qd[d] = orc_load(J->q, (size_t)r * D + d, J->q_dtype);
        /* 2. scores */
        double mx = -INFINITY;
        for (int t = 0; t < n; ++t) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qd[d] * K[(size_t)t * D + d];
            x[t] = J->scale * acc;
            if (x[t] > mx) mx = x[t];
        }
        /* 3. softmax weights and 4. weighted sum of V */
        double sum = 0.0;
        for (int t = 0; t < n; ++t) {
            x[t] = exp(x[t] - mx);
            sum += x[t];
        }
        for (int t = 0; t < n; ++t) {
            double w = x[t] / sum;
            for (int d = 0; d < D; ++d) o[d] += w * V[(size_t)t * D + d];
        }
    }
    free(K);
    free(V);
    free(x);
    free(qd);
    return NULL;
}

/* out[s][g][d] (fp64) = softmax_t(scale * q[s][g] . K_s[t]) . V_s[t] over the
 * context_lens[s] tokens of sequence s; zero rows where the context is empty.
 * q is [num_seqs][Hq][D] in q_dtype, the cache in kv_dtype; a cache element
 * stands for k_scale (v_scale) times its stored value.  nthreads <= 0 uses every online core.
 * Returns 0, or -1 if a table entry lies outside [0, num_blocks). */
int oracle_paged_decode_scaled(int q_dtype, int kv_dtype, double k_scale, double v_scale,
                               const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, int num_blocks, double scale, double* out, int nthreads) {
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return -2;
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    int64_t rows = (int64_t)num_seqs * num_q_heads;
    if (nthreads > rows) nthreads = rows > 0 ? (int)rows : 1;
    orc_job* jobs = (orc_job*)calloc((size_t)nthreads, sizeof(orc_job));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        orc_job j = {q_dtype, kv_dtype, k_scale, v_scale, q, k_cache, v_cache, block_tables, context_lens, max_blocks,
                     num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                     scale, out, rows * i / nthreads, rows * (i + 1) / nthreads, 0};
        jobs[i] = j;
    }
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, orc_attend_rows, &jobs[i]);
    orc_attend_rows(&jobs[0]);
    int status = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (i) pthread_join(th[i], NULL);
        if (jobs[i].status) status = jobs[i].status;
    }
    free(jobs);
    free(th);
    return status;
}

/* Multi-token queries (chunked prefill; "Batching and Scheduling", Example 5,
 * and "vLLM Architecture and Installation", Example 5: a step gives each
 * request a number of new tokens, one for a decoding request, a chunk of the
 * prompt for a prefilling one).  Sequence s brings n_s = query_start[s+1] -
 * query_start[s] new tokens, already appended, so its cache holds
 * context_lens[s] tokens and its new tokens sit at positions
 * context_lens[s] - n_s .. context_lens[s] - 1.  Query token i of s (row
 * query_start[s] + i of q and out, [T][Hq][D]) attends to the cached tokens at
 * positions 0 .. context_lens[s] - n_s + i: softmax(scale q.K^T).V over that
 * causal prefix, read through the block table, fp64. */
typedef struct {
    int q_dtype, kv_dtype;
    double k_scale, v_scale; /* a cache element stands for scale * its stored value */
    const void *q, *k_cache, *v_cache;
    const int32_t *tables, *qstart, *ctx;
    int max_blocks, num_seqs, hq, hkv, d, bs, num_blocks;
    double scale;
    double* out;
    int64_t first, last; /* rows (token, head) handled by this worker */
    int status;
} orc_pjob;

static void* orc_prefill_rows(void* arg) {
    orc_pjob* J = (orc_pjob*)arg;
    int G = J->hq / J->hkv, D = J->d;
    int64_t cap = 0;
    double *x = NULL, *qd = (double*)malloc(sizeof(double) * (size_t)D);
    for (int64_t r = J->first; r < J->last; ++r) {
        int64_t tok = r / J->hq;
        int g = (int)(r % J->hq), h = g / G;
        int s = 0;
        while (s + 1 < J->num_seqs && J->qstart[s + 1] <= tok) ++s; /* sequence of this token */
        int n = J->qstart[s + 1] - J->qstart[s];
        int i = (int)(tok - J->qstart[s]);
        int last = J->ctx[s] - n + i; /* position of this query token */
        double* o = J->out + r * D;
        for (int d = 0; d < D; ++d) o[d] = 0.0;
        if (last < 0) { J->status = -1; continue; }
        if (last + 1 > cap) {
            cap = last + 1;
            x = (double*)realloc(x, sizeof(double) * (size_t)cap);
        }
        for (int d = 0; d < D; ++d) qd[d] = orc_load(J->q, (size_t)r * D + d, J->q_dtype);
        double mx = -INFINITY;
        for (int t = 0; t <= last; ++t) { /* scores over the causal prefix */
            int64_t blk = J->tables[(int64_t)s * J->max_blocks + t / J->bs];
            if (blk < 0 || blk >= J->num_blocks) { J->status = -1; blk = 0; }
            size_t base = (size_t)(((blk * J->hkv + h) * J->bs + t % J->bs)) * D;
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qd[d] * (J->k_scale * orc_load(J->k_cache, base + d, J->kv_dtype));
            x[t] = J->scale * acc;
            if (x[t] > mx) mx = x[t];
        }
        double sum = 0.0;
        for (int t = 0; t <= last; ++t) {
            x[t] = exp(x[t] - mx);
            sum += x[t];
        }
        for (int t = 0; t <= last; ++t) {
            int64_t blk = J->tables[(int64_t)s * J->max_blocks + t / J->bs];
            if (blk < 0 || blk >= J->num_blocks) blk = 0;
            size_t base = (size_t)(((blk * J->hkv + h) * J->bs + t % J->bs)) * D;
            double w = x[t] / sum;
            for (int d = 0; d < D; ++d) o[d] += w * (J->v_scale * orc_load(J->v_cache, base + d, J->kv_dtype));
        }
    }
    free(x);
    free(qd);
    return NULL;
}

/* out[T][Hq][D] (fp64) of the multi-token queries described above, q in
 * q_dtype, the cache in kv_dtype, a cache element standing for k_scale
 * (v_scale) times its stored value (an E4M3 cache with its per-layer scales,
 * as in oracle_paged_decode_scaled).  Returns 0, -1 for a table entry outside
 * the pool or a chunk longer than its context, -2 for bad head counts. */
int oracle_paged_prefill_scaled(int q_dtype, int kv_dtype, double k_scale, double v_scale, const void* q,
                                const void* k_cache, const void* v_cache, const int32_t* block_tables,
                                int max_blocks, const int32_t* query_start, const int32_t* context_lens,
                                int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int num_blocks, double scale, double* out, int nthreads) {
    if (num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads) return -2;
    if (nthreads <= 0) nthreads = (int)sysconf(_SC_NPROCESSORS_ONLN);
    if (nthreads < 1) nthreads = 1;
    int64_t rows = (int64_t)(num_seqs > 0 ? query_start[num_seqs] : 0) * num_q_heads;
    if (nthreads > rows) nthreads = rows > 0 ? (int)rows : 1;
    orc_pjob* jobs = (orc_pjob*)calloc((size_t)nthreads, sizeof(orc_pjob));
    pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
    for (int i = 0; i < nthreads; ++i) {
        orc_pjob j = {q_dtype, kv_dtype, k_scale, v_scale, q, k_cache, v_cache, block_tables, query_start,
                      context_lens, max_blocks, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                      num_blocks, scale, out, rows * i / nthreads, rows * (i + 1) / nthreads, 0};
        jobs[i] = j;
    }
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, orc_prefill_rows, &jobs[i]);
    orc_prefill_rows(&jobs[0]);
    int status = 0;
    for (int i = 0; i < nthreads; ++i) {
        if (i) pthread_join(th[i], NULL);
        if (jobs[i].status) status = jobs[i].status;
    }
    free(jobs);
    free(th);
    return status;
}

/* The same with q and the cache in one dtype and no cache scaling. */
int oracle_paged_prefill(int dtype, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, int max_blocks, const int32_t* query_start,
                         const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, double scale, double* out,
                         int nthreads) {
    return oracle_paged_prefill_scaled(dtype, dtype, 1.0, 1.0, q, k_cache, v_cache, block_tables, max_blocks,
                                       query_start, context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                                       block_size, num_blocks, scale, out, nthreads);
}

/* Slot of every new token: token i of sequence s sits at position
 * context_lens[s] - n_s + i. */
void oracle_slot_mapping_varlen(const int32_t* block_tables, int max_blocks, const int32_t* query_start,
                                const int32_t* context_lens, int num_seqs, int block_size,
                                int32_t* slot_out) {
    for (int s = 0; s < num_seqs; ++s) {
        int n = query_start[s + 1] - query_start[s];
        for (int i = 0; i < n; ++i)
            slot_out[query_start[s] + i] =
                (int32_t)oracle_slot(block_tables, max_blocks, s, context_lens[s] - n + i, block_size);
    }
}

/* The same with q and the cache in one dtype and no cache scaling. */
int oracle_paged_decode(int dtype, const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                        int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int num_blocks, double scale, double* out, int nthreads) {
    return oracle_paged_decode_scaled(dtype, dtype, 1.0, 1.0, q, k_cache, v_cache, block_tables,
                                      max_blocks, context_lens, num_seqs, num_q_heads, num_kv_heads,
                                      head_dim, block_size, num_blocks, scale, out, nthreads);
}

int oracle_num_cores(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }
