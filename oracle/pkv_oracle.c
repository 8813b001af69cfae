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
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

static size_t orc_elem_bytes(int dtype) { return dtype == ORC_F32 ? 4u : 2u; }

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

typedef struct {
    int dtype;
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
                K[(size_t)t * D + d] = orc_load(J->k_cache, base + d, J->dtype);
                V[(size_t)t * D + d] = orc_load(J->v_cache, base + d, J->dtype);
            }
        }
        for (int d = 0; d < D; ++d) qd[d] = orc_load(J->q, (size_t)r * D + d, J->dtype);
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
 * q is [num_seqs][Hq][D] in `dtype`.  nthreads <= 0 uses every online core.
 * Returns 0, or -1 if a table entry lies outside [0, num_blocks). */
int oracle_paged_decode(int dtype, const void* q, const void* k_cache, const void* v_cache,
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
        orc_job j = {dtype, q, k_cache, v_cache, block_tables, context_lens, max_blocks,
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

int oracle_num_cores(void) { return (int)sysconf(_SC_NPROCESSORS_ONLN); }
