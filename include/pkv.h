/*
 * pkv.h -- C ABI of a paged KV cache and single-query (decode) attention over
 * it, for one GPU (sm_103a).
 *
 * The operations follow "vLLM Architecture and Installation", Example 3
 * (paged KV cache block tables) and "Batching and Scheduling", Example 1
 * (utilization of a single decoding request):
 *   - the cache is a pool of fixed-size blocks; each sequence owns a block
 *     table listing its physical blocks in logical order;
 *   - each step appends every running sequence's newest K/V row to the slot
 *     table[pos / block_size] * block_size + pos % block_size;
 *   - each sequence's single query token then attends over all of its cached
 *     tokens, read through its block table.
 *
 * Conventions for every call:
 *   - Tensor arguments are plain pointers.  "device" pointers must be
 *     addresses in the memory of the selected GPU; "host" pointers are
 *     ordinary CPU memory.  The caller owns every buffer it passes; the
 *     library frees only memory it allocated itself (kv_pool_create with a
 *     NULL buffer).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Device work is enqueued asynchronously on it; device pointers
 *     must stay valid until that work completes.
 *   - Arguments are validated on the host before anything is launched.  A
 *     failed validation returns a status code and launches nothing; no call
 *     throws or aborts.  kv_last_error() describes the last failure of the
 *     calling thread.
 *   - Errors that only the device can see (a block id outside the pool, a
 *     slot outside the pool, a context longer than its table) set a bit in a
 *     per-device status word and the offending item is skipped or clamped;
 *     kv_device_status() reports and clears it.
 *   - Calls are thread-safe as long as two threads do not write the same
 *     buffers at the same time.
 *
 * Pool layout in device memory (one pool serves every layer; a block id
 * addresses the same block in every layer):
 *   layer l, K: [num_blocks][num_kv_heads][block_size][head_dim]
 *   layer l, V: same shape, right after layer l's K
 *   so one (block, kv_head) tile of K is block_size*head_dim contiguous
 *   elements.  Block tables are int32 [num_seqs][max_blocks_per_seq], row
 *   major, entries past the sequence's last block are ignored (-1 by
 *   convention).  context_lens[s] counts every cached token of sequence s,
 *   including the one appended in the current step.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Every declaration below is exported from the shared library, which is
 * otherwise built with hidden symbol visibility. */
#if defined(__GNUC__)
#pragma GCC visibility push(default)
#endif

/* KV_FP8_E4M3: one-byte E4M3 codes (sign, 4-bit exponent with bias 7, 3-bit
 * fraction, no infinities, S.1111.111 = NaN, largest finite 448), a storage
 * type of KV pools only ("vLLM Architecture and Installation", Example 6:
 * an FP8 KV cache takes one byte per value).  A code b of a layer's K (V)
 * stands for k_scale (v_scale) * e4m3(b); the scales are fp32, one per layer
 * for K and one for V, owned by the caller and passed to every call.  The
 * library's quantizer never writes the NaN codes (it saturates at 448); NaN
 * codes written into a pool by other code are not guaranteed to propagate:
 * where the attention kernels convert codes with integer operations (V
 * always, K with an f16 q or 8 query heads per KV head) they read as +-480. */
typedef enum { KV_F32 = 0, KV_F16 = 1, KV_BF16 = 2, KV_FP8_E4M3 = 3 } kv_dtype_t;

typedef enum {
    KV_OK = 0,
    KV_ERR_INVALID_ARG = 1,         /* a pointer, size or shape is not acceptable */
    KV_ERR_UNSUPPORTED = 2,         /* valid, but not a shape/dtype the kernels cover */
    KV_ERR_OUT_OF_MEMORY = 3,       /* a library allocation failed */
    KV_ERR_OUT_OF_BLOCKS = 4,       /* host allocator: not enough free blocks */
    KV_ERR_WORKSPACE_TOO_SMALL = 5, /* see paged_decode_workspace_bytes */
    KV_ERR_CUDA = 6,                /* a CUDA runtime call failed */
    KV_ERR_DEVICE_CHECK = 7,        /* the device flagged a bad block id / slot / length */
    KV_ERR_DEVICE_TIMEOUT = 8,      /* a bounded wait inside a kernel ran out */
    KV_ERR_NOT_FOUND = 9            /* host allocator: unknown sequence id */
} kv_status_t;

/* Bits of the per-device status word (kv_device_status). */
#define KV_FLAG_BAD_BLOCK_ID   0x1u /* a table entry outside [0, num_blocks) was read */
#define KV_FLAG_BAD_SLOT       0x2u /* an append slot >= num_blocks*block_size */
#define KV_FLAG_BAD_CONTEXT    0x4u /* context_lens[s] < 0 or > max_blocks_per_seq*block_size */
#define KV_FLAG_TIMEOUT        0x8u /* a kernel gave up a bounded wait */
#define KV_FLAG_BAD_PLAN       0x10u /* a launch plan the kernel refuses (never set by this library's own planning) */

/* Human-readable name of a status code (static string). */
const char* kv_status_string(kv_status_t status);

/* Description of the last failed call on this thread ("" if none). */
const char* kv_last_error(void);

/* ------------------------------------------------------------------ pool */

typedef struct {
    int num_layers;
    int num_blocks;   /* physical blocks; a block holds block_size tokens */
    int block_size;   /* tokens per block (1..1024) */
    int num_kv_heads;
    int head_dim;     /* head_dim * element size must be a multiple of 16 bytes */
    kv_dtype_t dtype;
    int device;       /* CUDA device ordinal */
} kv_pool_config_t;

typedef struct kv_pool kv_pool_t;

/* Bytes of a pool: 2 (K and V) * num_layers * num_blocks * block_size *
 * num_kv_heads * head_dim * element size ("vLLM Architecture and
 * Installation", Example 6: 16 x 8 x (128 + 128) x 2 = 65,536 bytes per layer
 * per block).  Returns 0 for an invalid configuration. */
size_t kv_pool_bytes(const kv_pool_config_t* cfg);

/* Create a pool.  device_buffer: a device buffer of at least kv_pool_bytes()
 * bytes, 256-byte aligned, owned by the caller and adopted (not copied, not
 * freed); or NULL, in which case the library allocates (and later frees) the
 * memory with cudaMalloc.  The contents are not initialised. */
kv_status_t kv_pool_create(const kv_pool_config_t* cfg, void* device_buffer, size_t buffer_bytes,
                           kv_pool_t** pool_out);

/* Destroy a pool (frees only memory the library allocated).  NULL is a no-op. */
void kv_pool_destroy(kv_pool_t* pool);

/* Device addresses of layer `layer`'s K and V caches. */
kv_status_t kv_pool_layer(const kv_pool_t* pool, int layer, void** k_cache, void** v_cache);

/* Copy of the pool's configuration. */
kv_status_t kv_pool_config(const kv_pool_t* pool, kv_pool_config_t* cfg_out);

/* ---------------------------------------------------------------- append */

/* Slot of every sequence's newest token (position context_lens[s] - 1):
 *   slot_mapping[s] = table[s][p / block_size] * block_size + p % block_size,
 * or -1 where context_lens[s] <= 0 ("vLLM Architecture and Installation",
 * Example 3).  All pointers are device pointers: block_tables
 * int32[num_seqs][max_blocks_per_seq], context_lens int32[num_seqs],
 * slot_mapping int32[num_seqs] (written).  A table entry outside
 * [0, num_blocks) gives slot -1 and sets KV_FLAG_BAD_BLOCK_ID; a length past
 * the table gives -1 and sets KV_FLAG_BAD_CONTEXT. */
kv_status_t kv_slot_mapping(const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* context_lens, int num_seqs, int block_size,
                            int num_blocks, int32_t* slot_mapping, void* stream);

/* Write each token's K and V rows into layer `layer` of the pool at its slot
 * ("vLLM Architecture and Installation", Example 3: the slot mapping tells the
 * attention kernel where new keys and values go).  Bit-exact copy, no dtype
 * conversion (k and v have the pool's dtype).
 *   k, v          device [n_tokens][num_kv_heads][head_dim]
 *   slot_mapping  device int32[n_tokens]; a negative slot writes nothing;
 *                 a slot >= num_blocks*block_size writes nothing and sets
 *                 KV_FLAG_BAD_SLOT
 *   seq_ids       device int32[n_tokens] or NULL; not used for addressing,
 *                 a token whose seq_id is negative is padding and writes
 *                 nothing
 * Two tokens of one call must not share a slot (the result would be either
 * row). n_tokens == 0 is a no-op. */
kv_status_t kv_append(kv_pool_t* pool, int layer, const int32_t* seq_ids, int n_tokens,
                      const void* k, const void* v, const int32_t* slot_mapping, void* stream);

/* ------------------------------------------------------- decode attention */

typedef enum {
    KV_KERNEL_AUTO = 0, /* tensor-core kernel for f16/bf16, FFMA for f32 */
    KV_KERNEL_FFMA = 1, /* CUDA-core fp32 FMA kernel, any dtype */
    KV_KERNEL_MMA = 2   /* warp-level tensor-core kernel, f16/bf16 only */
} kv_kernel_t;

typedef struct {
    int num_ctas;        /* persistent grid size; 0 = SM count x ctas_per_sm */
    int ctas_per_sm;     /* 0 = 1 */
    int consumer_warps;  /* compute warps per CTA, 1..15; 0 = about 8 */
    kv_kernel_t kernel;
    int heads_per_stage; /* KV heads whose K/V rows of one block form one pipeline
                            stage; must divide num_kv_heads; 0 = the largest
                            divisor whose K slab of a block fits 32 KiB */
    int separate_reduce; /* 1: merge the partials of split sequences in a second
                            kernel; 0: the last CTA to finish a sequence merges
                            them inside the attention kernel */
    int no_pdl;          /* 1: plain launches; 0: programmatic dependent launch
                            (a kernel's prologue overlaps the previous kernel) */
    int early_reads;     /* 1: the caller promises that the launch just before
                            this call on the stream writes neither block_tables,
                            context_lens nor k_cache/v_cache; the kernel then
                            reads those (and starts streaming the cache) while
                            that launch finishes.  q, k_new/v_new, the
                            workspace and the outputs are still touched only
                            after it.  Ignored with no_pdl. */
    int test_stall;      /* testing only, 0 in normal use: when non-zero, the
                            producer of CTA 0 stops after one stage so that a
                            consumer's bounded wait (about 2 s) runs out; the
                            call then reports KV_ERR_DEVICE_TIMEOUT through
                            kv_device_status and the output is undefined */
} kv_decode_options_t;

/* Workspace bytes paged_decode_attention needs for these sizes on `device`
 * with these options (NULL = defaults). */
kv_status_t paged_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads,
                                         int head_dim, int device,
                                         const kv_decode_options_t* opts, size_t* bytes_out);

/* Zero the part of a workspace that must start at zero (the per-(sequence,
 * KV head) merge counters at its start), asynchronously on `stream`.  Call it
 * once after allocating a workspace (or zero the whole buffer); every
 * completed call of paged_decode_attention leaves the counters zero again.
 * After a call that reported KV_ERR_DEVICE_TIMEOUT, call it again. */
kv_status_t paged_decode_workspace_init(void* workspace, size_t workspace_bytes, int num_seqs,
                                        int num_kv_heads, void* stream);

/* Single-query attention over the paged cache, for every sequence s and query
 * head g (KV head h = g / (num_q_heads / num_kv_heads)):
 *   out[s][g] = sum_t softmax_t(scale * q[s][g] . K_s[t]) * V_s[t],
 *   t = 0 .. context_lens[s]-1, K_s[t] = k_cache[table[s][t / bs]][h][t % bs]
 * ("vLLM Architecture and Installation", Example 3; "Batching and
 * Scheduling", Example 1).  A sequence with context 0 gets a zero row.
 *   q            device [num_seqs][num_q_heads][head_dim], dtype
 *   k_cache,
 *   v_cache      device, one layer of a pool: [num_blocks][num_kv_heads]
 *                [block_size][head_dim], dtype; 16-byte aligned
 *   block_tables device int32 [num_seqs][max_blocks_per_seq]
 *   context_lens device int32 [num_seqs]
 *   out          device [num_seqs][num_q_heads][head_dim], out_dtype
 *                (KV_F32, or the same dtype as q)
 *   workspace    device scratch of workspace_bytes >= the size given by
 *                paged_decode_workspace_bytes for the same sizes and options,
 *                256-byte aligned, initialised once with
 *                paged_decode_workspace_init (or zero-filled); not to be
 *                shared by two calls in flight at once
 * Supported: head_dim 64 or 128, block_size 8..256 a multiple of 8,
 * num_q_heads / num_kv_heads in {1, 2, 4, 8}; dtype f32, f16 or bf16.
 * The work of all sequences -- (sequence, group of KV heads, block) items --
 * is split evenly over a persistent grid; each CTA writes an fp32 partial
 * (unnormalised output, running max, running sum) for every sequence/KV head
 * it only partly covers, and the partials are merged (log-sum-exp) by the
 * last CTA to finish that sequence or by a second kernel
 * (separate_reduce).  Accumulation is fp32 throughout. */
kv_status_t paged_decode_attention(const void* q, const void* k_cache, const void* v_cache,
                                   int num_blocks, const int32_t* block_tables,
                                   int max_blocks_per_seq, const int32_t* context_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, kv_dtype_t dtype, float scale, void* out,
                                   kv_dtype_t out_dtype, void* workspace, size_t workspace_bytes,
                                   const kv_decode_options_t* opts, void* stream);

/* One layer of one decode step in a single kernel: the append of every
 * sequence's newest token followed by the attention that reads it.
 * Equivalent to kv_slot_mapping + kv_append + paged_decode_attention with the
 * same arguments ("vLLM Architecture and Installation", Example 3: write the
 * new rows through the slot mapping, then read the history through the block
 * table), without the two extra launches.  For each sequence s with
 * context_lens[s] >= 1 (and seq_ids == NULL or seq_ids[s] >= 0) the rows
 * k_new[s], v_new[s] ([num_seqs][num_kv_heads][head_dim], device, 16-byte
 * aligned) are written to position context_lens[s] - 1, i.e. slot
 * table[s][p / bs] * bs + p % bs, and that position takes part in this
 * step's attention.  The block holding that slot must not be shared with
 * another sequence of the batch (copy-on-write is the caller's job).
 * slot_mapping: device int32[num_seqs] that receives the slots (-1 for an
 * empty sequence), or NULL.  The other arguments are those of
 * paged_decode_attention; k_cache and v_cache are written. */
kv_status_t paged_decode_append_attention(const void* q, const void* k_new, const void* v_new,
                                          const int32_t* seq_ids, void* k_cache, void* v_cache,
                                          int num_blocks, const int32_t* block_tables,
                                          int max_blocks_per_seq, const int32_t* context_lens,
                                          int num_seqs, int num_q_heads, int num_kv_heads,
                                          int head_dim, int block_size, kv_dtype_t dtype,
                                          float scale, void* out, kv_dtype_t out_dtype,
                                          int32_t* slot_mapping, void* workspace,
                                          size_t workspace_bytes, const kv_decode_options_t* opts,
                                          void* stream);

/* paged_decode_attention without a caller-provided workspace, for callers
 * that cannot allocate device memory (for instance an engine that gave all
 * free device memory to its KV-block pool at start-up, or code that is handed
 * only the tensors it works on).  The pages have no counterpart: this is an
 * interface convenience of this library.
 *   Scratch: a fixed 8 MiB array in the library's own device memory (held by
 *   every GPU that loads the library until the process exits); sizes that
 *   need more (paged_decode_workspace_bytes) are rejected with
 *   KV_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 *   Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 *   The first call on a device takes the array's device address (and may
 *   load the library's device code there): make it before any stream capture.
 *   The address is kept for the life of the process, so the library must not
 *   be called on a device after cudaDeviceReset there.
 *   Each accepted call clears the array's merge counters on `stream` right
 *   before its kernel; a refused call (any error status) queues nothing.
 *   All calls on a device share the array: calls that overlap on the GPU race.
 * The other arguments and the result are those of paged_decode_attention. */
kv_status_t paged_decode_attention_static(const void* q, const void* k_cache, const void* v_cache,
                                          int num_blocks, const int32_t* block_tables,
                                          int max_blocks_per_seq, const int32_t* context_lens,
                                          int num_seqs, int num_q_heads, int num_kv_heads,
                                          int head_dim, int block_size, kv_dtype_t dtype,
                                          float scale, void* out, kv_dtype_t out_dtype,
                                          const kv_decode_options_t* opts, void* stream);

/* Synchronise `stream`, then read and clear the status word of `device`.
 * flags_out (may be NULL) receives the KV_FLAG_* bits.  Returns KV_OK when no
 * bit was set, KV_ERR_DEVICE_TIMEOUT if the timeout bit was set, else
 * KV_ERR_DEVICE_CHECK. */
kv_status_t kv_device_status(int device, void* stream, uint32_t* flags_out);

/* -------------------------------------------------- multi-token queries */

/* A step in which sequence s brings n_s = query_start[s+1] - query_start[s]
 * new tokens: one for a decoding request, a chunk of the prompt for a
 * prefilling one ("Batching and Scheduling", Example 5 and "vLLM Architecture
 * and Installation", Example 5: a token budget per step and chunked prefill).
 * context_lens[s] counts every cached token of s including the n_s new ones,
 * which sit at positions context_lens[s] - n_s .. context_lens[s] - 1.
 * query_start: device int32[num_seqs + 1], non-decreasing, query_start[0] = 0,
 * query_start[num_seqs] = num_tokens.
 *
 * kv_slot_mapping_varlen: slot of every new token (slot_mapping, device
 * int32[num_tokens]): token i of s goes to table[s][p / bs] * bs + p % bs,
 * p = context_lens[s] - n_s + i.  Feed it to kv_append with the new rows.
 * A position outside the table gives -1 and sets KV_FLAG_BAD_CONTEXT, a bad
 * table entry -1 and KV_FLAG_BAD_BLOCK_ID. */
kv_status_t kv_slot_mapping_varlen(const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* query_start, const int32_t* context_lens,
                                   int num_seqs, int num_tokens, int block_size, int num_blocks,
                                   int32_t* slot_mapping, void* stream);

/* Bytes of the workspace paged_prefill_attention needs (device, 16-byte
 * aligned, no initialisation). */
size_t paged_prefill_workspace_bytes(int num_seqs);

/* Causal attention of the new tokens over the paged cache (after their
 * append): row t = query_start[s] + i of q and out ([num_tokens][Hq][D])
 * attends to the cached tokens of s at positions 0 .. context_lens[s] - n_s + i,
 * softmax(scale q.K^T).V with fp32 accumulation; query head g reads KV head
 * g / (Hq/Hkv).  dtype f16 or bf16 (q and the cache; block_size a multiple
 * of 16 up to 256) or f32 (block_size 1 .. 256; CUDA-core kernel, one warp
 * per token and query head, not tuned for speed), head_dim 64 or 128, Hq/Hkv
 * in {1, 2, 4, 8}; out_dtype KV_F32 or dtype.  A sequence with
 * n_s > context_lens[s] (or a length past its table) is skipped (its rows
 * are not written) and sets KV_FLAG_BAD_CONTEXT.  One CTA per (16 new
 * tokens, KV head) for f16/bf16; a decoding sequence (n_s = 1) is served
 * too, but paged_decode_attention is the faster call for a batch of those.
 * An E4M3 cache goes to paged_prefill_attention_fp8 (KV_ERR_INVALID_ARG
 * here). */
kv_status_t paged_prefill_attention(const void* q, const void* k_cache, const void* v_cache,
                                    int num_blocks, const int32_t* block_tables,
                                    int max_blocks_per_seq, const int32_t* query_start,
                                    const int32_t* context_lens, int num_seqs, int num_tokens,
                                    int num_q_heads, int num_kv_heads, int head_dim,
                                    int block_size, kv_dtype_t dtype, float scale, void* out,
                                    kv_dtype_t out_dtype, void* workspace, size_t workspace_bytes,
                                    void* stream);

/* ------------------------------------------------------- FP8 (E4M3) cache */

/* paged_prefill_attention over a KV_FP8_E4M3 cache ("vLLM Architecture and
 * Installation", Example 6, with the chunked prefill of Example 5): the keys
 * and values are k_scale (v_scale) times their codes' values.  q_dtype
 * KV_F16 or KV_BF16, head_dim 128, block_size a multiple of 16 up to 256;
 * out_dtype KV_F32 or q_dtype; the rest as paged_prefill_attention.  Each
 * block's codes are converted exactly to q's type in shared memory and the
 * scales folded into the score multiplier and the output. */
kv_status_t paged_prefill_attention_fp8(const void* q, kv_dtype_t q_dtype, const void* k_cache,
                                        const void* v_cache, float k_scale, float v_scale,
                                        int num_blocks, const int32_t* block_tables,
                                        int max_blocks_per_seq, const int32_t* query_start,
                                        const int32_t* context_lens, int num_seqs, int num_tokens,
                                        int num_q_heads, int num_kv_heads, int head_dim,
                                        int block_size, float scale, void* out, kv_dtype_t out_dtype,
                                        void* workspace, size_t workspace_bytes, void* stream);

/* kv_append into a KV_FP8_E4M3 pool: k and v are [n_tokens][Hkv][D] rows in
 * src_dtype (KV_F32, KV_F16 or KV_BF16); each value x is stored as the E4M3
 * code nearest to the fp32 quotient x / k_scale (x / v_scale), ties to the
 * even code, magnitudes from 448 up saturating to +-448.  Otherwise as
 * kv_append.  k_scale and v_scale must be finite and > 0. */
kv_status_t kv_append_fp8(kv_pool_t* pool, int layer, const int32_t* seq_ids, int n_tokens,
                          const void* k, const void* v, kv_dtype_t src_dtype,
                          const int32_t* slot_mapping, float k_scale, float v_scale, void* stream);

/* paged_decode_attention over an E4M3 cache ("vLLM Architecture and
 * Installation", Example 6): the same attention with K = k_scale * e4m3(k
 * code) and V = v_scale * e4m3(v code).  q is [num_seqs][Hq][D] in q_dtype
 * (KV_F16 or KV_BF16; it enters the tensor cores as f16, exact for |q| below
 * 65504 and above 2^-14); out_dtype is KV_F32 or q_dtype.  head_dim 128,
 * block_size a multiple of 16 up to 256.  Workspace and options as
 * paged_decode_attention (kernel KV_KERNEL_AUTO or KV_KERNEL_MMA). */
kv_status_t paged_decode_attention_fp8(const void* q, kv_dtype_t q_dtype, const void* k_cache,
                                       const void* v_cache, float k_scale, float v_scale,
                                       int num_blocks, const int32_t* block_tables,
                                       int max_blocks_per_seq, const int32_t* context_lens,
                                       int num_seqs, int num_q_heads, int num_kv_heads,
                                       int head_dim, int block_size, float scale, void* out,
                                       kv_dtype_t out_dtype, void* workspace,
                                       size_t workspace_bytes, const kv_decode_options_t* opts,
                                       void* stream);

/* paged_decode_append_attention over an E4M3 cache: k_new and v_new are in
 * q_dtype and are quantized as kv_append_fp8 does before this step reads
 * them; otherwise as paged_decode_attention_fp8. */
kv_status_t paged_decode_append_attention_fp8(const void* q, const void* k_new, const void* v_new,
                                              const int32_t* seq_ids, kv_dtype_t q_dtype,
                                              void* k_cache, void* v_cache, float k_scale,
                                              float v_scale, int num_blocks,
                                              const int32_t* block_tables, int max_blocks_per_seq,
                                              const int32_t* context_lens, int num_seqs,
                                              int num_q_heads, int num_kv_heads, int head_dim,
                                              int block_size, float scale, void* out,
                                              kv_dtype_t out_dtype, int32_t* slot_mapping,
                                              void* workspace, size_t workspace_bytes,
                                              const kv_decode_options_t* opts, void* stream);

/* ------------------------------------------------------ swap to host memory */

/* Preemption by swap ("Batching and Scheduling", Example 8): a request's KV
 * blocks are copied to CPU memory and later copied back, instead of being
 * dropped and computed again.
 *
 * A swapped block is all of one physical block across the pool: every layer's
 * K and V rows.  Host record layout, for block i of the list:
 *   [i][2 * num_layers][num_kv_heads][block_size][head_dim] elements,
 * unit 2*l holding layer l's K rows and unit 2*l + 1 its V rows, each in the
 * pool's own [Hkv][bs][D] order.  kv_swap_bytes(pool, n) is the size of n
 * records: n * 2 * num_layers * num_kv_heads * block_size * head_dim * elem.
 *
 * kv_swap_out copies pool blocks block_ids[0..n) to records 0..n of host_dst;
 * kv_swap_in copies records 0..n of host_src into pool blocks block_ids[0..n)
 * (which need not be the blocks they came from).  One kernel each, enqueued
 * on `stream`; the GPU reads and writes the host buffer directly, so it must
 * be memory the device addresses: page-locked host memory (cudaHostAlloc,
 * cudaHostRegister), managed memory or device memory, 16-byte aligned, at
 * least kv_swap_bytes(pool, n) bytes.  block_ids: int32[n], device-addressable
 * likewise.  Pageable host memory is refused with KV_ERR_INVALID_ARG.
 * Ownership stays with the caller; the host buffer must stay alive and
 * untouched by the CPU until the stream reaches the copy's end.
 * Block ids outside [0, num_blocks) are skipped and set
 * KV_FLAG_BAD_BLOCK_ID in the device status word.  Swap-in with a block id
 * listed twice leaves that block holding either record. */
size_t kv_swap_bytes(const kv_pool_t* pool, int num_blocks);
kv_status_t kv_swap_out(const kv_pool_t* pool, const int32_t* block_ids, int n, void* host_dst,
                        size_t host_bytes, void* stream);
kv_status_t kv_swap_in(kv_pool_t* pool, const int32_t* block_ids, int n, const void* host_src,
                       size_t host_bytes, void* stream);

/* --------------------------------------------------- host block allocator */

/* A host-side allocator of physical blocks, the bookkeeping that produces the
 * block tables ("vLLM Architecture and Installation", Example 3): a FIFO free
 * queue (initially blocks in increasing order, block 0 held back as the null
 * block when reserve_null_block is set); extending a sequence takes whole
 * blocks from the front of the queue, only when a token crosses a block
 * boundary; releasing a sequence returns its blocks, in table order, to the
 * back of the queue.  An extension that needs more blocks than are free fails
 * with KV_ERR_OUT_OF_BLOCKS and changes nothing. */
typedef struct kv_block_allocator kv_block_allocator_t;

kv_status_t kv_allocator_create(int num_blocks, int block_size, int reserve_null_block,
                                kv_block_allocator_t** out);
void kv_allocator_destroy(kv_block_allocator_t* a);
kv_status_t kv_allocator_extend(kv_block_allocator_t* a, int64_t seq_id, int new_tokens);
kv_status_t kv_allocator_release(kv_block_allocator_t* a, int64_t seq_id);
/* table_out (host, capacity entries) receives the sequence's blocks;
 * num_blocks_out / num_tokens_out may be NULL. */
kv_status_t kv_allocator_table(const kv_block_allocator_t* a, int64_t seq_id, int32_t* table_out,
                               int capacity, int* num_blocks_out, int* num_tokens_out);
kv_status_t kv_allocator_slot(const kv_block_allocator_t* a, int64_t seq_id, int position,
                              int32_t* slot_out);
/* The free queue, front first. */
kv_status_t kv_allocator_free_queue(const kv_block_allocator_t* a, int32_t* out, int capacity,
                                    int* count_out);

/* Sequence bookkeeping on the pool itself: the pool keeps one allocator of
 * its blocks (the semantics above, no null block), created on first use.
 * kv_seq_extend grows sequence seq_id by new_tokens tokens:
 *   *ctx_len_inout  in: the sequence's current length (0 for a new one; it must
 *                   match the pool's record), out: the new length;
 *   table_row       host int32 [max_blocks]: the sequence's block table,
 *                   padded with -1;
 *   slot_out        host int32 [new_tokens] (may be NULL when new_tokens is 0):
 *                   slot of each new token, block * block_size + offset
 *                   ("vLLM Architecture and Installation", Example 3).
 * A table that would not fit in max_blocks entries (KV_ERR_INVALID_ARG) or an
 * extension that needs more blocks than are free (KV_ERR_OUT_OF_BLOCKS)
 * changes nothing.  kv_seq_free returns the sequence's blocks to the back of
 * the free queue (KV_ERR_NOT_FOUND for an unknown sequence).  Host-side and
 * single-threaded per pool. */
kv_status_t kv_seq_extend(kv_pool_t* pool, int seq_id, int new_tokens, int32_t* table_row, int max_blocks,
                          int* ctx_len_inout, int32_t* slot_out);
kv_status_t kv_seq_free(kv_pool_t* pool, int seq_id);

/* ------------------------------------------ block pool with prefix caching */

/* The block pool of "Reading Inference Engine Codebases", Examples 12 and 13
 * (vLLM's KV cache manager and block pool), host side, single-threaded.
 *
 * Every full block of a request is indexed by a chained hash of its parent's
 * hash and its own token ids, so it names the whole prefix up to its end.
 * kv_prefix_pool_allocate(tokens) takes:
 *   1. the longest run of cached full blocks matching the request's prefix,
 *      at most (num_tokens - 1) / block_size blocks (the last token is always
 *      computed again); each hit gains a reference and leaves the free queue;
 *   2. ceil(num_tokens / block_size) minus the hits new blocks from the front
 *      of the free queue; a popped block that still has a hash loses it
 *      (eviction, reported in evicted_out); each new full block is cached
 *      under its prefix hash, with no de-duplication of equal blocks.
 * kv_prefix_pool_free(blocks) drops one reference per block, walking the list
 * tail first; a block reaching zero goes to the front of the free queue when
 * it has no hash, to the back when it has one (least recently used first).
 * The free queue starts as all blocks in increasing id order.
 *
 * tokens: host int32[num_tokens], any values.  blocks_out: host, capacity
 * entries, receives the request's blocks in table order.  cached_tokens_out
 * (may be NULL): hit blocks x block_size.  evicted_out (may be NULL) receives
 * up to evicted_capacity evicted block ids in eviction order;
 * num_evicted_out (may be NULL) the count.  When fewer blocks are free than
 * the request needs, KV_ERR_OUT_OF_BLOCKS and nothing changes.  Freeing a
 * block whose count is already zero, or an id out of range, is
 * KV_ERR_INVALID_ARG and nothing changes. */
typedef struct kv_prefix_pool kv_prefix_pool_t;

kv_status_t kv_prefix_pool_create(int num_blocks, int block_size, kv_prefix_pool_t** out);
void kv_prefix_pool_destroy(kv_prefix_pool_t* p);
kv_status_t kv_prefix_pool_allocate(kv_prefix_pool_t* p, const int32_t* tokens, int num_tokens,
                                    int32_t* blocks_out, int capacity, int* num_blocks_out,
                                    int* cached_tokens_out, int32_t* evicted_out,
                                    int evicted_capacity, int* num_evicted_out);
kv_status_t kv_prefix_pool_free(kv_prefix_pool_t* p, const int32_t* blocks, int n);
/* The free queue, front (next to be reused) first.  With out == NULL only
 * count_out is written. */
kv_status_t kv_prefix_pool_free_queue(const kv_prefix_pool_t* p, int32_t* out, int capacity,
                                      int* count_out);
/* Number of distinct cached prefix hashes and of blocks holding one. */
kv_status_t kv_prefix_pool_cache_size(const kv_prefix_pool_t* p, int* hashes_out,
                                      int* blocks_out);

#if defined(__GNUC__)
#pragma GCC visibility pop
#endif

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
