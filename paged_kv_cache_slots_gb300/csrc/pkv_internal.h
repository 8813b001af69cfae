// Internal interface between the C-ABI host layer (pkv_api.cpp) and the CUDA
// launchers (*.cu).  Plain structs of pointers and sizes; no torch types.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "pkv.h"

namespace pkv {

// Element types as stored in the pool, q and out (same codes as kv_dtype_t).
enum DType : int { kF32 = 0, kF16 = 1, kBF16 = 2, kFP8 = 3 };

__host__ __device__ inline int dtype_bytes(int dt) { return dt == kF32 ? 4 : dt == kFP8 ? 1 : 2; }

struct AppendArgs {
    const int32_t* seq_ids;       // [n_tokens] or nullptr
    const void* k;                // [n_tokens][Hkv][D]
    const void* v;
    const int32_t* slot_mapping;  // [n_tokens]
    void* k_cache;                // [NB][Hkv][bs][D]
    void* v_cache;
    uint32_t* status;             // device status word
    int n_tokens, num_kv_heads, head_dim, block_size, num_blocks, elem_bytes;
    int pdl;
    // Quantizing append into an E4M3 pool: k/v rows are in src_dtype and
    // are stored as codes of x / k_scale (x / v_scale).
    int quant;
    int src_dtype;
    float k_scale, v_scale;
};

// Block swap between the pool and a device-addressable host buffer.
struct SwapArgs {
    char* pool;               // pool base: layer l's K at 2l * layer_bytes, V at (2l + 1) * layer_bytes
    char* host;               // [n][2 * num_layers][unit_bytes]
    const int32_t* block_ids;  // [n] physical blocks
    uint32_t* status;
    int64_t layer_bytes;      // one of K or V of one layer
    int64_t unit_bytes;       // one block of one of K or V of one layer (multiple of 16)
    int n, num_layers, num_blocks;
    int to_host;              // 1: pool -> host (swap out), 0: host -> pool (swap in)
    int pdl;
};

struct SlotArgs {
    const int32_t* block_tables;
    const int32_t* context_lens;
    int32_t* slot_mapping;
    uint32_t* status;
    int max_blocks, num_seqs, block_size, num_blocks;
    int pdl;
};

// Everything the split-context decode kernels need.
//
// Work items are (sequence, head chunk, logical block) triples in that order;
// a head chunk is `heads_per_stage` consecutive KV heads, whose K (and V)
// rows of one block are contiguous in the pool, so one item is one pipeline
// stage of two contiguous copies.  Every pair (sequence, head chunk) with
// blocks starts with `phantom` items that carry no data (a ring stage that
// the producer completes without a copy and the consumers skip): a CTA whose
// range crosses into a pair takes that many fewer blocks, which pays for the
// switch between pairs.  W = chunks * sum_s (ceil(ctx_s / bs) + phantom,
// over the sequences with tokens); CTA c of num_ctas owns items
// [c*W/P, (c+1)*W/P).
struct DecodeArgs {
    const void* q;
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    void* out;
    float* part_o;      // [slots][Hc][G][D]  unnormalised partial outputs
    float* part_ml;     // [slots][Hc][G][2]  running max (log2 units) and sum
    int32_t* cum;       // [num_seqs + 1]     exclusive prefix of items per sequence
    int32_t* counters;  // [num_seqs * Hkv]   partials merged so far (zero between calls)
    uint32_t* status;
    // Fused append (paged_decode_append_attention): the new token's rows,
    // written at position context_lens[s] - 1 and used by this very step.
    const void* k_new;           // [num_seqs][Hkv][D] or nullptr (no append)
    const void* v_new;
    const int32_t* append_ids;   // [num_seqs] or nullptr; a negative entry: no append for s
    int32_t* slot_out;           // [num_seqs] or nullptr: slot of the newest token
    int num_blocks, max_blocks, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size;
    int dtype, out_dtype;  // q (and k_new, v_new) and output types
    int kv_dtype;          // cache type: dtype, or kFP8 (E4M3 codes)
    float scale_log2;      // scale * log2(e) (* k_scale for E4M3): scores in base-2 units
    float k_scale, v_scale;  // E4M3 cache: a code stands for scale * value (1 otherwise)
    int num_ctas;         // persistent grid size P
    int heads_per_stage;  // Hc: KV heads per pipeline stage (divides Hkv)
    int warps_per_head;   // R: consumer warps sharing one head's items
    int consumer_warps;   // Hc * R
    int stages;
    int smem_bytes;
    int fused_reduce;     // 1: the last CTA of a split pair merges it (no reduce kernel)
    int pdl;              // 1: launch with programmatic dependent launch
    int early_reads;      // 1: tables, lengths and cache may be read before the previous launch ends
    int test_stall;       // testing only: see kv_decode_options_t
    int device;           // CUDA ordinal the launch targets
    int phantom;          // items without data at the start of every (sequence, head chunk) pair
};

// Multi-token (chunked-prefill) attention and its plan.
struct PrefillArgs {
    const void* q;               // [T][Hq][D]
    const void* k_cache;
    const void* v_cache;
    const int32_t* block_tables;
    const int32_t* query_start;  // [B + 1]
    const int32_t* context_lens; // [B]
    void* out;                   // [T][Hq][D]
    int32_t* tile_cum;           // [B + 1] workspace: prefix of 16-token tiles per sequence
    uint32_t* status;
    int num_blocks, max_blocks, num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size;
    int dtype, out_dtype;
    int kv_dtype;      // the cache: dtype, or kFP8 (E4M3 codes)
    float scale_log2;  // scale * log2(e) (* k_scale for E4M3)
    float v_scale;     // E4M3: a V code stands for v_scale * value (1 otherwise)
    int stages, smem_bytes, grid_tiles;
    int tile_tokens;   // new tokens per CTA (16, or 128 / G on the tcgen05 path)
    int tensor_cores;  // 1: the tcgen05 kernel (head_dim 128)
    int pdl;
    int device;
};

// Shared-memory plan of the partial kernel.
struct DecodePlan {
    int stages;
    int smem_bytes;
    int stage_half_bytes;  // K (or V) bytes of one stage: Hc * bs * D * elem
};

bool decode_plan(int kernel, int dtype, int head_dim, int block_size, int group, int num_seqs,
                 int heads_per_stage, int warps_per_head, int smem_budget, DecodePlan* plan);

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream);
cudaError_t launch_slot_mapping(const SlotArgs& a, cudaStream_t stream);
cudaError_t launch_swap(const SwapArgs& a, int num_sms, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                           cudaStream_t stream);
cudaError_t launch_slot_mapping_varlen(const PrefillArgs& a, int32_t* slots, cudaStream_t stream);
cudaError_t launch_prefill_tc(const PrefillArgs& a, const CUtensorMap& tmap_k, const CUtensorMap& tmap_v,
                              cudaStream_t stream);
int prefill_tc_smem_bytes();
cudaError_t launch_decode_ffma(const DecodeArgs& a, cudaStream_t stream);
cudaError_t launch_decode_mma(const DecodeArgs& a, const CUtensorMap& tmap_k,
                              const CUtensorMap& tmap_v, cudaStream_t stream);
cudaError_t launch_decode_fp8(const DecodeArgs& a, const CUtensorMap& tmap_k,
                              const CUtensorMap& tmap_v, cudaStream_t stream);
cudaError_t launch_decode_reduce(const DecodeArgs& a, cudaStream_t stream);

// Largest dynamic shared memory a CTA may request on `device`.
int max_dynamic_smem(int device);

// Device address of the current device's status word.
cudaError_t status_word_address(uint32_t** ptr);

// paged_decode_attention that zeroes the workspace's merge counters on
// `stream` once every argument has been checked and the launch is planned,
// right before the launch; a call that is rejected touches nothing.
kv_status_t decode_attention_clearing_counters(const void* q, const void* k_cache, const void* v_cache,
                                               int num_blocks, const int32_t* block_tables, int max_blocks,
                                               const int32_t* context_lens, int num_seqs, int num_q_heads,
                                               int num_kv_heads, int head_dim, int block_size, int dtype,
                                               float scale, void* out, int out_dtype, void* workspace,
                                               size_t workspace_bytes, const void* opts, void* stream);

// Records a printf-style message for kv_last_error() on this thread and
// returns st.
kv_status_t report_error(kv_status_t st, const char* fmt, ...);

}  // namespace pkv
