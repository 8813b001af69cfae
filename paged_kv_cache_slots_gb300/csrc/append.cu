// KV append ("reshape into blocks") and newest-token slot mapping.
//
// Follows "vLLM Architecture and Installation", Example 3 (paged KV cache
// block tables): the slot of logical position p of a sequence is
// table[p / block_size] * block_size + p % block_size, and each scheduled
// token's new K and V rows are written to its slot.  Into an E4M3 pool (the
// FP8 KV cache of Example 6 on the same page) each value is quantized on the
// way: the code nearest to x / scale.
#include "device_utils.cuh"

namespace pkv {

// One warp per (token, kv head).  A row of head_dim elements is moved as
// 16-byte vectors: lanes [0, n) copy the K row, lanes [n, 2n) the V row
// (n = row bytes / 16; head_dim * elem is a multiple of 16 by validation).
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendArgs a) {
    pdl_allow_next();
    pdl_wait();
    const int warp = static_cast<int>((blockIdx.x * blockDim.x + threadIdx.x) >> 5);
    const int lane = threadIdx.x & 31;
    if (warp >= a.n_tokens * a.num_kv_heads) return;
    const int i = warp / a.num_kv_heads;
    const int h = warp - i * a.num_kv_heads;
    const int64_t slot = a.slot_mapping[i];
    if (slot < 0) return;
    if (a.seq_ids != nullptr && a.seq_ids[i] < 0) return;
    if (slot >= static_cast<int64_t>(a.num_blocks) * a.block_size) {
        if (lane == 0 && h == 0) raise_flag(a.status, kFlagBadSlot);
        return;
    }
    const int64_t blk = slot / a.block_size;
    const int64_t off = slot - blk * a.block_size;
    if (a.quant) {
        // E4M3 pool: lane e quantizes 16 elements of the K row (e < n) or of
        // the V row (n <= e < 2n), n = head_dim / 16 output chunks.
        const int n = a.head_dim >> 4;
        const int64_t srow = static_cast<int64_t>(a.head_dim) * dtype_bytes(a.src_dtype);
        const int64_t src = (static_cast<int64_t>(i) * a.num_kv_heads + h) * srow;
        const int64_t dst = ((blk * a.num_kv_heads + h) * a.block_size + off) * a.head_dim;
        for (int e = lane; e < 2 * n; e += 32) {
            const bool isv = e >= n;
            const int q = isv ? e - n : e;
            const uint4 val = quantize_chunk16(static_cast<const char*>(isv ? a.v : a.k) + src, q,
                                               a.src_dtype, isv ? a.v_scale : a.k_scale);
            *reinterpret_cast<uint4*>(static_cast<char*>(isv ? a.v_cache : a.k_cache) + dst + 16 * q) = val;
        }
        return;
    }
    const int64_t row_bytes = static_cast<int64_t>(a.head_dim) * a.elem_bytes;
    const int nvec = static_cast<int>(row_bytes >> 4);
    const int64_t src = (static_cast<int64_t>(i) * a.num_kv_heads + h) * row_bytes;
    const int64_t dst = ((blk * a.num_kv_heads + h) * a.block_size + off) * row_bytes;
    const uint4* ks = reinterpret_cast<const uint4*>(static_cast<const char*>(a.k) + src);
    const uint4* vs = reinterpret_cast<const uint4*>(static_cast<const char*>(a.v) + src);
    uint4* kd = reinterpret_cast<uint4*>(static_cast<char*>(a.k_cache) + dst);
    uint4* vd = reinterpret_cast<uint4*>(static_cast<char*>(a.v_cache) + dst);
    for (int e = lane; e < 2 * nvec; e += 32) {
        if (e < nvec)
            kd[e] = __ldg(ks + e);
        else
            vd[e - nvec] = __ldg(vs + (e - nvec));
    }
}

__global__ void __launch_bounds__(256) kv_slot_mapping_kernel(const SlotArgs a) {
    pdl_allow_next();
    pdl_wait();
    const int s = static_cast<int>(blockIdx.x * blockDim.x + threadIdx.x);
    if (s >= a.num_seqs) return;
    const int ctx = a.context_lens[s];
    int32_t slot = -1;
    if (ctx > 0) {
        const int pos = ctx - 1;
        const int j = pos / a.block_size;
        if (j >= a.max_blocks) {
            raise_flag(a.status, kFlagBadContext);
        } else {
            const int blk = a.block_tables[static_cast<int64_t>(s) * a.max_blocks + j];
            if (blk < 0 || blk >= a.num_blocks)
                raise_flag(a.status, kFlagBadBlock);
            else
                slot = blk * a.block_size + (pos - j * a.block_size);
        }
    } else if (ctx < 0) {
        raise_flag(a.status, kFlagBadContext);
    }
    a.slot_mapping[s] = slot;
}

cudaError_t launch_append(const AppendArgs& a, cudaStream_t stream) {
    const int64_t warps = static_cast<int64_t>(a.n_tokens) * a.num_kv_heads;
    if (warps == 0) return cudaSuccess;
    const int threads = 256;
    const int64_t blocks = (warps * 32 + threads - 1) / threads;
    return launch_kernel(kv_append_kernel, dim3(static_cast<unsigned>(blocks)), dim3(threads), 0,
                         stream, a.pdl != 0, a);
}

cudaError_t launch_slot_mapping(const SlotArgs& a, cudaStream_t stream) {
    if (a.num_seqs == 0) return cudaSuccess;
    const int threads = 256;
    return launch_kernel(kv_slot_mapping_kernel, dim3((a.num_seqs + threads - 1) / threads),
                         dim3(threads), 0, stream, a.pdl != 0, a);
}

}  // namespace pkv
