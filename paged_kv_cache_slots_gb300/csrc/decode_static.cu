// paged_decode_attention_static: paged_decode_attention with its scratch in a
// fixed-size array that lives in this library's device memory, for callers
// that cannot allocate device memory themselves.
//
// Who needs it: a serving engine that hands (nearly) all free device memory
// to its KV-block pool at start-up, so no allocator is left for per-call
// buffers; code that runs where allocation calls are not allowed or not
// available, such as a plugin that receives only the tensors it works on.
// Such a caller passes its inputs and outputs; the scratch comes from here.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds kStaticScratchBytes of it until the process exits.  Host
// code cannot use its name as an address (that would be a host-side stand-in,
// not device memory), so the device address is taken once per device with
// cudaGetSymbolAddress, with that device current, on the first call there.
// That first call may load the library's device code onto the device; make
// it before capturing a stream into a CUDA graph.
//
// Every call shares the one array per device and the array keeps the last
// call's contents: each accepted call clears the part that must start at
// zero (the merge counters) on its stream right before the kernel runs; a
// call that is refused queues nothing.  Two calls that overlap on the GPU
// (different streams, no ordering between them) race on the array and give
// undefined results.
//
// The device address is cached for the life of the process.  After
// cudaDeviceReset the device's module is loaded afresh and the cached
// address is stale: a process that resets a device must not call the
// library on it again (the status word's address is cached the same way).
#include <cuda_runtime.h>

#include <mutex>

#include "pkv.h"
#include "pkv_internal.h"

namespace {

// Largest scratch this entry point serves: enough for, e.g., 256 sequences x
// 32 query heads x head_dim 128 on a 152-SM GPU (about 6.8 MB).
constexpr size_t kStaticScratchBytes = size_t{8} << 20;

__device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of this device's array (taken once per device).
cudaError_t scratch_address(int device, void** out) {
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[device] == nullptr) {
        void* p = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[device] = p;
    }
    *out = g_scratch_addr[device];
    return cudaSuccess;
}

}  // namespace

extern "C" kv_status_t paged_decode_attention_static(
    const void* q, const void* k_cache, const void* v_cache, int num_blocks,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, kv_dtype_t dtype, float scale,
    void* out, kv_dtype_t out_dtype, const kv_decode_options_t* opts, void* stream) {
    int device = -1;
    if (cudaGetDevice(&device) != cudaSuccess) return KV_ERR_CUDA;
    if (device < 0 || device >= kMaxDevices) return KV_ERR_UNSUPPORTED;
    void* scratch = nullptr;
    if (scratch_address(device, &scratch) != cudaSuccess) return KV_ERR_CUDA;
    // Sizes that need more scratch than the array holds are refused here,
    // before anything is queued, with both sizes in kv_last_error().
    if (num_seqs > 0 && num_kv_heads > 0 && num_q_heads > 0 && head_dim > 0 &&
        num_q_heads % num_kv_heads == 0) {
        size_t need = 0;
        const kv_status_t st = paged_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads,
                                                            head_dim, device, opts, &need);
        if (st != KV_OK) return st;
        if (need > kStaticScratchBytes)
            return pkv::report_error(KV_ERR_WORKSPACE_TOO_SMALL,
                                     "static scratch workspace holds %zu bytes, these sizes need %zu",
                                     kStaticScratchBytes, need);
    }
    // Every other check runs inside; the merge counters are zeroed on
    // `stream` only once the call is accepted, right before its launch.
    return pkv::decode_attention_clearing_counters(q, k_cache, v_cache, num_blocks, block_tables,
                                                   max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                                                   num_kv_heads, head_dim, block_size, dtype, scale, out,
                                                   out_dtype, scratch, kStaticScratchBytes, opts, stream);
}
