// C ABI of the paged KV cache library: validation, pool bookkeeping, launch
// planning, tensor-map encoding and status handling.  Every argument is
// checked here, before anything reaches the device.
#include "pkv.h"

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <deque>
#include <mutex>
#include <new>
#include <unordered_map>
#include <vector>

#include "pkv_internal.h"

using namespace pkv;

namespace {

thread_local char g_last_error[512] = "";

kv_status_t fail(kv_status_t st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

kv_status_t cuda_fail(cudaError_t e, const char* what) {
    return fail(KV_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool valid_dtype(int d) { return d == KV_F32 || d == KV_F16 || d == KV_BF16; }
bool valid_pool_dtype(int d) { return valid_dtype(d) || d == KV_FP8_E4M3; }
bool valid_scale(float x) { return std::isfinite(x) && x > 0.f; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Restores the caller's current device on scope exit.
struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) return;
        ok = (prev == dev) || (cudaSetDevice(dev) == cudaSuccess);
    }
    ~DeviceGuard() {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
uint32_t* g_status_ptr[kMaxDevices] = {};
int g_sm_count[kMaxDevices] = {};
int g_max_smem[kMaxDevices] = {};
int g_smem_per_sm[kMaxDevices] = {};

// Per-device facts and the status word of the current device.
kv_status_t device_info(int* dev_out, uint32_t** status, int* sms, int* max_smem, int* smem_sm) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
    if (dev < 0 || dev >= kMaxDevices) return fail(KV_ERR_UNSUPPORTED, "device ordinal %d", dev);
    std::lock_guard<std::mutex> lock(g_dev_mutex);
    if (g_status_ptr[dev] == nullptr) {
        int v = 0;
        if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(SM count)");
        g_sm_count[dev] = v;
        g_max_smem[dev] = max_dynamic_smem(dev);
        if ((e = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) !=
            cudaSuccess)
            return cuda_fail(e, "cudaDeviceGetAttribute(shared memory per SM)");
        g_smem_per_sm[dev] = v;
        uint32_t* p = nullptr;
        if ((e = status_word_address(&p)) != cudaSuccess) return cuda_fail(e, "status word address");
        g_status_ptr[dev] = p;
    }
    if (dev_out) *dev_out = dev;
    if (status) *status = g_status_ptr[dev];
    if (sms) *sms = g_sm_count[dev];
    if (max_smem) *max_smem = g_max_smem[dev];
    if (smem_sm) *smem_sm = g_smem_per_sm[dev];
    return KV_OK;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct Options {
    int num_ctas, ctas_per_sm, consumer_warps, kernel, heads_per_stage, separate_reduce, no_pdl,
        early_reads, test_stall;
};

kv_status_t read_options(const kv_decode_options_t* o, Options* out) {
    Options r{0, 1, 0, KV_KERNEL_AUTO, 0, 0, 0, 0, 0};
    if (o) {
        if (o->num_ctas < 0 || o->ctas_per_sm < 0 || o->consumer_warps < 0 ||
            o->consumer_warps > 15 || o->ctas_per_sm > 8 || o->heads_per_stage < 0 ||
            o->heads_per_stage > 15)
            return fail(KV_ERR_INVALID_ARG, "decode options out of range");
        if (o->kernel != KV_KERNEL_AUTO && o->kernel != KV_KERNEL_FFMA && o->kernel != KV_KERNEL_MMA)
            return fail(KV_ERR_INVALID_ARG, "unknown kernel selector %d", static_cast<int>(o->kernel));
        if (o->num_ctas) r.num_ctas = o->num_ctas;
        if (o->ctas_per_sm) r.ctas_per_sm = o->ctas_per_sm;
        r.consumer_warps = o->consumer_warps;
        r.kernel = o->kernel;
        r.heads_per_stage = o->heads_per_stage;
        r.separate_reduce = o->separate_reduce != 0;
        r.no_pdl = o->no_pdl != 0;
        r.early_reads = o->early_reads != 0;
        r.test_stall = o->test_stall != 0;
    }
    *out = r;
    return KV_OK;
}

int grid_size(const Options& o, int sms) { return o.num_ctas > 0 ? o.num_ctas : sms * o.ctas_per_sm; }

// Workspace layout: counters [B*Hkv] int32 (must be zero between calls),
// partial O, partial (max, sum), per-sequence prefix [B+1].  The partial
// areas are sized for any head chunking: slots * Hc <= (P + B) * Hkv.
struct WsLayout {
    size_t counters, part_o, part_ml, cum, total;
};

WsLayout workspace_layout(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int ctas) {
    WsLayout w;
    const size_t rows = (static_cast<size_t>(ctas) + num_seqs) * num_q_heads;  // (P + B) * Hkv * G
    w.counters = 0;
    w.part_o = align256(static_cast<size_t>(num_seqs) * num_kv_heads * 4);
    w.part_ml = w.part_o + align256(rows * head_dim * 4);
    w.cum = w.part_ml + align256(rows * 2 * 4);
    w.total = w.cum + align256(static_cast<size_t>(num_seqs + 1) * 4);
    return w;
}

// KV heads per pipeline stage: the largest divisor of Hkv whose K slab of one
// block fits 32 KiB (and, for the tensor copies, 256 box rows).
int auto_heads_per_stage(int num_kv_heads, int block_size, int head_dim, int dtype, bool tensor) {
    const int head_bytes = block_size * head_dim * dtype_bytes(dtype);
    for (int hc = num_kv_heads < 15 ? num_kv_heads : 15; hc > 1; --hc) {
        if (num_kv_heads % hc) continue;
        if (hc * head_bytes > 32768) continue;
        if (tensor && hc * block_size > 256) continue;
        return hc;
    }
    return 1;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// 2-D view of one layer's cache: rows = num_blocks*Hkv*bs, row = head_dim
// elements; box = 128 bytes (64 f16/bf16 or 128 E4M3 elements) x box_rows
// rows (Hc heads of one block), 128-byte swizzle.
kv_status_t encode_cache_map(CUtensorMap* map, const void* base, int dtype, int rows, int head_dim,
                             int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
    const int eb = dtype_bytes(dtype);
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(head_dim), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(head_dim) * eb};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / eb), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1u, 1u};
    const CUtensorMapDataType type = dtype == KV_BF16   ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                     : dtype == KV_F16  ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                        : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = enc(map, type,
                     2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                     CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                     CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(KV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", static_cast<int>(r));
    return KV_OK;
}

}  // namespace

kv_status_t pkv::report_error(kv_status_t st, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_last_error, sizeof g_last_error, fmt, ap);
    va_end(ap);
    return st;
}

// ------------------------------------------------------------------ pool
struct kv_pool {
    kv_pool_config_t cfg;
    char* base;
    bool owned;
    size_t layer_bytes;  // one of K or V for one layer
    kv_block_allocator_t* alloc = nullptr;  // kv_seq_extend / kv_seq_free, created on first use
};

// ---------------------------------------------------------------- allocator
struct kv_block_allocator {
    int num_blocks = 0, block_size = 0;
    std::deque<int32_t> free_q;
    struct Seq {
        std::vector<int32_t> table;
        int64_t tokens = 0;
    };
    std::unordered_map<int64_t, Seq> seqs;
};

namespace {

// Moves blocks between the pool and a buffer the GPU can address.
kv_status_t swap_blocks(kv_pool_t* p, const int32_t* block_ids, int n, void* host,
                        size_t host_bytes, bool to_host, void* stream) {
    const char* what = to_host ? "kv_swap_out" : "kv_swap_in";
    if (!p) return fail(KV_ERR_INVALID_ARG, "%s: null pool", what);
    if (n < 0) return fail(KV_ERR_INVALID_ARG, "%s: %d blocks", what, n);
    if (n == 0) return KV_OK;
    if (!block_ids || !host) return fail(KV_ERR_INVALID_ARG, "%s: null pointer", what);
    const size_t need = kv_swap_bytes(p, n);
    if (host_bytes < need)
        return fail(KV_ERR_INVALID_ARG, "%s: host buffer of %zu bytes < %zu needed", what,
                    host_bytes, need);
    if (!aligned(host, 16)) return fail(KV_ERR_INVALID_ARG, "%s: host buffer must be 16-byte aligned", what);
    DeviceGuard g(p->cfg.device);
    if (!g.ok) return fail(KV_ERR_CUDA, "cannot select device %d", p->cfg.device);
    // The kernel dereferences both pointers: they must be memory the GPU
    // addresses (page-locked or registered host memory, managed or device
    // memory), not plain pageable memory.
    void* dev_ptrs[2] = {host, const_cast<int32_t*>(block_ids)};
    for (int k = 0; k < 2; ++k) {
        cudaPointerAttributes attr{};
        cudaError_t e = cudaPointerGetAttributes(&attr, dev_ptrs[k]);
        if (e != cudaSuccess) {
            cudaGetLastError();
            return cuda_fail(e, "cudaPointerGetAttributes");
        }
        if (attr.type == cudaMemoryTypeUnregistered)
            return fail(KV_ERR_INVALID_ARG,
                        "%s: %s is pageable host memory; use page-locked (cudaHostAlloc / "
                        "cudaHostRegister), managed or device memory", what,
                        k == 0 ? "the host buffer" : "block_ids");
        if (attr.type == cudaMemoryTypeHost) {
            if (!attr.devicePointer)
                return fail(KV_ERR_INVALID_ARG, "%s: host memory not mapped for the device", what);
            dev_ptrs[k] = attr.devicePointer;
        }
    }
    uint32_t* status = nullptr;
    int sms = 0;
    if (kv_status_t st = device_info(nullptr, &status, &sms, nullptr, nullptr)) return st;
    SwapArgs a{p->base,
               static_cast<char*>(dev_ptrs[0]),
               static_cast<const int32_t*>(dev_ptrs[1]),
               status,
               static_cast<int64_t>(p->layer_bytes),
               static_cast<int64_t>(p->layer_bytes / p->cfg.num_blocks),
               n,
               p->cfg.num_layers,
               p->cfg.num_blocks,
               to_host ? 1 : 0,
               1};
    cudaError_t e = launch_swap(a, sms, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "swap launch");
    return KV_OK;
}

}  // namespace

extern "C" {

const char* kv_status_string(kv_status_t s) {
    switch (s) {
        case KV_OK: return "KV_OK";
        case KV_ERR_INVALID_ARG: return "KV_ERR_INVALID_ARG";
        case KV_ERR_UNSUPPORTED: return "KV_ERR_UNSUPPORTED";
        case KV_ERR_OUT_OF_MEMORY: return "KV_ERR_OUT_OF_MEMORY";
        case KV_ERR_OUT_OF_BLOCKS: return "KV_ERR_OUT_OF_BLOCKS";
        case KV_ERR_WORKSPACE_TOO_SMALL: return "KV_ERR_WORKSPACE_TOO_SMALL";
        case KV_ERR_CUDA: return "KV_ERR_CUDA";
        case KV_ERR_DEVICE_CHECK: return "KV_ERR_DEVICE_CHECK";
        case KV_ERR_DEVICE_TIMEOUT: return "KV_ERR_DEVICE_TIMEOUT";
        case KV_ERR_NOT_FOUND: return "KV_ERR_NOT_FOUND";
    }
    return "KV_ERR_UNKNOWN";
}

const char* kv_last_error(void) { return g_last_error; }

size_t kv_pool_bytes(const kv_pool_config_t* c) {
    if (!c || c->num_layers <= 0 || c->num_blocks <= 0 || c->block_size <= 0 || c->num_kv_heads <= 0 ||
        c->head_dim <= 0 || !valid_pool_dtype(c->dtype))
        return 0;
    return 2ull * c->num_layers * c->num_blocks * c->block_size * c->num_kv_heads * c->head_dim *
           static_cast<size_t>(dtype_bytes(c->dtype));
}

kv_status_t kv_pool_create(const kv_pool_config_t* cfg, void* buffer, size_t buffer_bytes,
                           kv_pool_t** out) {
    if (!cfg || !out) return fail(KV_ERR_INVALID_ARG, "kv_pool_create: null argument");
    *out = nullptr;
    const size_t bytes = kv_pool_bytes(cfg);
    if (bytes == 0) return fail(KV_ERR_INVALID_ARG, "kv_pool_create: invalid configuration");
    if (cfg->block_size > 1024) return fail(KV_ERR_INVALID_ARG, "block_size %d > 1024", cfg->block_size);
    if ((static_cast<size_t>(cfg->head_dim) * dtype_bytes(cfg->dtype)) % 16)
        return fail(KV_ERR_INVALID_ARG, "head_dim * element size must be a multiple of 16 bytes");
    if (static_cast<int64_t>(cfg->num_blocks) * cfg->block_size >= (int64_t{1} << 31) ||
        static_cast<int64_t>(cfg->num_blocks) * cfg->block_size * cfg->num_kv_heads >= (int64_t{1} << 31))
        return fail(KV_ERR_UNSUPPORTED, "pool too large for 32-bit slot / row indices");
    if (cfg->device < 0) return fail(KV_ERR_INVALID_ARG, "device %d", cfg->device);
    if (buffer) {
        if (buffer_bytes < bytes)
            return fail(KV_ERR_INVALID_ARG, "buffer of %zu bytes < %zu needed", buffer_bytes, bytes);
        if (!aligned(buffer, 256)) return fail(KV_ERR_INVALID_ARG, "pool buffer must be 256-byte aligned");
    }
    kv_pool* p = new (std::nothrow) kv_pool;
    if (!p) return fail(KV_ERR_OUT_OF_MEMORY, "host allocation failed");
    p->cfg = *cfg;
    p->layer_bytes = bytes / (2ull * cfg->num_layers);
    p->owned = buffer == nullptr;
    p->base = static_cast<char*>(buffer);
    if (!buffer) {
        DeviceGuard g(cfg->device);
        if (!g.ok) {
            delete p;
            return fail(KV_ERR_CUDA, "cannot select device %d", cfg->device);
        }
        void* mem = nullptr;
        cudaError_t e = cudaMalloc(&mem, bytes);
        if (e != cudaSuccess) {
            delete p;
            cudaGetLastError();
            return fail(KV_ERR_OUT_OF_MEMORY, "cudaMalloc(%zu): %s", bytes, cudaGetErrorString(e));
        }
        p->base = static_cast<char*>(mem);
    }
    *out = p;
    return KV_OK;
}

void kv_pool_destroy(kv_pool_t* p) {
    if (!p) return;
    if (p->owned && p->base) {
        DeviceGuard g(p->cfg.device);
        cudaFree(p->base);
    }
    kv_allocator_destroy(p->alloc);
    delete p;
}

kv_status_t kv_pool_layer(const kv_pool_t* p, int layer, void** k, void** v) {
    if (!p || !k || !v) return fail(KV_ERR_INVALID_ARG, "kv_pool_layer: null argument");
    if (layer < 0 || layer >= p->cfg.num_layers)
        return fail(KV_ERR_INVALID_ARG, "layer %d outside [0, %d)", layer, p->cfg.num_layers);
    *k = p->base + (2ull * layer) * p->layer_bytes;
    *v = p->base + (2ull * layer + 1) * p->layer_bytes;
    return KV_OK;
}

kv_status_t kv_pool_config(const kv_pool_t* p, kv_pool_config_t* c) {
    if (!p || !c) return fail(KV_ERR_INVALID_ARG, "kv_pool_config: null argument");
    *c = p->cfg;
    return KV_OK;
}

kv_status_t kv_slot_mapping(const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                            int num_seqs, int block_size, int num_blocks, int32_t* slot_mapping,
                            void* stream) {
    if (num_seqs < 0 || max_blocks <= 0 || block_size <= 0 || num_blocks <= 0)
        return fail(KV_ERR_INVALID_ARG, "kv_slot_mapping: sizes out of range");
    if (num_seqs == 0) return KV_OK;
    if (!block_tables || !context_lens || !slot_mapping)
        return fail(KV_ERR_INVALID_ARG, "kv_slot_mapping: null pointer");
    if (static_cast<int64_t>(num_blocks) * block_size >= (int64_t{1} << 31))
        return fail(KV_ERR_UNSUPPORTED, "slots do not fit in int32");
    uint32_t* status = nullptr;
    if (kv_status_t st = device_info(nullptr, &status, nullptr, nullptr, nullptr)) return st;
    SlotArgs a{block_tables, context_lens, slot_mapping, status, max_blocks, num_seqs, block_size, num_blocks,
               1};
    cudaError_t e = launch_slot_mapping(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "slot mapping launch");
    return KV_OK;
}

kv_status_t kv_append(kv_pool_t* p, int layer, const int32_t* seq_ids, int n_tokens, const void* k,
                      const void* v, const int32_t* slot_mapping, void* stream) {
    if (!p) return fail(KV_ERR_INVALID_ARG, "kv_append: null pool");
    if (n_tokens < 0) return fail(KV_ERR_INVALID_ARG, "kv_append: n_tokens %d", n_tokens);
    if (p->cfg.dtype == KV_FP8_E4M3)
        return fail(KV_ERR_INVALID_ARG, "kv_append: an E4M3 pool takes kv_append_fp8 (with scales)");
    void *kc = nullptr, *vc = nullptr;
    if (kv_status_t st = kv_pool_layer(p, layer, &kc, &vc)) return st;
    if (n_tokens == 0) return KV_OK;
    if (!k || !v || !slot_mapping) return fail(KV_ERR_INVALID_ARG, "kv_append: null pointer");
    if (!aligned(k, 16) || !aligned(v, 16))
        return fail(KV_ERR_INVALID_ARG, "kv_append: k and v must be 16-byte aligned");
    if (static_cast<int64_t>(n_tokens) * p->cfg.num_kv_heads >= (int64_t{1} << 31) / 32)
        return fail(KV_ERR_UNSUPPORTED, "kv_append: too many tokens in one call");
    uint32_t* status = nullptr;
    if (kv_status_t st = device_info(nullptr, &status, nullptr, nullptr, nullptr)) return st;
    AppendArgs a{seq_ids, k, v, slot_mapping, kc, vc, status, n_tokens, p->cfg.num_kv_heads,
                 p->cfg.head_dim, p->cfg.block_size, p->cfg.num_blocks, dtype_bytes(p->cfg.dtype), 1,
                 0, p->cfg.dtype, 1.f, 1.f};
    cudaError_t e = launch_append(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return KV_OK;
}

kv_status_t kv_append_fp8(kv_pool_t* p, int layer, const int32_t* seq_ids, int n_tokens, const void* k,
                          const void* v, kv_dtype_t src_dtype, const int32_t* slot_mapping, float k_scale,
                          float v_scale, void* stream) {
    if (!p) return fail(KV_ERR_INVALID_ARG, "kv_append_fp8: null pool");
    if (p->cfg.dtype != KV_FP8_E4M3)
        return fail(KV_ERR_INVALID_ARG, "kv_append_fp8: the pool is not KV_FP8_E4M3");
    if (!valid_dtype(src_dtype)) return fail(KV_ERR_INVALID_ARG, "kv_append_fp8: source dtype %d", src_dtype);
    if (!valid_scale(k_scale) || !valid_scale(v_scale))
        return fail(KV_ERR_INVALID_ARG, "kv_append_fp8: scales must be finite and > 0");
    if (n_tokens < 0) return fail(KV_ERR_INVALID_ARG, "kv_append_fp8: n_tokens %d", n_tokens);
    if (p->cfg.head_dim % 16)
        return fail(KV_ERR_UNSUPPORTED, "kv_append_fp8: head_dim must be a multiple of 16");
    void *kc = nullptr, *vc = nullptr;
    if (kv_status_t st = kv_pool_layer(p, layer, &kc, &vc)) return st;
    if (n_tokens == 0) return KV_OK;
    if (!k || !v || !slot_mapping) return fail(KV_ERR_INVALID_ARG, "kv_append_fp8: null pointer");
    if (!aligned(k, 16) || !aligned(v, 16))
        return fail(KV_ERR_INVALID_ARG, "kv_append_fp8: k and v must be 16-byte aligned");
    if (static_cast<int64_t>(n_tokens) * p->cfg.num_kv_heads >= (int64_t{1} << 31) / 32)
        return fail(KV_ERR_UNSUPPORTED, "kv_append_fp8: too many tokens in one call");
    uint32_t* status = nullptr;
    if (kv_status_t st = device_info(nullptr, &status, nullptr, nullptr, nullptr)) return st;
    AppendArgs a{seq_ids, k, v, slot_mapping, kc, vc, status, n_tokens, p->cfg.num_kv_heads,
                 p->cfg.head_dim, p->cfg.block_size, p->cfg.num_blocks, 1, 1,
                 1, src_dtype, k_scale, v_scale};
    cudaError_t e = launch_append(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "append launch");
    return KV_OK;
}

size_t kv_swap_bytes(const kv_pool_t* p, int num_blocks) {
    if (!p || num_blocks < 0) return 0;
    return static_cast<size_t>(num_blocks) * 2 * p->layer_bytes / p->cfg.num_blocks *
           p->cfg.num_layers;
}

kv_status_t kv_swap_out(const kv_pool_t* p, const int32_t* block_ids, int n, void* host_dst,
                        size_t host_bytes, void* stream) {
    return swap_blocks(const_cast<kv_pool_t*>(p), block_ids, n, host_dst, host_bytes, true, stream);
}

kv_status_t kv_swap_in(kv_pool_t* p, const int32_t* block_ids, int n, const void* host_src,
                       size_t host_bytes, void* stream) {
    return swap_blocks(p, block_ids, n, const_cast<void*>(host_src), host_bytes, false, stream);
}

kv_status_t paged_decode_workspace_bytes(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                         int device, const kv_decode_options_t* opts, size_t* bytes) {
    if (!bytes) return fail(KV_ERR_INVALID_ARG, "null bytes_out");
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        num_q_heads % num_kv_heads)
        return fail(KV_ERR_INVALID_ARG, "workspace: sizes out of range");
    Options o;
    if (kv_status_t st = read_options(opts, &o)) return st;
    int sms = 0;
    if (o.num_ctas <= 0) {
        DeviceGuard g(device);
        if (!g.ok) return fail(KV_ERR_CUDA, "cannot select device %d", device);
        if (kv_status_t st = device_info(nullptr, nullptr, &sms, nullptr, nullptr)) return st;
    }
    *bytes = workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, grid_size(o, sms)).total;
    return KV_OK;
}

kv_status_t paged_decode_workspace_init(void* workspace, size_t workspace_bytes, int num_seqs,
                                        int num_kv_heads, void* stream) {
    if (num_seqs < 0 || num_kv_heads <= 0) return fail(KV_ERR_INVALID_ARG, "workspace init: sizes");
    const size_t n = static_cast<size_t>(num_seqs) * num_kv_heads * 4;
    if (n == 0) return KV_OK;
    if (!workspace || workspace_bytes < n) return fail(KV_ERR_INVALID_ARG, "workspace init: buffer");
    cudaError_t e = cudaMemsetAsync(workspace, 0, n, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    return KV_OK;
}

static kv_status_t decode_impl(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                               const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, kv_dtype_t dtype, float scale, void* out,
                               kv_dtype_t out_dtype, void* workspace, size_t workspace_bytes,
                               const kv_decode_options_t* opts, void* stream, const void* k_new,
                               const void* v_new, const int32_t* append_ids, int32_t* slot_out,
                               kv_dtype_t kv_dtype, float k_scale, float v_scale,
                               bool clear_counters = false) {
    const bool fp8 = kv_dtype == KV_FP8_E4M3;
    if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 || max_blocks <= 0)
        return fail(KV_ERR_INVALID_ARG, "paged_decode_attention: sizes out of range");
    if (num_q_heads % num_kv_heads)
        return fail(KV_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                    num_kv_heads);
    const int G = num_q_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(KV_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4 or 8 (got %d)", G);
    if (head_dim != 64 && head_dim != 128) return fail(KV_ERR_UNSUPPORTED, "head_dim %d", head_dim);
    if (block_size < 1 || block_size > 256) return fail(KV_ERR_UNSUPPORTED, "block_size %d", block_size);
    if (!valid_dtype(dtype) || !valid_dtype(out_dtype))
        return fail(KV_ERR_INVALID_ARG, "unknown dtype");
    if (fp8) {
        if (dtype != KV_F16 && dtype != KV_BF16)
            return fail(KV_ERR_UNSUPPORTED, "an E4M3 cache takes an f16 or bf16 q");
        if (head_dim != 128) return fail(KV_ERR_UNSUPPORTED, "an E4M3 cache needs head_dim 128");
        if (!valid_scale(k_scale) || !valid_scale(v_scale))
            return fail(KV_ERR_INVALID_ARG, "k_scale and v_scale must be finite and > 0");
    } else if (kv_dtype != dtype) {
        return fail(KV_ERR_INVALID_ARG, "the cache must have q's dtype (or be E4M3)");
    }
    if (out_dtype != KV_F32 && out_dtype != dtype)
        return fail(KV_ERR_UNSUPPORTED, "out_dtype must be KV_F32 or the input dtype");
    if (!std::isfinite(scale)) return fail(KV_ERR_INVALID_ARG, "scale is not finite");
    if (static_cast<int64_t>(num_seqs) * num_kv_heads * max_blocks >= (int64_t{1} << 31) ||
        static_cast<int64_t>(num_blocks) * num_kv_heads * block_size >= (int64_t{1} << 31))
        return fail(KV_ERR_UNSUPPORTED, "sizes exceed 32-bit tile / row indices");
    Options o;
    if (kv_status_t st = read_options(opts, &o)) return st;
    int kernel = o.kernel;
    const bool mma_ok = (dtype == KV_F16 || dtype == KV_BF16) && block_size % 16 == 0;
    if (kernel == KV_KERNEL_AUTO) kernel = mma_ok ? KV_KERNEL_MMA : KV_KERNEL_FFMA;
    if (kernel == KV_KERNEL_MMA && !mma_ok)
        return fail(KV_ERR_UNSUPPORTED, "tensor-core kernel needs f16/bf16 and block_size % 16 == 0");
    if (fp8 && kernel != KV_KERNEL_MMA)
        return fail(KV_ERR_UNSUPPORTED, "an E4M3 cache is read by the tensor-core kernel only "
                                        "(block_size a multiple of 16)");
    if (num_seqs == 0) return KV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !context_lens || !out || !workspace)
        return fail(KV_ERR_INVALID_ARG, "paged_decode_attention: null pointer");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16) ||
        !aligned(workspace, 256))
        return fail(KV_ERR_INVALID_ARG,
                    "alignment: caches, q and out need 16 bytes, the workspace 256 bytes");
    if ((k_new == nullptr) != (v_new == nullptr))
        return fail(KV_ERR_INVALID_ARG, "k_new and v_new go together");
    if (k_new && (!aligned(k_new, 16) || !aligned(v_new, 16)))
        return fail(KV_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    int dev = 0, sms = 0, max_smem = 0, smem_sm = 0;
    uint32_t* status = nullptr;
    if (kv_status_t st = device_info(&dev, &status, &sms, &max_smem, &smem_sm)) return st;
    const int P = grid_size(o, sms);
    const WsLayout wl = workspace_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, P);
    if (workspace_bytes < wl.total)
        return fail(KV_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", workspace_bytes,
                    wl.total);
    // Head chunking and warps: Hc KV heads per stage, R warps per head.
    int hc = o.heads_per_stage;
    if (hc == 0) {
        hc = auto_heads_per_stage(num_kv_heads, block_size, head_dim, kv_dtype, kernel == KV_KERNEL_MMA);
    } else if (num_kv_heads % hc) {
        return fail(KV_ERR_INVALID_ARG, "heads_per_stage %d does not divide num_kv_heads %d", hc,
                    num_kv_heads);
    }
    if (kernel == KV_KERNEL_MMA && hc * block_size > 256)
        return fail(KV_ERR_UNSUPPORTED, "heads_per_stage * block_size must be <= 256 for the tensor copies");
    const int target = o.consumer_warps ? o.consumer_warps : 8;
    int R = target / hc;
    if (R < 1) R = 1;
    while (hc * R > 15 && R > 1) --R;
    if (hc * R > 15) return fail(KV_ERR_UNSUPPORTED, "more than 15 consumer warps");
    int budget = max_smem;
    if (o.ctas_per_sm > 1) {
        const int share = smem_sm / o.ctas_per_sm - 1024;
        if (share < budget) budget = share;
    }
    // Fewer warps per head when the ring would hold less than two stages per
    // replica (each replica owns every R-th stage).
    DecodePlan plan{};
    bool planned = false;
    for (; R >= 1; --R) {
        planned = decode_plan(kernel, kv_dtype, head_dim, block_size, G, num_seqs, hc, R, budget, &plan);
        if (planned && (plan.stages >= 2 * R || R == 1)) break;
        if (planned && o.consumer_warps) break;  // an explicit warp count is kept if it fits at all
    }
    if (!planned) return fail(KV_ERR_UNSUPPORTED, "shared memory cannot hold two stages for these sizes");

    char* ws = static_cast<char*>(workspace);
    DecodeArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.out = out;
    a.counters = reinterpret_cast<int32_t*>(ws + wl.counters);
    a.part_o = reinterpret_cast<float*>(ws + wl.part_o);
    a.part_ml = reinterpret_cast<float*>(ws + wl.part_ml);
    a.cum = reinterpret_cast<int32_t*>(ws + wl.cum);
    a.status = status;
    a.num_blocks = num_blocks;
    a.max_blocks = max_blocks;
    a.num_seqs = num_seqs;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.dtype = dtype;
    a.out_dtype = out_dtype;
    a.kv_dtype = kv_dtype;
    a.k_scale = fp8 ? k_scale : 1.f;
    a.v_scale = fp8 ? v_scale : 1.f;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634 *
                                      static_cast<double>(a.k_scale));
    a.num_ctas = P;
    a.heads_per_stage = hc;
    a.warps_per_head = R;
    a.consumer_warps = hc * R;
    a.stages = plan.stages;
    a.smem_bytes = plan.smem_bytes;
    a.fused_reduce = o.separate_reduce ? 0 : 1;
    a.pdl = o.no_pdl ? 0 : 1;
    a.early_reads = (o.early_reads && !o.no_pdl) ? 1 : 0;
    a.test_stall = o.test_stall;
    // Phantom items per pair: about the time a CTA loses switching to the
    // next pair (the partial's stores, the merge arrival's release fence,
    // the next q: 3-5 us measured) in stages' worth of streaming, i.e.
    // 300 KiB of stage data: 5 items for 64 KiB stages, 8 (the cap) for the
    // E4M3 stages of 32 KiB (the best of 0, 100, 200, 300 and 400 KiB in an
    // A/B on one box).  Not with too few items to split (fewer than two a
    // CTA even with every table entry used).
    {
        const int64_t stage_bytes = 2 * static_cast<int64_t>(plan.stage_half_bytes);
        const int64_t max_items = static_cast<int64_t>(num_seqs) * (num_kv_heads / hc) * max_blocks;
        int ph = static_cast<int>((int64_t{300} * 1024 + stage_bytes / 2) / stage_bytes);
        a.phantom = max_items >= 2 * static_cast<int64_t>(P) ? (ph > 8 ? 8 : ph) : 0;
    }
    a.device = dev;
    a.k_new = k_new;
    a.v_new = v_new;
    a.append_ids = append_ids;
    a.slot_out = slot_out;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    CUtensorMap tk, tv;
    if (kernel == KV_KERNEL_MMA) {
        const int rows = num_blocks * num_kv_heads * block_size;
        if (kv_status_t st = encode_cache_map(&tk, k_cache, kv_dtype, rows, head_dim, hc * block_size)) return st;
        if (kv_status_t st = encode_cache_map(&tv, v_cache, kv_dtype, rows, head_dim, hc * block_size)) return st;
    }
    if (clear_counters) {
        e = cudaMemsetAsync(ws + wl.counters, 0, static_cast<size_t>(num_seqs) * num_kv_heads * 4, s);
        if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync");
    }
    if (kernel == KV_KERNEL_MMA) {
        e = fp8 ? launch_decode_fp8(a, tk, tv, s) : launch_decode_mma(a, tk, tv, s);
    } else {
        e = launch_decode_ffma(a, s);
    }
    if (e != cudaSuccess) return cuda_fail(e, "decode partial launch");
    if (!a.fused_reduce) {
        e = launch_decode_reduce(a, s);
        if (e != cudaSuccess) return cuda_fail(e, "decode reduce launch");
    }
    return KV_OK;
}

kv_status_t paged_decode_attention(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                                   const int32_t* block_tables, int max_blocks, const int32_t* context_lens,
                                   int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, kv_dtype_t dtype, float scale, void* out,
                                   kv_dtype_t out_dtype, void* workspace, size_t workspace_bytes,
                                   const kv_decode_options_t* opts, void* stream) {
    return decode_impl(q, k_cache, v_cache, num_blocks, block_tables, max_blocks, context_lens, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, dtype, scale, out, out_dtype,
                       workspace, workspace_bytes, opts, stream, nullptr, nullptr, nullptr, nullptr,
                       dtype, 1.f, 1.f);
}

kv_status_t paged_decode_append_attention(const void* q, const void* k_new, const void* v_new,
                                          const int32_t* seq_ids, void* k_cache, void* v_cache,
                                          int num_blocks, const int32_t* block_tables, int max_blocks,
                                          const int32_t* context_lens, int num_seqs, int num_q_heads,
                                          int num_kv_heads, int head_dim, int block_size,
                                          kv_dtype_t dtype, float scale, void* out, kv_dtype_t out_dtype,
                                          int32_t* slot_mapping, void* workspace,
                                          size_t workspace_bytes, const kv_decode_options_t* opts,
                                          void* stream) {
    if (num_seqs > 0 && (!k_new || !v_new))
        return fail(KV_ERR_INVALID_ARG, "paged_decode_append_attention: null k_new / v_new");
    return decode_impl(q, k_cache, v_cache, num_blocks, block_tables, max_blocks, context_lens, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, dtype, scale, out, out_dtype,
                       workspace, workspace_bytes, opts, stream, k_new, v_new, seq_ids, slot_mapping,
                       dtype, 1.f, 1.f);
}

kv_status_t paged_decode_attention_fp8(const void* q, kv_dtype_t q_dtype, const void* k_cache,
                                       const void* v_cache, float k_scale, float v_scale, int num_blocks,
                                       const int32_t* block_tables, int max_blocks,
                                       const int32_t* context_lens, int num_seqs, int num_q_heads,
                                       int num_kv_heads, int head_dim, int block_size, float scale,
                                       void* out, kv_dtype_t out_dtype, void* workspace,
                                       size_t workspace_bytes, const kv_decode_options_t* opts,
                                       void* stream) {
    return decode_impl(q, k_cache, v_cache, num_blocks, block_tables, max_blocks, context_lens, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, q_dtype, scale, out, out_dtype,
                       workspace, workspace_bytes, opts, stream, nullptr, nullptr, nullptr, nullptr,
                       KV_FP8_E4M3, k_scale, v_scale);
}

kv_status_t paged_decode_append_attention_fp8(const void* q, const void* k_new, const void* v_new,
                                              const int32_t* seq_ids, kv_dtype_t q_dtype, void* k_cache,
                                              void* v_cache, float k_scale, float v_scale, int num_blocks,
                                              const int32_t* block_tables, int max_blocks,
                                              const int32_t* context_lens, int num_seqs, int num_q_heads,
                                              int num_kv_heads, int head_dim, int block_size, float scale,
                                              void* out, kv_dtype_t out_dtype, int32_t* slot_mapping,
                                              void* workspace, size_t workspace_bytes,
                                              const kv_decode_options_t* opts, void* stream) {
    if (num_seqs > 0 && (!k_new || !v_new))
        return fail(KV_ERR_INVALID_ARG, "paged_decode_append_attention_fp8: null k_new / v_new");
    return decode_impl(q, k_cache, v_cache, num_blocks, block_tables, max_blocks, context_lens, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, q_dtype, scale, out, out_dtype,
                       workspace, workspace_bytes, opts, stream, k_new, v_new, seq_ids, slot_mapping,
                       KV_FP8_E4M3, k_scale, v_scale);
}

// ------------------------------------------------------ multi-token queries
size_t paged_prefill_workspace_bytes(int num_seqs) {
    if (num_seqs < 0) return 0;
    return align256(static_cast<size_t>(num_seqs + 1) * 4);
}

kv_status_t kv_slot_mapping_varlen(const int32_t* block_tables, int max_blocks, const int32_t* query_start,
                                   const int32_t* context_lens, int num_seqs, int num_tokens, int block_size,
                                   int num_blocks, int32_t* slot_mapping, void* stream) {
    if (num_seqs < 0 || num_tokens < 0 || max_blocks <= 0 || block_size <= 0 || num_blocks <= 0)
        return fail(KV_ERR_INVALID_ARG, "kv_slot_mapping_varlen: sizes out of range");
    if (num_seqs == 0) return KV_OK;
    if (!block_tables || !query_start || !context_lens || (num_tokens > 0 && !slot_mapping))
        return fail(KV_ERR_INVALID_ARG, "kv_slot_mapping_varlen: null pointer");
    uint32_t* status = nullptr;
    if (kv_status_t st = device_info(nullptr, &status, nullptr, nullptr, nullptr)) return st;
    PrefillArgs a{};
    a.block_tables = block_tables;
    a.query_start = query_start;
    a.context_lens = context_lens;
    a.status = status;
    a.num_blocks = num_blocks;
    a.max_blocks = max_blocks;
    a.num_seqs = num_seqs;
    a.num_tokens = num_tokens;
    a.block_size = block_size;
    a.pdl = 1;
    cudaError_t e = launch_slot_mapping_varlen(a, slot_mapping, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "varlen slot mapping launch");
    return KV_OK;
}

static kv_status_t prefill_impl(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                                const int32_t* block_tables, int max_blocks, const int32_t* query_start,
                                const int32_t* context_lens, int num_seqs, int num_tokens, int num_q_heads,
                                int num_kv_heads, int head_dim, int block_size, kv_dtype_t dtype,
                                kv_dtype_t kv_dtype, float k_scale, float v_scale, float scale, void* out,
                                kv_dtype_t out_dtype, void* workspace, size_t workspace_bytes, void* stream) {
    const bool fp8 = kv_dtype == KV_FP8_E4M3;
    if (num_seqs < 0 || num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
        max_blocks <= 0)
        return fail(KV_ERR_INVALID_ARG, "paged_prefill_attention: sizes out of range");
    if (num_q_heads % num_kv_heads)
        return fail(KV_ERR_INVALID_ARG, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                    num_kv_heads);
    const int G = num_q_heads / num_kv_heads;
    if (G != 1 && G != 2 && G != 4 && G != 8)
        return fail(KV_ERR_UNSUPPORTED, "query heads per KV head must be 1, 2, 4 or 8 (got %d)", G);
    if (head_dim != 64 && head_dim != 128) return fail(KV_ERR_UNSUPPORTED, "head_dim %d", head_dim);
    if (dtype == KV_F32 && !fp8) {
        if (block_size < 1 || block_size > 256)
            return fail(KV_ERR_UNSUPPORTED, "block_size must be 1 .. 256");
    } else if (block_size % 16 || block_size < 16 || block_size > 256) {
        return fail(KV_ERR_UNSUPPORTED, "multi-token queries on f16/bf16 need block_size a multiple of 16 up to 256");
    }
    if (fp8) {
        if (dtype != KV_F16 && dtype != KV_BF16)
            return fail(KV_ERR_UNSUPPORTED, "an E4M3 cache takes an f16 or bf16 q");
        if (head_dim != 128) return fail(KV_ERR_UNSUPPORTED, "an E4M3 cache needs head_dim 128");
        if (!valid_scale(k_scale) || !valid_scale(v_scale))
            return fail(KV_ERR_INVALID_ARG, "k_scale and v_scale must be finite and > 0");
    } else if (dtype != KV_F32 && dtype != KV_F16 && dtype != KV_BF16) {
        return fail(KV_ERR_INVALID_ARG, "unknown dtype");
    }
    if (out_dtype != KV_F32 && out_dtype != dtype)
        return fail(KV_ERR_UNSUPPORTED, "out_dtype must be KV_F32 or the input dtype");
    if (!std::isfinite(scale)) return fail(KV_ERR_INVALID_ARG, "scale is not finite");
    if (static_cast<int64_t>(num_blocks) * num_kv_heads * block_size >= (int64_t{1} << 31))
        return fail(KV_ERR_UNSUPPORTED, "sizes exceed 32-bit row indices");
    if (num_seqs == 0 || num_tokens == 0) return KV_OK;
    if (!q || !k_cache || !v_cache || !block_tables || !query_start || !context_lens || !out || !workspace)
        return fail(KV_ERR_INVALID_ARG, "paged_prefill_attention: null pointer");
    if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(q, 16) || !aligned(out, 16) ||
        !aligned(workspace, 16))
        return fail(KV_ERR_INVALID_ARG, "alignment: caches, q, out and the workspace need 16 bytes");
    if (workspace_bytes < paged_prefill_workspace_bytes(num_seqs))
        return fail(KV_ERR_WORKSPACE_TOO_SMALL, "workspace %zu bytes < %zu needed", workspace_bytes,
                    paged_prefill_workspace_bytes(num_seqs));
    int dev = 0, max_smem = 0;
    uint32_t* status = nullptr;
    if (kv_status_t st = device_info(&dev, &status, nullptr, &max_smem, nullptr)) return st;
    // The tcgen05 kernel: f16/bf16 cache, head_dim 128, blocks that tile 64-key tiles evenly.
    const bool tc = !fp8 && dtype != KV_F32 && head_dim == 128 &&
                    (block_size % 64 == 0 || 64 % block_size == 0) && prefill_tc_smem_bytes() <= max_smem;
    // Stages of the warp-MMA kernel hold K and V in q's 2-byte type (an E4M3
    // block converted); E4M3 adds two raw slots of codes.
    const int stage_bytes = 2 * block_size * head_dim * 2;
    const int raw_bytes = fp8 ? 4 * block_size * head_dim : 0;
    int stages = (max_smem - 2048 - 64 - raw_bytes) / stage_bytes;
    if (stages > 4) stages = 4;
    if (!tc && dtype != KV_F32 && stages < 2) return fail(KV_ERR_UNSUPPORTED, "shared memory cannot hold two stages");
    PrefillArgs a{};
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.query_start = query_start;
    a.context_lens = context_lens;
    a.out = out;
    a.tile_cum = static_cast<int32_t*>(workspace);
    a.status = status;
    a.num_blocks = num_blocks;
    a.max_blocks = max_blocks;
    a.num_seqs = num_seqs;
    a.num_tokens = num_tokens;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.block_size = block_size;
    a.dtype = dtype;
    a.out_dtype = out_dtype;
    a.kv_dtype = fp8 ? KV_FP8_E4M3 : dtype;
    a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634 *
                                      static_cast<double>(fp8 ? k_scale : 1.f));
    a.v_scale = fp8 ? v_scale : 1.f;
    a.stages = stages;
    a.smem_bytes = tc ? prefill_tc_smem_bytes()
                      : fp8 ? 1024 + stages * stage_bytes + 1024 + raw_bytes
                            : 1024 + stages * stage_bytes + stages * 16 + 32;
    a.tensor_cores = tc ? 1 : 0;
    a.tile_tokens = tc ? 128 / G : 16;
    const int64_t tiles = (static_cast<int64_t>(num_tokens) + a.tile_tokens - 1) / a.tile_tokens + num_seqs;
    if (tiles >= (int64_t{1} << 31)) return fail(KV_ERR_UNSUPPORTED, "too many query tiles");
    a.grid_tiles = static_cast<int>(tiles);
    a.pdl = 1;
    a.device = dev;
    CUtensorMap tk{}, tv{};
    if (!fp8 && dtype != KV_F32) {  // E4M3 tiles come by bulk copies, f32 rows by plain loads
        const int rows = num_blocks * num_kv_heads * block_size;
        const int box_rows = tc ? (block_size < 64 ? block_size : 64) : block_size;
        if (kv_status_t st = encode_cache_map(&tk, k_cache, dtype, rows, head_dim, box_rows)) return st;
        if (kv_status_t st = encode_cache_map(&tv, v_cache, dtype, rows, head_dim, box_rows)) return st;
    }
    cudaError_t e = launch_prefill(a, tk, tv, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "prefill launch");
    return KV_OK;
}

kv_status_t paged_prefill_attention(const void* q, const void* k_cache, const void* v_cache, int num_blocks,
                                    const int32_t* block_tables, int max_blocks, const int32_t* query_start,
                                    const int32_t* context_lens, int num_seqs, int num_tokens, int num_q_heads,
                                    int num_kv_heads, int head_dim, int block_size, kv_dtype_t dtype,
                                    float scale, void* out, kv_dtype_t out_dtype, void* workspace,
                                    size_t workspace_bytes, void* stream) {
    if (dtype == KV_FP8_E4M3)
        return fail(KV_ERR_INVALID_ARG, "paged_prefill_attention: an E4M3 cache goes to paged_prefill_attention_fp8");
    return prefill_impl(q, k_cache, v_cache, num_blocks, block_tables, max_blocks, query_start, context_lens,
                        num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size, dtype, dtype, 1.f,
                        1.f, scale, out, out_dtype, workspace, workspace_bytes, stream);
}

kv_status_t paged_prefill_attention_fp8(const void* q, kv_dtype_t q_dtype, const void* k_cache,
                                        const void* v_cache, float k_scale, float v_scale, int num_blocks,
                                        const int32_t* block_tables, int max_blocks, const int32_t* query_start,
                                        const int32_t* context_lens, int num_seqs, int num_tokens,
                                        int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                        float scale, void* out, kv_dtype_t out_dtype, void* workspace,
                                        size_t workspace_bytes, void* stream) {
    return prefill_impl(q, k_cache, v_cache, num_blocks, block_tables, max_blocks, query_start, context_lens,
                        num_seqs, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size, q_dtype,
                        KV_FP8_E4M3, k_scale, v_scale, scale, out, out_dtype, workspace, workspace_bytes, stream);
}

kv_status_t kv_device_status(int device, void* stream, uint32_t* flags_out) {
    DeviceGuard g(device);
    if (!g.ok) return fail(KV_ERR_CUDA, "cannot select device %d", device);
    uint32_t* status = nullptr;
    if (kv_status_t st = device_info(nullptr, &status, nullptr, nullptr, nullptr)) return st;
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    uint32_t flags = 0;
    if ((e = cudaMemcpy(&flags, status, sizeof flags, cudaMemcpyDeviceToHost)) != cudaSuccess)
        return cuda_fail(e, "reading the status word");
    if (flags && (e = cudaMemset(status, 0, sizeof flags)) != cudaSuccess)
        return cuda_fail(e, "clearing the status word");
    if (flags_out) *flags_out = flags;
    if (!flags) return KV_OK;
    if (flags & KV_FLAG_TIMEOUT) return fail(KV_ERR_DEVICE_TIMEOUT, "a kernel gave up a bounded wait");
    return fail(KV_ERR_DEVICE_CHECK, "device check flags 0x%x", flags);
}

// ------------------------------------------------------------ allocator
kv_status_t kv_allocator_create(int num_blocks, int block_size, int reserve_null_block,
                                kv_block_allocator_t** out) {
    if (!out) return fail(KV_ERR_INVALID_ARG, "null out");
    *out = nullptr;
    if (num_blocks <= 0 || block_size <= 0) return fail(KV_ERR_INVALID_ARG, "allocator sizes");
    kv_block_allocator* a = new (std::nothrow) kv_block_allocator;
    if (!a) return fail(KV_ERR_OUT_OF_MEMORY, "host allocation failed");
    a->num_blocks = num_blocks;
    a->block_size = block_size;
    for (int b = reserve_null_block ? 1 : 0; b < num_blocks; ++b) a->free_q.push_back(b);
    *out = a;
    return KV_OK;
}

void kv_allocator_destroy(kv_block_allocator_t* a) { delete a; }

kv_status_t kv_allocator_extend(kv_block_allocator_t* a, int64_t seq_id, int new_tokens) {
    if (!a || new_tokens < 0) return fail(KV_ERR_INVALID_ARG, "kv_allocator_extend arguments");
    auto it = a->seqs.find(seq_id);
    const int64_t have_tokens = it == a->seqs.end() ? 0 : it->second.tokens;
    const size_t have_blocks = it == a->seqs.end() ? 0 : it->second.table.size();
    const int64_t total = have_tokens + new_tokens;
    const int64_t need_blocks = (total + a->block_size - 1) / a->block_size - static_cast<int64_t>(have_blocks);
    if (need_blocks > static_cast<int64_t>(a->free_q.size()))
        return fail(KV_ERR_OUT_OF_BLOCKS, "sequence %lld needs %lld blocks, %zu free",
                    static_cast<long long>(seq_id), static_cast<long long>(need_blocks), a->free_q.size());
    auto& s = a->seqs[seq_id];
    for (int64_t i = 0; i < need_blocks; ++i) {
        s.table.push_back(a->free_q.front());
        a->free_q.pop_front();
    }
    s.tokens = total;
    return KV_OK;
}

kv_status_t kv_allocator_release(kv_block_allocator_t* a, int64_t seq_id) {
    if (!a) return fail(KV_ERR_INVALID_ARG, "null allocator");
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return fail(KV_ERR_NOT_FOUND, "unknown sequence %lld", static_cast<long long>(seq_id));
    for (int32_t b : it->second.table) a->free_q.push_back(b);
    a->seqs.erase(it);
    return KV_OK;
}

kv_status_t kv_allocator_table(const kv_block_allocator_t* a, int64_t seq_id, int32_t* table_out,
                               int capacity, int* num_blocks_out, int* num_tokens_out) {
    if (!a || capacity < 0 || (capacity > 0 && !table_out)) return fail(KV_ERR_INVALID_ARG, "kv_allocator_table arguments");
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return fail(KV_ERR_NOT_FOUND, "unknown sequence %lld", static_cast<long long>(seq_id));
    const auto& t = it->second.table;
    if (static_cast<int>(t.size()) > capacity && table_out)
        return fail(KV_ERR_INVALID_ARG, "table of %zu blocks does not fit in %d entries", t.size(), capacity);
    for (size_t i = 0; i < t.size() && table_out; ++i) table_out[i] = t[i];
    if (num_blocks_out) *num_blocks_out = static_cast<int>(t.size());
    if (num_tokens_out) *num_tokens_out = static_cast<int>(it->second.tokens);
    return KV_OK;
}

kv_status_t kv_allocator_slot(const kv_block_allocator_t* a, int64_t seq_id, int position, int32_t* slot_out) {
    if (!a || !slot_out) return fail(KV_ERR_INVALID_ARG, "kv_allocator_slot arguments");
    auto it = a->seqs.find(seq_id);
    if (it == a->seqs.end()) return fail(KV_ERR_NOT_FOUND, "unknown sequence %lld", static_cast<long long>(seq_id));
    const auto& t = it->second.table;
    if (position < 0 || static_cast<int64_t>(position) >= static_cast<int64_t>(t.size()) * a->block_size)
        return fail(KV_ERR_INVALID_ARG, "position %d outside the sequence's blocks", position);
    *slot_out = t[position / a->block_size] * a->block_size + position % a->block_size;
    return KV_OK;
}

kv_status_t kv_seq_extend(kv_pool_t* p, int seq_id, int new_tokens, int32_t* table_row, int max_blocks,
                          int* ctx_len_inout, int32_t* slot_out) {
    if (!p || !table_row || !ctx_len_inout || max_blocks <= 0 || new_tokens < 0 || (new_tokens > 0 && !slot_out))
        return fail(KV_ERR_INVALID_ARG, "kv_seq_extend arguments");
    if (!p->alloc) {
        if (kv_status_t st = kv_allocator_create(p->cfg.num_blocks, p->cfg.block_size, 0, &p->alloc)) return st;
    }
    kv_block_allocator* a = p->alloc;
    auto it = a->seqs.find(seq_id);
    const int64_t have = it == a->seqs.end() ? 0 : it->second.tokens;
    if (*ctx_len_inout != have)
        return fail(KV_ERR_INVALID_ARG, "sequence %d holds %lld tokens, the caller says %d", seq_id,
                    static_cast<long long>(have), *ctx_len_inout);
    const int64_t total = have + new_tokens;
    const int64_t blocks = (total + a->block_size - 1) / a->block_size;
    if (blocks > max_blocks)
        return fail(KV_ERR_INVALID_ARG, "sequence %d would need %lld table entries, %d given", seq_id,
                    static_cast<long long>(blocks), max_blocks);
    if (kv_status_t st = kv_allocator_extend(a, seq_id, new_tokens)) return st;
    const auto& t = a->seqs[seq_id].table;
    for (int i = 0; i < max_blocks; ++i) table_row[i] = i < static_cast<int>(t.size()) ? t[i] : -1;
    for (int i = 0; i < new_tokens; ++i) {
        const int64_t pos = have + i;
        slot_out[i] = t[pos / a->block_size] * a->block_size + static_cast<int32_t>(pos % a->block_size);
    }
    *ctx_len_inout = static_cast<int>(total);
    return KV_OK;
}

kv_status_t kv_seq_free(kv_pool_t* p, int seq_id) {
    if (!p) return fail(KV_ERR_INVALID_ARG, "null pool");
    if (!p->alloc) return fail(KV_ERR_NOT_FOUND, "unknown sequence %d", seq_id);
    return kv_allocator_release(p->alloc, seq_id);
}

kv_status_t kv_allocator_free_queue(const kv_block_allocator_t* a, int32_t* out, int capacity, int* count_out) {
    if (!a || capacity < 0 || (capacity > 0 && !out)) return fail(KV_ERR_INVALID_ARG, "kv_allocator_free_queue arguments");
    const int n = static_cast<int>(a->free_q.size());
    if (count_out) *count_out = n;
    if (out) {
        if (n > capacity) return fail(KV_ERR_INVALID_ARG, "free queue of %d does not fit in %d", n, capacity);
        int i = 0;
        for (int32_t b : a->free_q) out[i++] = b;
    }
    return KV_OK;
}

}  // extern "C"

namespace pkv {
kv_status_t decode_attention_clearing_counters(const void* q, const void* k_cache, const void* v_cache,
                                               int num_blocks, const int32_t* block_tables, int max_blocks,
                                               const int32_t* context_lens, int num_seqs, int num_q_heads,
                                               int num_kv_heads, int head_dim, int block_size, int dtype,
                                               float scale, void* out, int out_dtype, void* workspace,
                                               size_t workspace_bytes, const void* opts, void* stream) {
    const kv_dtype_t dt = static_cast<kv_dtype_t>(dtype);
    return decode_impl(q, k_cache, v_cache, num_blocks, block_tables, max_blocks, context_lens, num_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, dt, scale, out,
                       static_cast<kv_dtype_t>(out_dtype), workspace, workspace_bytes,
                       static_cast<const kv_decode_options_t*>(opts), stream, nullptr, nullptr, nullptr,
                       nullptr, dt, 1.f, 1.f, /*clear_counters=*/true);
}
}  // namespace pkv
