// Swap of whole KV blocks between the pool and host memory ("Batching and
// Scheduling", Example 8: preemption by swap copies a request's KV entries to
// CPU memory and back instead of computing them again).
//
// A swapped block is every layer's K and V rows of one physical block; in
// the host buffer block i of the list occupies one contiguous record of
// 2 * num_layers units, unit j = 2 * layer + (0 for K, 1 for V), each unit the
// block's [Hkv][bs][D] rows as laid out in the pool.  In the pool unit j of
// block b starts at base + j * layer_bytes + b * unit_bytes, in the host
// record at host + (i * 2 * num_layers + j) * unit_bytes.
//
// The host buffer is page-locked memory that the GPU addresses directly
// (over NVLink-C2C on Grace systems, PCIe elsewhere), so one kernel moves
// the data with no staging copy in device memory: each CTA moves units of
// unit_bytes as 16-byte vectors, several loads in flight per thread before
// the stores, to cover the link's latency.
#include "device_utils.cuh"

namespace pkv {

namespace {

constexpr int kSwapThreads = 256;
constexpr int kSwapUnroll = 4;

__global__ void __launch_bounds__(kSwapThreads) kv_swap_kernel(const SwapArgs a) {
    pdl_allow_next();
    pdl_wait();
    const int64_t units = static_cast<int64_t>(a.n) * 2 * a.num_layers;
    const int64_t nvec = a.unit_bytes >> 4;
    for (int64_t u = blockIdx.x; u < units; u += gridDim.x) {
        const int64_t i = u / (2 * a.num_layers);
        const int64_t j = u - i * 2 * a.num_layers;
        const int32_t b = a.block_ids[i];
        if (b < 0 || b >= a.num_blocks) {
            if (threadIdx.x == 0 && j == 0) raise_flag(a.status, kFlagBadBlock);
            continue;
        }
        char* dev = a.pool + j * a.layer_bytes + static_cast<int64_t>(b) * a.unit_bytes;
        char* host = a.host + u * a.unit_bytes;
        const uint4* src = reinterpret_cast<const uint4*>(a.to_host ? dev : host);
        uint4* dst = reinterpret_cast<uint4*>(a.to_host ? host : dev);
        for (int64_t v0 = threadIdx.x; v0 < nvec; v0 += kSwapThreads * kSwapUnroll) {
            uint4 r[kSwapUnroll];
#pragma unroll
            for (int k = 0; k < kSwapUnroll; ++k) {
                const int64_t v = v0 + k * kSwapThreads;
                if (v < nvec) r[k] = __ldcs(src + v);
            }
#pragma unroll
            for (int k = 0; k < kSwapUnroll; ++k) {
                const int64_t v = v0 + k * kSwapThreads;
                if (v < nvec) __stcs(dst + v, r[k]);
            }
        }
    }
}

}  // namespace

cudaError_t launch_swap(const SwapArgs& a, int num_sms, cudaStream_t stream) {
    const int64_t units = static_cast<int64_t>(a.n) * 2 * a.num_layers;
    if (units == 0) return cudaSuccess;
    // Eight resident CTAs per SM keep enough 16-byte loads in flight; more
    // units than that are taken in a grid-stride loop.
    const int64_t cap = static_cast<int64_t>(num_sms > 0 ? num_sms : 1) * 8;
    const unsigned grid = static_cast<unsigned>(units < cap ? units : cap);
    return launch_kernel(kv_swap_kernel, dim3(grid), dim3(kSwapThreads), 0, stream, a.pdl != 0, a);
}

}  // namespace pkv
