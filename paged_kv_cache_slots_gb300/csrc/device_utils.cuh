// Device helpers: mbarriers, bulk/tensor async copies (TMA), warp-level
// tensor-core fragments, fast base-2 exponent, status flags.  Inline PTX
// written for sm_103a.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include <utility>

#include "pkv_internal.h"

namespace pkv {

// Status bits (same values as KV_FLAG_* in pkv.h).
constexpr uint32_t kFlagBadBlock = 0x1u;
constexpr uint32_t kFlagBadSlot = 0x2u;
constexpr uint32_t kFlagBadContext = 0x4u;
constexpr uint32_t kFlagTimeout = 0x8u;
constexpr uint32_t kFlagBadPlan = 0x10u;

// A bounded wait gives up after this many nanoseconds of the global timer.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

__device__ __forceinline__ void raise_flag(uint32_t* status, uint32_t bit) {
    if (status) atomicOr(status, bit);
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
                     smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return done != 0;
}

// As mbar_try_wait, but the thread may sleep up to `hint_ns` waiting for the
// phase (it resumes as soon as the phase completes), so a wait does not keep
// issuing polls that the other warps of its scheduler could have used.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return done != 0;
}

// Wait for phase `parity` of `bar` to complete.  Gives up (returns false and
// raises the timeout flag) after kWaitLimitNs, or at once if *abort is set
// (checked at least every 10 us).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort, uint32_t* status) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = global_timer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 10000u)) return true;
        if (*abort) return false;
        if (global_timer_ns() - t0 > kWaitLimitNs) {
            *abort = 1;
            raise_flag(status, kFlagTimeout);
            return false;
        }
    }
}

// ------------------------------------------------------- async bulk copies
// Order this thread's earlier generic-proxy shared-memory accesses before
// later async-proxy (TMA) accesses to the same memory.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Contiguous global -> shared copy completed on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).  L2 evict-first: every tile is read once.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                          uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// Bring `bytes` of global memory into L2 (bytes % 16 == 0, 16-byte aligned
// address); no completion, a hint only.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}

// 2-D tiled tensor copy (box given by the tensor map) completed on `bar`.
__device__ __forceinline__ void tensor_load_2d(void* dst, const CUtensorMap* map, int x, int y,
                                               uint64_t* bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

__device__ __forceinline__ void prefetch_tensor_map(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// L2 evict-last: tiles that other CTAs read again soon (prefill tiles).
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ------------------------------------------- programmatic dependent launch
// Wait until the grid this launch depends on has completed and its memory
// is visible (a no-op when the launch has no programmatic dependency).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Allow the next launch in the stream to start being scheduled now; it still
// waits in pdl_wait() for this grid to complete before touching memory.
__device__ __forceinline__ void pdl_allow_next() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// L2-coherent load (bypasses L1): for data other CTAs wrote in this launch.
__device__ __forceinline__ float load_cg(const float* p) { return __ldcg(p); }

// 16 bytes global -> shared through L2 only (cp.async.cg), completed by
// cp_async_wait_all() in the same thread.
__device__ __forceinline__ void cp_async_16(uint32_t dst_smem, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst_smem), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() {
    asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

// ----------------------------------------------------------- named barrier
__device__ __forceinline__ void named_barrier_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// --------------------------------------------------------------- math
// 2^x on the special-function unit (PTX ex2.approx.ftz.f32; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------- element load / convert
template <int DT>
struct Elem;
template <>
struct Elem<kF32> {
    using T = float;
    static __device__ __forceinline__ float to_float(T x) { return x; }
    static __device__ __forceinline__ T from_float(float x) { return x; }
};
template <>
struct Elem<kF16> {
    using T = __half;
    static __device__ __forceinline__ float to_float(T x) { return __half2float(x); }
    static __device__ __forceinline__ T from_float(float x) { return __float2half_rn(x); }
};
template <>
struct Elem<kBF16> {
    using T = __nv_bfloat16;
    static __device__ __forceinline__ float to_float(T x) { return __bfloat162float(x); }
    static __device__ __forceinline__ T from_float(float x) { return __float2bfloat16_rn(x); }
};

// ------------------------------------------------------------------- E4M3
// A cached E4M3 byte b stands for scale * e4m3(b); a value x is stored as the
// E4M3 code nearest to the fp32 quotient x / scale (round to nearest even,
// saturating at +-448, the conversion instruction's satfinite mode).

// Loads element i of a row of src_dtype (f32, f16 or bf16) as fp32.
__device__ __forceinline__ float load_as_float(const void* row, int i, int src_dtype) {
    if (src_dtype == kF32) return static_cast<const float*>(row)[i];
    if (src_dtype == kF16) return __half2float(static_cast<const __half*>(row)[i]);
    return __bfloat162float(static_cast<const __nv_bfloat16*>(row)[i]);
}

// Two fp32 values -> two E4M3 codes (x0 in the low byte).
__device__ __forceinline__ uint16_t e4m3x2_from_floats(float x0, float x1) {
    return static_cast<uint16_t>(
        __nv_cvt_float2_to_fp8x2(make_float2(x0, x1), __NV_SATFINITE, __NV_E4M3));
}

// Codes of elements 16q .. 16q+15 of a source row (src_dtype), each divided
// by `scale` in fp32 first: one 16-byte chunk of a quantized row.
__device__ __forceinline__ uint4 quantize_chunk16(const void* row, int q, int src_dtype, float scale) {
    uint32_t w[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        const int i = 16 * q + 4 * k;
        const uint16_t lo = e4m3x2_from_floats(__fdiv_rn(load_as_float(row, i, src_dtype), scale),
                                               __fdiv_rn(load_as_float(row, i + 1, src_dtype), scale));
        const uint16_t hi = e4m3x2_from_floats(__fdiv_rn(load_as_float(row, i + 2, src_dtype), scale),
                                               __fdiv_rn(load_as_float(row, i + 3, src_dtype), scale));
        w[k] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
    }
    return make_uint4(w[0], w[1], w[2], w[3]);
}

// Two E4M3 codes (low byte first) -> f16x2 (exact: every E4M3 value is an f16).
__device__ __forceinline__ uint32_t e4m3x2_to_half2(uint16_t v) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
    return static_cast<uint32_t>(h.x) | (static_cast<uint32_t>(h.y) << 16);
}

// E4M3 -> f16 in integer operations, exactly, times 2^-8: an E4M3 code
// s.eeee.mmm read as the f16 bit pattern s.0eeee.mmm0000000 has exponent
// field eeee, i.e. the same value scaled by 2^(7 - 15), subnormals included.
// Two codes of a 32-bit word are converted at once, each into one 16-bit
// half of the result.
//
// Codes in bytes 1 and 3 of r (bytes 0 and 2 ignored): each code's sign
// already sits at bit 15 of its half, and its seven magnitude bits move down
// one place to bits 13..7 -- one shift and one three-input logic operation.
__device__ __forceinline__ uint32_t e4m3x2_odd_bytes_to_half2_shifted(uint32_t r) {
    return ((r >> 1) & 0x3F803F80u) | (r & 0x80008000u);
}

// Codes in bytes 0 and 2 of r (bytes 1 and 3 ignored): moved up one byte
// first, then as above.
__device__ __forceinline__ uint32_t e4m3x2_even_bytes_to_half2_shifted(uint32_t r) {
    return e4m3x2_odd_bytes_to_half2_shifted(r << 8);
}

// Store an fp32 value as out_dtype (round to nearest even).
__device__ __forceinline__ void store_out(void* out, int64_t idx, float v, int out_dtype) {
    if (out_dtype == kF32)
        static_cast<float*>(out)[idx] = v;
    else if (out_dtype == kF16)
        static_cast<__half*>(out)[idx] = __float2half_rn(v);
    else
        static_cast<__nv_bfloat16*>(out)[idx] = __float2bfloat16_rn(v);
}

// Launch `kernel` on `stream`, optionally as a programmatic dependent of the
// previous launch in the stream (its prologue may overlap that launch's tail).
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t stream, bool pdl, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace pkv
