// Shared-memory planning of the decode kernels, the cross-CTA reduce kernel
// and the per-device status word.
#include "decode_kernel.cuh"

namespace pkv {

// One status word per device (each device holds its own copy of this
// variable once the library's module is loaded there).  Kernels OR flag bits
// into it; the host reads and clears it with kv_device_status.
__device__ uint32_t g_status_word;

cudaError_t status_word_address(uint32_t** ptr) {
    return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_status_word);
}

bool decode_plan(int kernel, int dtype, int head_dim, int block_size, int group, int num_seqs,
                 int heads_per_stage, int warps_per_head, int smem_budget, DecodePlan* plan) {
    const int half = heads_per_stage * block_size * head_dim * dtype_bytes(dtype);
    const bool scratch = (kernel == 1);  // the FFMA consumer keeps per-warp score rows
    const int nc = heads_per_stage * warps_per_head;
    const SmemLayout fixed = smem_layout(0, half, num_seqs, nc, warps_per_head, group, head_dim,
                                         block_size, scratch);
    const int per_stage = 2 * half + 16;  // K + V, two mbarriers
    int stages = (smem_budget - fixed.total) / per_stage;
    if (stages > kMaxStages) stages = kMaxStages;
    // With R warps per head taking items round-robin, a stage must always be
    // reused by the same replica: item t and item t - stages then belong to
    // one warp, which waited for the older phase before it waits for the
    // newer one.  Otherwise a warp could test the parity of a stage whose
    // previous fill (another replica's item) has not completed yet, and the
    // two phases would alias.
    stages -= stages % warps_per_head;
    if (stages < 2 || stages < warps_per_head) return false;
    const SmemLayout L = smem_layout(stages, half, num_seqs, nc, warps_per_head, group, head_dim,
                                     block_size, scratch);
    if (L.total > smem_budget) return false;
    plan->stages = stages;
    plan->smem_bytes = L.total;
    plan->stage_half_bytes = half;
    return true;
}

// ------------------------------------------------------------------ reduce
// One CTA per (sequence, KV head): merge the partials of a pair split over
// several CTAs (log-sum-exp in base 2), zero the rows of an empty sequence,
// skip pairs the partial kernel finished itself.  CTAs between the first and
// last owner whose item range is empty (more CTAs than items) wrote nothing
// and are skipped.
__global__ void __launch_bounds__(128) paged_decode_reduce_kernel(const DecodeArgs a) {
    pdl_allow_next();
    pdl_wait();
    const int sh = blockIdx.x;
    const int s = sh / a.num_kv_heads;
    const int h = sh - s * a.num_kv_heads;
    const int G = a.num_q_heads / a.num_kv_heads;
    const int D = a.head_dim, Hc = a.heads_per_stage;
    const int chunks = a.num_kv_heads / Hc;
    const int hc = h / Hc, hw = h - hc * Hc;
    const int nb = (a.cum[s + 1] - a.cum[s]) / chunks;
    const int64_t out0 = (static_cast<int64_t>(s) * a.num_q_heads + h * G) * D;
    if (nb == 0) {
        for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) store_out(a.out, out0 + idx, 0.f, a.out_dtype);
        return;
    }
    const int64_t W = a.cum[a.num_seqs];
    const int64_t P = a.num_ctas;
    const int64_t pa = a.cum[s] + static_cast<int64_t>(hc) * nb;
    const int ca = cta_of_item(pa, W, a.num_ctas);
    const int cb = cta_of_item(pa + nb - 1, W, a.num_ctas);
    if (ca == cb) return;
    const int pair = s * chunks + hc;
    for (int idx = threadIdx.x; idx < G * D; idx += blockDim.x) {
        const int g = idx / D, d = idx - g * D;
        float M = -INFINITY;
        for (int c = ca; c <= cb; ++c) {
            if (cta_is_empty(c, W, P)) continue;
            M = fmaxf(M, a.part_ml[(((static_cast<int64_t>(c) + pair) * Hc + hw) * G + g) * 2]);
        }
        float Lsum = 0.f, O = 0.f;
        for (int c = ca; c <= cb; ++c) {
            if (cta_is_empty(c, W, P)) continue;
            const int64_t sl = ((static_cast<int64_t>(c) + pair) * Hc + hw) * G + g;
            const float wgt = fast_exp2(a.part_ml[sl * 2] - M);
            Lsum += wgt * a.part_ml[sl * 2 + 1];
            O += wgt * a.part_o[sl * D + d];
        }
        store_out(a.out, out0 + idx, O / Lsum, a.out_dtype);
    }
}

cudaError_t launch_decode_reduce(const DecodeArgs& a, cudaStream_t stream) {
    const int n = a.num_seqs * a.num_kv_heads;
    if (n == 0) return cudaSuccess;
    return launch_kernel(paged_decode_reduce_kernel, dim3(n), dim3(128), 0, stream, a.pdl != 0, a);
}

int max_dynamic_smem(int device) {
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, device) != cudaSuccess)
        return 0;
    return v;
}

}  // namespace pkv
