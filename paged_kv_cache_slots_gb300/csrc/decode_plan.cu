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
// and are skipped.  Parts are taken 32 at a time: warp 0 reads their (max,
// sum) pairs, one part a lane, and folds them into each head's running max
// and sum, leaving the parts' weights in shared memory; then every thread
// rescales its outputs and adds the parts' outputs, several loads in flight.
__global__ void __launch_bounds__(128) paged_decode_reduce_kernel(const DecodeArgs a) {
    constexpr int kChunk = 32, kMaxG = 8, kPer = kMaxG * 128 / 128;  // outputs a thread, G*D <= 1024
    __shared__ float wgt[kChunk][kMaxG];  // exp2(m - M) of (part, head) in the current chunk
    __shared__ float rescale[kMaxG];      // exp2(M_old - M) of each head for this chunk
    __shared__ float run_m[kMaxG], run_l[kMaxG];
    pdl_allow_next();
    pdl_wait();
    const int sh = blockIdx.x;
    const int s = sh / a.num_kv_heads;
    const int h = sh - s * a.num_kv_heads;
    const int G = a.num_q_heads / a.num_kv_heads;
    const int D = a.head_dim, Hc = a.heads_per_stage;
    const int chunks = a.num_kv_heads / Hc;
    const int hc = h / Hc, hw = h - hc * Hc;
    const int nbv = (a.cum[s + 1] - a.cum[s]) / chunks;  // the pair's items, phantoms first
    const int nb = nbv > 0 ? nbv - a.phantom : 0;       // its blocks
    const int64_t out0 = (static_cast<int64_t>(s) * a.num_q_heads + h * G) * D;
    const int tid = threadIdx.x;
    if (nb == 0) {
        for (int idx = tid; idx < G * D; idx += blockDim.x) store_out(a.out, out0 + idx, 0.f, a.out_dtype);
        return;
    }
    const int64_t W = a.cum[a.num_seqs];
    const int64_t P = a.num_ctas;
    const int64_t pa = a.cum[s] + static_cast<int64_t>(hc) * nbv + a.phantom;  // its first block
    const int ca = cta_of_item(pa, W, a.num_ctas);
    const int cb = cta_of_item(pa + nb - 1, W, a.num_ctas);
    if (ca == cb) return;
    const int pair = s * chunks + hc;
    if (tid < kMaxG) {
        run_m[tid] = -INFINITY;
        run_l[tid] = 0.f;
    }
    float acc[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) acc[k] = 0.f;
    for (int c0 = ca; c0 <= cb; c0 += kChunk) {
        __syncthreads();  // the previous chunk's weights are used up
        if (tid < 32) {
            const int c = c0 + tid;
            const bool valid = c <= cb && !cta_is_empty(c, W, P);
            const int64_t sl = ((static_cast<int64_t>(c) + pair) * Hc + hw) * G;
            for (int g = 0; g < G; ++g) {
                float m = -INFINITY, l = 0.f;
                if (valid) {
                    const float2 ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml + (sl + g) * 2));
                    m = ml.x;
                    l = ml.y;
                }
                float mx = m;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
                const float m_old = run_m[g];
                const float m_new = fmaxf(m_old, mx);
                const float w = valid ? fast_exp2(m - m_new) : 0.f;
                wgt[tid][g] = w;
                float ls = w * l;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) ls += __shfl_xor_sync(0xffffffffu, ls, o);
                __syncwarp();
                if (tid == 0) {
                    const float al = m_old == -INFINITY ? 0.f : fast_exp2(m_old - m_new);
                    rescale[g] = al;
                    run_l[g] = run_l[g] * al + ls;
                    run_m[g] = m_new;
                }
                __syncwarp();
            }
        }
        __syncthreads();
        const int nc = min(kChunk, cb - c0 + 1);
#pragma unroll
        for (int k = 0; k < kPer; ++k) {
            const int idx = tid + 128 * k;
            if (idx < G * D) acc[k] *= rescale[idx / D];
        }
#pragma unroll 4
        for (int j = 0; j < nc; ++j) {
            const int64_t base = ((static_cast<int64_t>(c0 + j) + pair) * Hc + hw) * G * D;
#pragma unroll
            for (int k = 0; k < kPer; ++k) {
                const int idx = tid + 128 * k;
                if (idx >= G * D) continue;
                const float w = wgt[j][idx / D];
                if (w != 0.f) acc[k] += w * __ldcg(a.part_o + base + idx);  // empty parts hold no data
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
        const int idx = tid + 128 * k;
        if (idx < G * D) store_out(a.out, out0 + idx, acc[k] / run_l[idx / D], a.out_dtype);
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
