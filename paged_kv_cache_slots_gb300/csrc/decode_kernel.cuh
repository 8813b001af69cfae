// Split-context decode attention over a paged KV cache (persistent kernel).
//
// What is computed ("vLLM Architecture and Installation", Example 3;
// "Batching and Scheduling", Example 1): for every sequence s and query head
// g, softmax over the sequence's cached tokens of scale * q.k, applied to V,
// with K/V read through the block table.  Query heads h*G .. h*G+G-1 share KV
// head h, and one CTA reads each (block, kv head) tile from HBM once for the
// whole group.
//
// Work split.  The work space is every (sequence, kv head, logical block)
// triple, in that order; W = sum_s Hkv * ceil(ctx_s / bs) tiles.  CTA c of P
// owns tiles [c*W/P, (c+1)*W/P): the load is balanced to one tile whatever
// the length mix.  A run of tiles of one (sequence, kv head) pair inside one
// CTA is a segment.  A segment that covers its whole pair writes the final
// output; otherwise it writes an fp32 partial (unnormalised O, running max,
// running sum) to partial slot c + pair, which is unique because segments
// sorted by position increase c + pair by at least one each step.  The
// reduce kernel merges the partials of each split pair.
//
// Inside a CTA, warp 0 is the producer: it reads table entries 32 at a time
// and streams each tile's K and V into a ring of shared-memory stages with
// asynchronous bulk copies completing on mbarriers.  The other warps consume
// tiles round-robin, each keeping an online-softmax state (scores in base-2
// units) for the current segment, and merge their states through shared
// memory at the end of the segment.
#pragma once

#include <atomic>

#include "device_utils.cuh"

namespace pkv {

constexpr int kMaxStages = 32;

struct SmemLayout {
    int ring, full_bar, empty_bar, flags, scan, cum, merge, scratch, total;
};

// Offsets from a 1024-byte aligned base; `total` includes the alignment slack.
__host__ __device__ inline SmemLayout smem_layout(int stages, int tile_bytes, int num_seqs,
                                                  int consumer_warps, int group, int head_dim,
                                                  int block_size, bool scratch) {
    SmemLayout L;
    int o = 0;
    L.ring = o;
    o += stages * 2 * tile_bytes;
    L.full_bar = o;
    o += stages * 8;
    L.empty_bar = o;
    o += stages * 8;
    L.flags = o;
    o += 16;
    L.scan = o;
    o += 32 * 4;
    L.cum = o;
    o += ((num_seqs + 1) * 4 + 15) & ~15;
    L.merge = o;
    o += consumer_warps * group * (head_dim + 2) * 4;
    L.scratch = o;
    if (scratch) o += consumer_warps * ((block_size * group * 4 + 15) & ~15);
    L.total = o + 1024;
    return L;
}

// Tile index -> CTA that owns it: the c with floor(c*W/P) <= x < floor((c+1)*W/P).
__host__ __device__ inline int cta_of_tile(int64_t x, int64_t W, int P) {
    return static_cast<int>(((x + 1) * P - 1) / W);
}

// Largest s in [0, n) with cum[s] <= i (cum non-decreasing, cum[0] == 0).
__device__ __forceinline__ int find_sequence(const int32_t* cum, int n, int i) {
    int lo = 0, hi = n;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (cum[mid] <= i)
            lo = mid;
        else
            hi = mid;
    }
    return lo;
}

__device__ __forceinline__ int clamp_context(const DecodeArgs& a, int s, bool flag) {
    int c = a.context_lens[s];
    const int cap = a.max_blocks * a.block_size;
    if (c < 0 || c > cap) {
        if (flag) raise_flag(a.status, kFlagBadContext);
        c = c < 0 ? 0 : cap;
    }
    return c;
}

// cum[s] = Hkv * sum_{s' < s} ceil(ctx_s' / bs); cum[num_seqs] = W.
static __device__ void build_prefix(const DecodeArgs& a, int32_t* cum, int32_t* scan) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    int carry = 0;
    for (int base = 0; base < a.num_seqs; base += blockDim.x) {
        const int s = base + tid;
        int v = 0;
        if (s < a.num_seqs) {
            const int c = clamp_context(a, s, blockIdx.x == 0);
            v = (c + a.block_size - 1) / a.block_size * a.num_kv_heads;
        }
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) scan[wid] = x;
        __syncthreads();
        if (wid == 0) {
            int t = lane < nwarps ? scan[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            scan[lane] = t;  // inclusive prefix of warp totals
        }
        __syncthreads();
        const int warp_off = wid > 0 ? scan[wid - 1] : 0;
        if (s < a.num_seqs) cum[s] = carry + warp_off + x - v;
        carry += scan[nwarps - 1];
        __syncthreads();
    }
    if (tid == 0) cum[a.num_seqs] = carry;
    __syncthreads();
}

// ------------------------------------------------------------------ producer
// kTensor: tiles arrive through 2-D tensor maps with a 128-byte swizzle (box
// of 64 elements x block_size rows, one box per 64-element half of the row);
// otherwise as plain contiguous bulk copies.
template <bool kTensor>
__device__ void produce(const DecodeArgs& a, uint8_t* ring, uint64_t* full, uint64_t* empty,
                        const int32_t* cum, int start, int end, int tile_bytes,
                        const CUtensorMap* tmk, const CUtensorMap* tmv, volatile int* abort) {
    const int lane = threadIdx.x & 31;
    const uint64_t policy = policy_evict_first();
    const int stage_bytes = 2 * tile_bytes;
    const int64_t row_elems = a.head_dim;
    const int eb = dtype_bytes(a.dtype);
    int issued = 0;  // tiles whose copies were issued (lane 0)
    bool ok = true;
    for (int base = start; base < end && ok; base += 32) {
        const int i = base + lane;
        int64_t row = 0;  // first pool row of the tile: (blk * Hkv + h) * bs
        if (i < end) {
            const int s = find_sequence(cum, a.num_seqs, i);
            const int nb = (cum[s + 1] - cum[s]) / a.num_kv_heads;
            const int r = i - cum[s];
            const int h = r / nb;
            const int j = r - h * nb;
            int blk = __ldg(a.block_tables + static_cast<int64_t>(s) * a.max_blocks + j);
            if (blk < 0 || blk >= a.num_blocks) {
                raise_flag(a.status, kFlagBadBlock);
                blk = 0;
            }
            row = (static_cast<int64_t>(blk) * a.num_kv_heads + h) * a.block_size;
        }
        const int n = min(32, end - base);
        for (int k = 0; k < n; ++k) {
            const int64_t rk = __shfl_sync(0xffffffffu, row, k);
            int good = 1;
            if (lane == 0) {
                const int t = base + k - start;
                const int stage = t % a.stages;
                const int round = t / a.stages;
                // Test-only stall: CTA 0 stops after its first tile, so that a
                // consumer's bounded wait for the second one runs out.
                if (a.test_stall && blockIdx.x == 0 && t == 1) good = 0;
                if (good && round > 0)
                    good = mbar_wait_bounded(&empty[stage], (round - 1) & 1, abort, a.status);
                if (good) {
                    uint8_t* kd = ring + stage * stage_bytes;
                    uint8_t* vd = kd + tile_bytes;
                    mbar_arrive_expect_tx(&full[stage], stage_bytes);
                    if constexpr (kTensor) {
                        const int halves = a.head_dim / 64;
                        const int half_bytes = tile_bytes / halves;
                        for (int hf = 0; hf < halves; ++hf) {
                            tensor_load_2d(kd + hf * half_bytes, tmk, hf * 64, static_cast<int>(rk),
                                           &full[stage], policy);
                            tensor_load_2d(vd + hf * half_bytes, tmv, hf * 64, static_cast<int>(rk),
                                           &full[stage], policy);
                        }
                    } else {
                        const int64_t off = rk * row_elems * eb;
                        bulk_load(kd, static_cast<const char*>(a.k_cache) + off, tile_bytes,
                                  &full[stage], policy);
                        bulk_load(vd, static_cast<const char*>(a.v_cache) + off, tile_bytes,
                                  &full[stage], policy);
                    }
                    ++issued;
                }
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) {
                ok = false;
                break;
            }
        }
    }
    // Wait (bounded) until every copy this producer issued has landed, so
    // that no copy outlives the CTA's shared memory, whatever the consumers did.
    if (lane == 0) {
        for (int st = 0; st < a.stages && st < issued; ++st) {
            const int last = st + ((issued - 1 - st) / a.stages) * a.stages;
            const uint32_t parity = (last / a.stages) & 1;
            const uint64_t t0 = global_timer_ns();
            while (!mbar_try_wait(&full[st], parity)) {
                if (global_timer_ns() - t0 > kWaitLimitNs) {
                    raise_flag(a.status, kFlagTimeout);
                    break;
                }
            }
        }
    }
    __syncwarp();
}

// ---------------------------------------------------------------- the kernel
// Policy provides: State, begin(), tile(), publish(), kTensor, kScratch.
template <class Policy>
__global__ void __launch_bounds__(32 * 16, 1)
    paged_decode_partial_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                                const __grid_constant__ CUtensorMap tmv) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int G = a.num_q_heads / a.num_kv_heads;
    const int tile_bytes = a.block_size * a.head_dim * dtype_bytes(a.dtype);
    const SmemLayout L = smem_layout(a.stages, tile_bytes, a.num_seqs, a.consumer_warps, G,
                                     a.head_dim, a.block_size, Policy::kScratch);
    uint8_t* ring = base + L.ring;
    uint64_t* full = reinterpret_cast<uint64_t*>(base + L.full_bar);
    uint64_t* empty = reinterpret_cast<uint64_t*>(base + L.empty_bar);
    volatile int* abort = reinterpret_cast<volatile int*>(base + L.flags);
    int32_t* scan = reinterpret_cast<int32_t*>(base + L.scan);
    int32_t* cum = reinterpret_cast<int32_t*>(base + L.cum);
    float* merge = reinterpret_cast<float*>(base + L.merge);

    const int tid = threadIdx.x;
    if (tid == 0) {
        for (int st = 0; st < a.stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], 1);
        }
        *abort = 0;
        fence_barrier_init();
    }
    if constexpr (Policy::kTensor) {
        if (tid == 0) {
            prefetch_tensor_map(&tmk);
            prefetch_tensor_map(&tmv);
        }
    }
    build_prefix(a, cum, scan);  // ends with __syncthreads
    if (blockIdx.x == 0) {
        for (int s = tid; s <= a.num_seqs; s += blockDim.x) a.cum[s] = cum[s];
    }
    const int64_t W = cum[a.num_seqs];
    const int P = a.num_ctas;
    const int start = static_cast<int>(static_cast<int64_t>(blockIdx.x) * W / P);
    const int end = static_cast<int>((static_cast<int64_t>(blockIdx.x) + 1) * W / P);
    if (start >= end) return;

    const int warp = tid >> 5, lane = tid & 31;
    if (warp == 0) {
        produce<Policy::kTensor>(a, ring, full, empty, cum, start, end, tile_bytes, &tmk, &tmv,
                                 abort);
        return;
    }
    const int w = warp - 1;
    const int NC = a.consumer_warps;
    float* scratch = Policy::kScratch
                         ? reinterpret_cast<float*>(base + L.scratch) +
                               w * ((a.block_size * G * 4 + 15) & ~15) / 4
                         : nullptr;
    Policy pol;
    typename Policy::State st;
    int seg = start;
    while (seg < end) {
        const int s = find_sequence(cum, a.num_seqs, seg);
        const int nb = (cum[s + 1] - cum[s]) / a.num_kv_heads;
        const int h = (seg - cum[s]) / nb;
        const int pair_a = cum[s] + h * nb;
        const int pair_b = pair_a + nb;
        const int seg_end = min(pair_b, end);
        const int ctx = clamp_context(a, s, false);
        pol.begin(st, a, s, h, G);
        int first = seg + (((w - (seg - start)) % NC) + NC) % NC;
        for (int i = first; i < seg_end; i += NC) {
            const int t = i - start;
            const int stage = t % a.stages;
            const bool ok = mbar_wait_bounded(&full[stage], (t / a.stages) & 1, abort, a.status);
            if (ok) {
                const int j = i - pair_a;
                const int n_valid = min(a.block_size, ctx - j * a.block_size);
                uint8_t* kt = ring + stage * 2 * tile_bytes;
                pol.tile(st, a, kt, kt + tile_bytes, n_valid, G, scratch);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
        }
        // Merge the consumer warps' states for this segment.
        float* mw = merge + w * G * (a.head_dim + 2);
        pol.publish(st, a, mw, G);
        named_barrier_sync(1, NC * 32);
        const bool whole = (pair_a >= start) && (pair_b <= end);
        const int pair = s * a.num_kv_heads + h;
        const int slot = blockIdx.x + pair;
        const int D = a.head_dim;
        if (!*abort) {
            for (int idx = (w << 5) + lane; idx < G * D; idx += NC * 32) {
                const int g = idx / D, d = idx - g * D;
                float M = -INFINITY;
                for (int u = 0; u < NC; ++u) M = fmaxf(M, merge[(u * G + g) * (D + 2) + D]);
                float Lsum = 0.f, O = 0.f;
                for (int u = 0; u < NC; ++u) {
                    const float* mu = merge + (u * G + g) * (D + 2);
                    const float wgt = fast_exp2(mu[D] - M);
                    Lsum += wgt * mu[D + 1];
                    O += wgt * mu[d];
                }
                if (whole) {
                    const int64_t oi = (static_cast<int64_t>(s) * a.num_q_heads + h * G + g) * D + d;
                    store_out(a.out, oi, O / Lsum, a.out_dtype);
                } else {
                    a.part_o[(static_cast<int64_t>(slot) * G + g) * D + d] = O;
                    if (d == 0) {
                        a.part_ml[(static_cast<int64_t>(slot) * G + g) * 2 + 0] = M;
                        a.part_ml[(static_cast<int64_t>(slot) * G + g) * 2 + 1] = Lsum;
                    }
                }
            }
        }
        named_barrier_sync(1, NC * 32);
        seg = seg_end;
    }
}

// Launch the partial kernel of `Policy`.  The dynamic shared-memory limit is
// raised once per device (not on every launch, so that launches captured in
// a CUDA graph make no attribute calls).
template <class Policy>
cudaError_t launch_partial(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                           cudaStream_t stream) {
    static std::atomic<int> configured[64];
    auto kern = paged_decode_partial_kernel<Policy>;
    const bool cacheable = a.device >= 0 && a.device < 64;
    if (!cacheable || configured[a.device].load() < a.smem_bytes) {
        cudaError_t e =
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, a.smem_bytes);
        if (e != cudaSuccess) return e;
        if (cacheable) configured[a.device].store(a.smem_bytes);
    }
    kern<<<a.num_ctas, 32 * (1 + a.consumer_warps), a.smem_bytes, stream>>>(a, tmk, tmv);
    return cudaGetLastError();
}

}  // namespace pkv
