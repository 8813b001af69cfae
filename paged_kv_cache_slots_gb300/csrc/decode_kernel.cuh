// Split-context decode attention over a paged KV cache (persistent kernel).
//
// What is computed ("vLLM Architecture and Installation", Example 3;
// "Batching and Scheduling", Example 1): for every sequence s and query head
// g, softmax over the sequence's cached tokens of scale * q.k, applied to V,
// with K/V read through the block table.  Query heads h*G .. h*G+G-1 share KV
// head h, and each (block, KV head) tile is read from HBM once for the whole
// group.
//
// Work split.  A work item is (sequence, head chunk, logical block), where a
// head chunk is Hc consecutive KV heads: their K rows of one block are
// contiguous in the pool ([block][head][token][dim]), so an item is one
// pipeline stage filled by two contiguous copies (K, V) of Hc*bs*D elements.
// Items are ordered sequence-major, and every (sequence, head chunk) pair
// starts with `phantom` items without data (a stage the producer completes
// without a copy, skipped by the consumers), so that a CTA whose range
// crosses into a pair -- and pays for the switch: a partial's stores, the
// merge arrival's fence, the next q -- takes that many fewer blocks.
// W = chunks * sum_s (ceil(ctx_s / bs) + phantom) over the sequences with
// tokens.  CTA c of P owns items [c*W/P, (c+1)*W/P): every CTA streams the
// same number of items (to within one) whatever the length mix.  The run of one (sequence,
// head chunk) pair inside one CTA is a segment.  A segment covering its whole
// pair writes the final output; otherwise it writes fp32 partials
// (unnormalised O, running max, running sum) to slot c + pair, unique because
// segments sorted by position increase c + pair by at least one each step.
// The partials of a split pair are merged (log-sum-exp, base 2) either by the
// last warp to finish that (sequence, head) -- it counts arrivals on a
// per-(sequence, head) counter that it resets to zero -- or by the separate
// reduce kernel.
//
// Inside a CTA, warp 0 produces: it resolves table entries 32 items at a time
// and issues each item's two copies into a ring of shared-memory stages,
// completing on mbarrier transaction counts.  Consumer warp w works on head
// w % Hc of every chunk; R = consumer_warps / Hc warps per head take that
// head's items round-robin and merge their states through shared memory at
// the end of a segment (no merge when R == 1).
#pragma once

#include <atomic>

#include "device_utils.cuh"

namespace pkv {

constexpr int kMaxStages = 32;
constexpr int kPrefetchItems = 8;       // items past the first ring fill brought into L2 early
constexpr int kPrefetchMinItems = 128;  // ... when the CTA's range has at least this many

struct SmemLayout {
    int ring, full_bar, empty_bar, flags, scan, cum, merge, scratch, total;
};

// Offsets from a 1024-byte aligned base; `total` includes the alignment slack.
__host__ __device__ inline SmemLayout smem_layout(int stages, int stage_half_bytes, int num_seqs,
                                                  int consumer_warps, int warps_per_head, int group,
                                                  int head_dim, int block_size, bool scratch) {
    SmemLayout L;
    int o = 0;
    L.ring = o;
    o += stages * 2 * stage_half_bytes;
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
    if (warps_per_head > 1) o += consumer_warps * group * (head_dim + 2) * 4;
    L.scratch = o;
    if (scratch) o += consumer_warps * ((block_size * group * 4 + 15) & ~15);
    L.total = o + 1024;
    return L;
}

// Item index -> CTA that owns it: the c with floor(c*W/P) <= x < floor((c+1)*W/P).
__host__ __device__ inline int cta_of_item(int64_t x, int64_t W, int P) {
    return static_cast<int>(((x + 1) * P - 1) / W);
}

__host__ __device__ inline bool cta_is_empty(int64_t c, int64_t W, int64_t P) {
    return c * W / P == (c + 1) * W / P;
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

// cum[s] = chunks * sum_{s' < s, ctx_s' > 0} (ceil(ctx_s' / bs) + phantom);
// cum[num_seqs] = W.
static __device__ void build_prefix(const DecodeArgs& a, int chunks, int32_t* cum, int32_t* scan) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    int carry = 0;
    for (int base = 0; base < a.num_seqs; base += blockDim.x) {
        const int s = base + tid;
        int v = 0;
        if (s < a.num_seqs) {
            const int c = clamp_context(a, s, blockIdx.x == 0);
            const int nb = (c + a.block_size - 1) / a.block_size;
            v = nb > 0 ? (nb + a.phantom) * chunks : 0;
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
// kTensor: stages arrive through 2-D tensor maps with a 128-byte swizzle (box
// of 128 bytes x Hc*bs rows, one box per 128-byte slice of the row);
// otherwise as two plain contiguous bulk copies.
template <bool kTensor>
static __device__ void produce(const DecodeArgs& a, uint8_t* ring, uint64_t* full, uint64_t* empty,
                        const int32_t* cum, int chunks, int start, int end, int half_bytes,
                        const CUtensorMap* tmk, const CUtensorMap* tmv, volatile int* abort) {
    const int lane = threadIdx.x & 31;
    const uint64_t policy = policy_evict_first();
    const int stage_bytes = 2 * half_bytes;
    const int64_t row_bytes = static_cast<int64_t>(a.head_dim) * dtype_bytes(a.kv_dtype);
    int issued = 0;  // items whose copies were issued (lane 0)
    int stage = 0, round = 0;
    bool ok = true;
    for (int base = start; base < end && ok; base += 32) {
        const int i = base + lane;
        int64_t row = -1;  // first pool row of the item: (blk * Hkv + hc * Hc) * bs; -1: no data
        if (i < end) {
            const int s = find_sequence(cum, a.num_seqs, i);
            const int nbv = (cum[s + 1] - cum[s]) / chunks;  // the pair's items, phantoms included
            const int r = i - cum[s];
            const int hc = r / nbv;
            const int j = r - hc * nbv - a.phantom;
            if (j >= 0) {
                int blk = __ldg(a.block_tables + static_cast<int64_t>(s) * a.max_blocks + j);
                if (blk < 0 || blk >= a.num_blocks) {
                    raise_flag(a.status, kFlagBadBlock);
                    blk = 0;
                }
                row = (static_cast<int64_t>(blk) * a.num_kv_heads + hc * a.heads_per_stage) * a.block_size;
            }
        }
        // With early reads the cache is not written by the launch still
        // running, and this CTA typically starts while that launch's last
        // CTAs finish: the items just past the first ring fill are brought
        // into L2 now, so that they stream from L2 later.  Only for long
        // ranges: with a few dozen items a CTA (a layer of ~80 us) the
        // prefetches slowed the previous launch's last CTAs more than they
        // saved (batch-32 step -2.6 %); with hundreds (a layer of ~550 us)
        // the step gained 1.6 %.
        if (a.early_reads && base == start && end - start >= kPrefetchMinItems && lane >= a.stages &&
            lane < a.stages + kPrefetchItems && i < end && row >= 0) {
            const int64_t off = row * row_bytes;
            prefetch_l2(static_cast<const char*>(a.k_cache) + off, half_bytes);
            prefetch_l2(static_cast<const char*>(a.v_cache) + off, half_bytes);
        }
        const int n = min(32, end - base);
        for (int k = 0; k < n; ++k) {
            const int64_t rk = __shfl_sync(0xffffffffu, row, k);
            int good = 1;
            if (lane == 0) {
                // Test-only stall: CTA 0 stops after its first item, so that a
                // consumer's bounded wait for the second one runs out.
                if (a.test_stall && blockIdx.x == 0 && base + k - start == 1) good = 0;
                if (good && round > 0)
                    good = mbar_wait_bounded(&empty[stage], (round - 1) & 1, abort, a.status);
                if (good && rk < 0) {  // a phantom item: the stage completes without data
                    mbar_arrive(&full[stage]);
                    ++issued;
                } else if (good) {
                    uint8_t* kd = ring + stage * stage_bytes;
                    uint8_t* vd = kd + half_bytes;
                    mbar_arrive_expect_tx(&full[stage], stage_bytes);
                    if constexpr (kTensor) {
                        // One box per 128-byte slice of the row (64 f16/bf16
                        // or 128 E4M3 elements).
                        const int per = 128 / static_cast<int>(dtype_bytes(a.kv_dtype));
                        const int slices = a.head_dim / per;
                        const int slice_bytes = half_bytes / slices;
                        for (int sl = 0; sl < slices; ++sl) {
                            tensor_load_2d(kd + sl * slice_bytes, tmk, sl * per, static_cast<int>(rk),
                                           &full[stage], policy);
                            tensor_load_2d(vd + sl * slice_bytes, tmv, sl * per, static_cast<int>(rk),
                                           &full[stage], policy);
                        }
                    } else {
                        const int64_t off = rk * row_bytes;
                        bulk_load(kd, static_cast<const char*>(a.k_cache) + off, half_bytes,
                                  &full[stage], policy);
                        bulk_load(vd, static_cast<const char*>(a.v_cache) + off, half_bytes,
                                  &full[stage], policy);
                    }
                    ++issued;
                }
            }
            if (++stage == a.stages) {
                stage = 0;
                ++round;
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

// ------------------------------------------------- merge of split pairs
// Called by one warp per (sequence s, KV head h) after it wrote its partial
// for slot c + pair.  Counts the arrival; the warp that arrives last merges
// the partials of (s, h) into the output and resets the counter.
//
// The merge keeps its L2 round trips few: lane l fetches (max, sum) of part
// l / G, head l % G in one load, the weights are shared by shuffles, and the
// partial outputs of two parts (all G heads, D/32 dims per lane) are loaded
// together before they are used.
template <int G, int D, int kPre>
__device__ __forceinline__ void merge_parts(const DecodeArgs& a, int s, int h, int hw, int pair,
                                            int ca, int cb, int64_t W) {
    constexpr int VD = D / 32;
    const int lane = threadIdx.x & 31;
    const int Hc = a.heads_per_stage;
    const int64_t P = a.num_ctas;
    const int kp = lane / G, kg = lane % G;  // this lane's (part, head) for the (max, sum) loads
    float acc[G][VD];
    float M[G], Lsum[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        M[g] = -INFINITY;
        Lsum[g] = 0.f;
#pragma unroll
        for (int i = 0; i < VD; ++i) acc[g][i] = 0.f;
    }
    int c = ca;
    while (c <= cb) {
        // This lane's part: the kp-th CTA with a non-empty item range from c
        // on.  With W >= P every CTA holds items.  With fewer items than CTAs
        // a CTA holds at most one, and the first CTA from c on that holds any
        // holds item floor(c W / P): the kp-th is the CTA of that item + kp.
        int my_c;
        if (W >= P) {
            my_c = c + kp <= cb ? c + kp : -1;
        } else {
            const int64_t x = static_cast<int64_t>(c) * W / P + kp;
            my_c = -1;
            if (x < W) {
                const int cx = cta_of_item(x, W, P);
                if (cx <= cb) my_c = cx;
            }
        }
        const int n = __popc(__ballot_sync(0xffffffffu, my_c >= 0 && kg == 0));
        if (n == 0) break;
        c = __shfl_sync(0xffffffffu, my_c, (n - 1) * G) + 1;
        // The partial outputs of the first kPre parts are loaded together with
        // the (max, sum) pairs, so that a typical merge (a pair split over a
        // handful of CTAs) waits for fewer rounds of loads.
        float pre[kPre][G][VD];
#pragma unroll
        for (int k = 0; k < kPre; ++k) {
            const int ck = __shfl_sync(0xffffffffu, my_c, (k < n ? k : 0) * G);
            const int64_t s0 = ((static_cast<int64_t>(ck) + pair) * Hc + hw) * G;
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int i = 0; i < VD; ++i)
                    pre[k][g][i] = k < n ? __ldcg(a.part_o + (s0 + g) * D + lane + 32 * i) : 0.f;
        }
        float2 ml = make_float2(-INFINITY, 0.f);
        if (my_c >= 0) {
            const int64_t sl = ((static_cast<int64_t>(my_c) + pair) * Hc + hw) * G + kg;
            ml = __ldcg(reinterpret_cast<const float2*>(a.part_ml + sl * 2));
        }
        // New running max per head; rescale what was accumulated so far.
        float w_lane = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float mg = -INFINITY;
            for (int k = 0; k < n; ++k) mg = fmaxf(mg, __shfl_sync(0xffffffffu, ml.x, k * G + g));
            const float mn = fmaxf(M[g], mg);
            const float al = fast_exp2(M[g] - mn);
            M[g] = mn;
            Lsum[g] *= al;
#pragma unroll
            for (int i = 0; i < VD; ++i) acc[g][i] *= al;
            if (kg == g && my_c >= 0) w_lane = fast_exp2(ml.x - mn);
        }
        const float wl = w_lane * ml.y;
#pragma unroll
        for (int g = 0; g < G; ++g)
            for (int k = 0; k < n; ++k) Lsum[g] += __shfl_sync(0xffffffffu, wl, k * G + g);
#pragma unroll
        for (int k = 0; k < kPre; ++k) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float w = __shfl_sync(0xffffffffu, w_lane, (k < n ? k : 0) * G + g);
                if (k >= n) w = 0.f;
#pragma unroll
                for (int i = 0; i < VD; ++i) acc[g][i] += w * pre[k][g][i];
            }
        }
        // The remaining partial outputs, two parts per round of loads.
        for (int k = kPre; k < n; k += 2) {
            const int c0 = __shfl_sync(0xffffffffu, my_c, k * G);
            const int c1 = __shfl_sync(0xffffffffu, my_c, (k + 1 < n ? k + 1 : k) * G);
            const int64_t s0 = ((static_cast<int64_t>(c0) + pair) * Hc + hw) * G;
            const int64_t s1 = ((static_cast<int64_t>(c1) + pair) * Hc + hw) * G;
            float v0[G][VD], v1[G][VD];
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int i = 0; i < VD; ++i) {
                    v0[g][i] = __ldcg(a.part_o + (s0 + g) * D + lane + 32 * i);
                    v1[g][i] = __ldcg(a.part_o + (s1 + g) * D + lane + 32 * i);
                }
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float w0 = __shfl_sync(0xffffffffu, w_lane, k * G + g);
                float w1 = __shfl_sync(0xffffffffu, w_lane, (k + 1 < n ? k + 1 : k) * G + g);
                if (k + 1 >= n) w1 = 0.f;
#pragma unroll
                for (int i = 0; i < VD; ++i) acc[g][i] += w0 * v0[g][i] + w1 * v1[g][i];
            }
        }
    }
    const int64_t o0 = (static_cast<int64_t>(s) * a.num_q_heads + h * G) * D;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float inv = 1.f / Lsum[g];
#pragma unroll
        for (int i = 0; i < VD; ++i)
            store_out(a.out, o0 + g * D + lane + 32 * i, acc[g][i] * inv, a.out_dtype);
    }
}

// The merge of a pair split over n <= kSlots * 32/G parts ca .. ca+n-1, none
// empty.  Lane l loads (max, sum) of parts l / G + j * 32/G, head l % G
// (j < kSlots);
// xor shuffles over lanes holding the same head give each head's max M and
// sum L in one round.  The outputs are then summed part by part in slot
// order (one fma per part), so the result does not depend on where they are
// read from:
// - scratch: this warp's slice of the CTA's ring (scratch_parts parts), free
//   at the end of the CTA's item range; the parts' outputs are copied there
//   in chunks of 16-byte copies, the first issued together with the (max,
//   sum) loads: one round of loads per chunk;
// - otherwise from L2, kPre parts per round of loads.
template <int G, int D, int kPre, int kSlots>
__device__ __forceinline__ void merge_parts_small(const DecodeArgs& a, int s, int h, int hw, int pair,
                                                  int ca, int n, float* scratch, int scratch_parts) {
    constexpr int VD = D / 32;
    constexpr int kPart = G * D;  // floats of one part's outputs
    constexpr int kLaneParts = 32 / G;  // parts per round of (max, sum) loads
    const int lane = threadIdx.x & 31;
    const int Hc = a.heads_per_stage;
    auto part_out = [&](int k) {
        return a.part_o + ((static_cast<int64_t>(ca + k) + pair) * Hc + hw) * kPart;
    };
    auto stage_parts = [&](int k0, int k1) {  // parts [k0, k1) to scratch
        const uint32_t dst0 = smem_addr(scratch);
        for (int e = lane; e < (k1 - k0) * (kPart / 4); e += 32) {
            const int k = e / (kPart / 4);
            cp_async_16(dst0 + 16u * static_cast<uint32_t>(e), part_out(k0 + k) + 4 * (e - k * (kPart / 4)));
        }
    };
    const int chunk = scratch ? scratch_parts : 0;
    if (chunk) stage_parts(0, min(n, chunk));
    const int kp = lane / G, kg = lane % G;
    float m[kSlots], l[kSlots];
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
        m[j] = -INFINITY;
        l[j] = 0.f;
        const int k = kp + j * kLaneParts;
        if (k < n) {
            const float2 ml = __ldcg(reinterpret_cast<const float2*>(
                a.part_ml + (((static_cast<int64_t>(ca + k) + pair) * Hc + hw) * G + kg) * 2));
            m[j] = ml.x;
            l[j] = ml.y;
        }
    }
    float M = m[0];
#pragma unroll
    for (int j = 1; j < kSlots; ++j) M = fmaxf(M, m[j]);
#pragma unroll
    for (int o = G; o < 32; o <<= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
    float w[kSlots];
    float L = 0.f;
#pragma unroll
    for (int j = 0; j < kSlots; ++j) {
        w[j] = kp + j * kLaneParts < n ? fast_exp2(m[j] - M) : 0.f;
        L += w[j] * l[j];
    }
#pragma unroll
    for (int o = G; o < 32; o <<= 1) L += __shfl_xor_sync(0xffffffffu, L, o);
    // Weight of part k, head g (k < n): held by lane (k % kLaneParts) * G + g, slot k / kLaneParts.
    auto weight = [&](int k, int g) {
        const int j = k / kLaneParts;  // the same on every lane
        float wj = w[0];
#pragma unroll
        for (int t = 1; t < kSlots; ++t)
            if (j == t) wj = w[t];
        return __shfl_sync(0xffffffffu, wj, (k % kLaneParts) * G + g);
    };
    float acc[G][VD];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int i = 0; i < VD; ++i) acc[g][i] = 0.f;
    if (chunk) {
        for (int k0 = 0; k0 < n; k0 += chunk) {
            const int k1 = min(n, k0 + chunk);
            if (k0 > 0) {
                __syncwarp();  // the previous chunk is read
                stage_parts(k0, k1);
            }
            cp_async_wait_all();
            __syncwarp();
            for (int k = k0; k < k1; ++k) {
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float wk = weight(k, g);
#pragma unroll
                    for (int i = 0; i < VD; ++i)
                        acc[g][i] = fmaf(wk, scratch[(k - k0) * kPart + g * D + lane + 32 * i], acc[g][i]);
                }
            }
        }
    } else {
        for (int k0 = 0; k0 < n; k0 += kPre) {
            float v[kPre][G][VD];
#pragma unroll
            for (int j = 0; j < kPre; ++j) {
                const float* src = part_out(k0 + j < n ? k0 + j : 0);
#pragma unroll
                for (int g = 0; g < G; ++g)
#pragma unroll
                    for (int i = 0; i < VD; ++i)
                        v[j][g][i] = k0 + j < n ? __ldcg(src + g * D + lane + 32 * i) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < kPre; ++j) {
                if (k0 + j >= n) break;
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    const float wk = weight(k0 + j, g);
#pragma unroll
                    for (int i = 0; i < VD; ++i) acc[g][i] = fmaf(wk, v[j][g][i], acc[g][i]);
                }
            }
        }
    }
    const int64_t o0 = (static_cast<int64_t>(s) * a.num_q_heads + h * G) * D;
#pragma unroll
    for (int g = 0; g < G; ++g) {
        const float inv = 1.f / __shfl_sync(0xffffffffu, L, g);  // lane g holds head g's sum
#pragma unroll
        for (int i = 0; i < VD; ++i)
            store_out(a.out, o0 + g * D + lane + 32 * i, acc[g][i] * inv, a.out_dtype);
    }
}

// Count one arrival on a merge counter (gpu scope, acquire + release): the
// writes ordered before it (the warp's partial, through the warp barrier
// before it) are visible to whoever counts later, and the partials of every
// warp that counted before are visible after it.
__device__ __forceinline__ int counter_arrive(int32_t* counter) {
    int prev;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], 1;" : "=r"(prev) : "l"(counter) : "memory");
    return prev;
}

// Parts whose outputs the merge loads together with the (max, sum) pairs:
// up to 32 values a lane in a kernel built for at most 384 threads (168
// registers a thread), 16 in one built for 512 (128 registers); 1 to 4.
__host__ __device__ constexpr int merge_prefetch(int G, int D, int max_threads) {
    const int per_part = G * (D / 32);
    const int k = (max_threads <= 32 * 12 ? 32 : 16) / per_part;
    return k < 1 ? 1 : (k > 4 ? 4 : k);
}

// scratch: this warp's slice of the free ring (scratch_floats floats), or
// null when the ring is still in use.
template <int G, int D, int kPre>
__device__ void merge_if_last(const DecodeArgs& a, int s, int h, int hw, int pair, int nparts,
                              int ca, int cb, int64_t W, float* scratch, int scratch_floats) {
    const int lane = threadIdx.x & 31;
    int32_t* counter = a.counters + static_cast<int64_t>(s) * a.num_kv_heads + h;
    __syncwarp();  // the warp's partial stores come before lane 0's release
    int prev = 0;
    if (lane == 0) prev = counter_arrive(counter);
    prev = __shfl_sync(0xffffffffu, prev, 0);
    if (prev != nparts - 1) return;
    __syncwarp();  // and every lane's loads after lane 0's acquire
    // Which warp merges depends on timing, so the choice of path depends on
    // the pair only; the ring (when free) changes where the loads come from,
    // not the arithmetic.
    // (One slot a lane covers the usual split over a few CTAs; four, up to
    // 128/G parts, a small batch spread over many.)
    if (W >= a.num_ctas && nparts * G <= 32)
        merge_parts_small<G, D, kPre, 1>(a, s, h, hw, pair, ca, nparts, scratch, scratch_floats / (G * D));
    else if (W >= a.num_ctas && nparts * G <= 128)
        merge_parts_small<G, D, kPre, 4>(a, s, h, hw, pair, ca, nparts, scratch, scratch_floats / (G * D));
    else
        merge_parts<G, D, kPre>(a, s, h, hw, pair, ca, cb, W);
    __syncwarp();
    if (lane == 0) *counter = 0;
}

// Combine the R warps' states of head hw (shared memory, [warp][g][D+2]) and
// write the final output (whole pair) or the CTA's partial.  One warp.
static __device__ void combine_replicas(const DecodeArgs& a, const float* merge, int hw, int Hc, int R,
                                 int G, bool whole, int s, int h, float* part_o, float* part_ml) {
    const int lane = threadIdx.x & 31;
    const int D = a.head_dim;
    for (int g = 0; g < G; ++g) {
        float M = -INFINITY;
        for (int r = 0; r < R; ++r) M = fmaxf(M, merge[((hw + r * Hc) * G + g) * (D + 2) + D]);
        float Lsum = 0.f;
        for (int r = 0; r < R; ++r) {
            const float* mr = merge + ((hw + r * Hc) * G + g) * (D + 2);
            Lsum += fast_exp2(mr[D] - M) * mr[D + 1];
        }
        const int64_t o0 = (static_cast<int64_t>(s) * a.num_q_heads + h * G + g) * D;
        for (int d = lane; d < D; d += 32) {
            float O = 0.f;
            for (int r = 0; r < R; ++r) {
                const float* mr = merge + ((hw + r * Hc) * G + g) * (D + 2);
                O += fast_exp2(mr[D] - M) * mr[d];
            }
            if (whole)
                store_out(a.out, o0 + d, O / Lsum, a.out_dtype);
            else
                part_o[g * D + d] = O;
        }
        if (!whole && lane == 0) {
            part_ml[g * 2] = M;
            part_ml[g * 2 + 1] = Lsum;
        }
    }
}

// ------------------------------------------------------------ fused append
// The warp that consumes the last block of (s, h) writes the new token's K
// and V rows (k_new[s][h], v_new[s][h]) into row r of that block: into the
// staged tile in shared memory (so this step attends to it) and into the
// pool in HBM (so later steps do).  Returns whether it wrote.
template <class Policy>
__device__ __forceinline__ bool append_row(const DecodeArgs& a, const Policy& pol, uint8_t* kt,
                                           uint8_t* vt, int s, int h, int hw, int j, int r) {
    const int lane = threadIdx.x & 31;
    const int blk = a.block_tables[static_cast<int64_t>(s) * a.max_blocks + j];
    if (blk < 0 || blk >= a.num_blocks) return false;  // already flagged by the producer
    // The slot is reported whether or not this sequence appends (as kv_slot_mapping does).
    if (a.slot_out && h == 0 && lane == 0) a.slot_out[s] = blk * a.block_size + r;
    if (a.append_ids && a.append_ids[s] < 0) return false;
    const int eb = dtype_bytes(a.dtype);      // k_new / v_new
    const int ce = dtype_bytes(a.kv_dtype);   // cache
    const int nchunk = a.head_dim * ce / 16;  // 16-byte chunks of one cached row
    const int64_t src = (static_cast<int64_t>(s) * a.num_kv_heads + h) * a.head_dim * eb;
    const int64_t dst = ((static_cast<int64_t>(blk) * a.num_kv_heads + h) * a.block_size + r) *
                        static_cast<int64_t>(a.head_dim) * ce;
    for (int e = lane; e < 2 * nchunk; e += 32) {
        const bool isv = e >= nchunk;
        const int q = isv ? e - nchunk : e;
        const char* row = static_cast<const char*>(isv ? a.v_new : a.k_new) + src;
        const uint4 val = a.kv_dtype == kFP8
                              ? quantize_chunk16(row, q, a.dtype, isv ? a.v_scale : a.k_scale)
                              : __ldg(reinterpret_cast<const uint4*>(row) + q);
        *(reinterpret_cast<uint4*>(const_cast<char*>(
              static_cast<const char*>(isv ? a.v_cache : a.k_cache)) + dst) + q) = val;
        pol.patch_chunk(a, isv ? vt : kt, hw, r, q, val);
    }
    __syncwarp();
    return true;
}

// ---------------------------------------------------------------- the kernel
// Policy provides: State, begin(), tile(), write_state(), write_partial(),
// write_final(), kTensor, kScratch, kPairs (and tile2() when kPairs), and
// kMaxThreads, the largest block it is launched with (its register budget).
template <class Policy>
__global__ void __launch_bounds__(Policy::kMaxThreads, 1)
    paged_decode_partial_kernel(const DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
                                const __grid_constant__ CUtensorMap tmv) {
    extern __shared__ uint8_t smem_raw[];
    pdl_allow_next();
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int G = a.num_q_heads / a.num_kv_heads;
    const int Hc = a.heads_per_stage, R = a.warps_per_head, NC = a.consumer_warps;
    const int chunks = a.num_kv_heads / Hc;
    const int D = a.head_dim;
    const int half_bytes = Hc * a.block_size * D * dtype_bytes(a.kv_dtype);
    const SmemLayout L = smem_layout(a.stages, half_bytes, a.num_seqs, NC, R, G, D, a.block_size,
                                     Policy::kScratch);
    uint8_t* ring = base + L.ring;
    uint64_t* full = reinterpret_cast<uint64_t*>(base + L.full_bar);
    uint64_t* empty = reinterpret_cast<uint64_t*>(base + L.empty_bar);
    volatile int* abort = reinterpret_cast<volatile int*>(base + L.flags);
    int32_t* scan = reinterpret_cast<int32_t*>(base + L.scan);
    int32_t* cum = reinterpret_cast<int32_t*>(base + L.cum);
    float* merge = reinterpret_cast<float*>(base + L.merge);

    const int tid = threadIdx.x;
    if (a.stages % R != 0) {  // see decode_plan: the ring must be a multiple of R
        if (tid == 0 && blockIdx.x == 0) raise_flag(a.status, kFlagBadPlan);
        return;
    }
    if (tid == 0) {
        for (int st = 0; st < a.stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], Hc);  // one arrival per head of the chunk
        }
        *abort = 0;
        fence_barrier_init();
        if constexpr (Policy::kTensor) {
            prefetch_tensor_map(&tmk);
            prefetch_tensor_map(&tmv);
        }
    }
    // Everything above touches only this CTA's shared memory and parameters.
    // With early_reads the caller promises that the previous launch on the
    // stream writes neither the tables, the lengths nor the K/V cache, so the
    // prefix, the table entries and the first stages are fetched while that
    // launch finishes; everything else (q, the new rows, the workspace, the
    // outputs) is touched only after waiting for it.
    if (!a.early_reads) pdl_wait();
    build_prefix(a, chunks, cum, scan);  // ends with __syncthreads
    const int64_t W = cum[a.num_seqs];
    const int P = a.num_ctas;
    const int start = static_cast<int>(static_cast<int64_t>(blockIdx.x) * W / P);
    const int end = static_cast<int>((static_cast<int64_t>(blockIdx.x) + 1) * W / P);
    const int warp = tid >> 5, lane = tid & 31;
    if (warp == 0 && start < end) {
        produce<Policy::kTensor>(a, ring, full, empty, cum, chunks, start, end, half_bytes, &tmk,
                                 &tmv, abort);
        return;
    }
    if (a.early_reads) pdl_wait();
    // Global writes of the prologue, by the threads that are not producing.
    const int wt = start < end ? tid - 32 : tid;
    const int nwt = start < end ? static_cast<int>(blockDim.x) - 32 : static_cast<int>(blockDim.x);
    if (blockIdx.x == 0 && !a.fused_reduce) {
        for (int s = wt; s <= a.num_seqs; s += nwt) a.cum[s] = cum[s];
    }
    // Sequences with no tokens: zero rows (fused merge) and slot -1 (CTA s mod P).
    for (int s = blockIdx.x; s < a.num_seqs; s += P) {
        if (cum[s + 1] != cum[s]) continue;
        if (a.slot_out && wt == 0) a.slot_out[s] = -1;
        if (!a.fused_reduce) continue;
        const int64_t o0 = static_cast<int64_t>(s) * a.num_q_heads * D;
        for (int e = wt; e < a.num_q_heads * D; e += nwt) store_out(a.out, o0 + e, 0.f, a.out_dtype);
    }
    if (start >= end) return;

    const int w = warp - 1;
    const int hw = w % Hc;  // head within the chunk
    const int rr = w / Hc;  // replica among the R warps of that head
    float* scratch = Policy::kScratch
                         ? reinterpret_cast<float*>(base + L.scratch) +
                               w * ((a.block_size * G * 4 + 15) & ~15) / 4
                         : nullptr;
    Policy pol;
    typename Policy::State st;
    int seg = start;
    while (seg < end) {
        const int s = find_sequence(cum, a.num_seqs, seg);
        const int nbv = (cum[s + 1] - cum[s]) / chunks;  // the pair's items, phantoms included
        const int nb = nbv - a.phantom;                    // its blocks
        const int hc = (seg - cum[s]) / nbv;
        const int pair_a = cum[s] + hc * nbv;
        const int pair_b = pair_a + nbv;
        const int seg_end = min(pair_b, end);
        const int h = hc * Hc + hw;
        const int ctx = clamp_context(a, s, false);
        pol.begin(st, a, s, h, G);
        const int first = seg + (((rr - (seg - start)) % R) + R) % R;
        // Ring position of item `first` (item t = i - start sits in stage
        // t % stages, phase (t / stages) & 1); advanced by R per item below.
        int stage = (first - start) % a.stages;
        uint32_t phase = static_cast<uint32_t>((first - start) / a.stages) & 1u;
        for (int i = first; i < seg_end;) {
            // With a policy that takes two 16-token blocks at once, this warp
            // takes items i and i + R together when both belong to the run.
            // Waiting for the second while holding the first needs the
            // producer to have refilled stage (i + R) % stages, i.e. item
            // i + R - stages to be released: true when stages >= 2R.
            const int j = i - pair_a - a.phantom;  // block index; negative: a phantom item
            bool two = false;
            if constexpr (Policy::kPairs)
                two = a.block_size == 16 && i + R < seg_end && a.stages >= 2 * R && j >= 0;
            int stage2 = stage + R;  // R divides the ring size, so this wraps exactly at the end
            uint32_t phase2 = phase;
            if (stage2 >= a.stages) {
                stage2 -= a.stages;
                phase2 ^= 1u;
            }
            bool ok = mbar_wait_bounded(&full[stage], phase, abort, a.status);
            if (ok && two) ok = mbar_wait_bounded(&full[stage2], phase2, abort, a.status);
            if (ok && j >= 0) {
                const int n_valid = min(a.block_size, ctx - j * a.block_size);
                uint8_t* kt = ring + stage * 2 * half_bytes;
                bool patched = a.k_new && j == nb - 1 && append_row(a, pol, kt, kt + half_bytes, s, h, hw, j, n_valid - 1);
                if constexpr (Policy::kPairs) {
                    if (two) {
                        const int j1 = j + R;
                        const int n1 = min(a.block_size, ctx - j1 * a.block_size);
                        uint8_t* kt1 = ring + stage2 * 2 * half_bytes;
                        if (a.k_new && j1 == nb - 1)
                            patched |= append_row(a, pol, kt1, kt1 + half_bytes, s, h, hw, j1, n1 - 1);
                        pol.tile2(st, a, kt, kt + half_bytes, n_valid, kt1, kt1 + half_bytes, n1, hw, G);
                    }
                }
                if (!two) pol.tile(st, a, kt, kt + half_bytes, hw, n_valid, G, scratch);
                if (patched) fence_proxy_async_smem();  // generic writes before the next TMA fill
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[stage]);
                if (two) mbar_arrive(&empty[stage2]);
            }
            i += two ? 2 * R : R;
            stage = stage2;
            phase = phase2;
            if (two) {
                stage += R;
                if (stage >= a.stages) {
                    stage -= a.stages;
                    phase ^= 1u;
                }
            }
        }
        // The pair's blocks are its items [pair_r, pair_b) (phantoms first).
        // A segment holding none of them is not a part of the pair: it
        // writes nothing and counts no arrival (the same on every warp).
        const int pair_r = pair_a + a.phantom;
        const bool whole = (pair_r >= start) && (pair_b <= end);
        const bool blocks = max(seg, pair_r) < seg_end;
        const int pair = s * chunks + hc;
        const int64_t sl = (static_cast<int64_t>(blockIdx.x + pair) * Hc + hw) * G;
        bool partial = false;  // this warp wrote the CTA's partial of (s, h)
        if (!blocks) {
        } else if (R == 1) {
            if (!*abort) {
                if (whole) {
                    pol.write_final(st, a, s, h, G);
                } else {
                    pol.write_partial(st, a, a.part_o + sl * D, a.part_ml + sl * 2, G);
                    partial = true;
                }
            }
        } else {
            // Merge the R warps of each head through shared memory.
            pol.write_state(st, a, merge + w * G * (D + 2), D + 2, G);
            named_barrier_sync(1, NC * 32);
            if (rr == 0 && !*abort) {
                combine_replicas(a, merge, hw, Hc, R, G, whole, s, h, a.part_o + sl * D,
                                 a.part_ml + sl * 2);
                partial = !whole;
            }
            named_barrier_sync(1, NC * 32);
        }
        // A split pair at the end of the range: once every consumer warp is
        // past its last stage, the ring's shared memory is free (the producer
        // issued nothing after the range's last item) and the merge may stage
        // the parts there, one slice a warp.
        float* staging = nullptr;
        int staging_floats = 0;
        if (R == 1 && a.fused_reduce && seg_end == end && !whole && blocks) {
            named_barrier_sync(1, NC * 32);
            staging_floats = (a.stages * 2 * half_bytes / NC / 4) & ~3;
            staging = reinterpret_cast<float*>(ring) + w * staging_floats;
        }
        if (partial && a.fused_reduce) {
            // The parts: the CTAs holding the pair's blocks.  With fewer
            // items than CTAs each block has its own CTA.
            const int ca = cta_of_item(pair_r, W, P);
            const int cb = cta_of_item(pair_b - 1, W, P);
            const int nparts = W >= P ? cb - ca + 1 : pair_b - pair_r;
            constexpr int T = Policy::kMaxThreads, DD = Policy::kD;
            switch (G) {
                case 1:
                    merge_if_last<1, DD, merge_prefetch(1, DD, T)>(a, s, h, hw, pair, nparts, ca, cb, W,
                                                                  staging, staging_floats);
                    break;
                case 2:
                    merge_if_last<2, DD, merge_prefetch(2, DD, T)>(a, s, h, hw, pair, nparts, ca, cb, W,
                                                                  staging, staging_floats);
                    break;
                case 4:
                    merge_if_last<4, DD, merge_prefetch(4, DD, T)>(a, s, h, hw, pair, nparts, ca, cb, W,
                                                                  staging, staging_floats);
                    break;
                default:
                    merge_if_last<8, DD, merge_prefetch(8, DD, T)>(a, s, h, hw, pair, nparts, ca, cb, W,
                                                                  staging, staging_floats);
                    break;
            }
        }
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
    if (32 * (1 + a.consumer_warps) > Policy::kMaxThreads) return cudaErrorInvalidValue;
    return launch_kernel(kern, dim3(a.num_ctas), dim3(32 * (1 + a.consumer_warps)),
                         static_cast<size_t>(a.smem_bytes), stream, a.pdl != 0, a, tmk, tmv);
}

}  // namespace pkv
