// Multi-token queries over the paged cache (chunked prefill: "Batching and
// Scheduling", Example 5; "vLLM Architecture and Installation", Example 5).
//
// A step gives sequence s n_s = query_start[s+1] - query_start[s] new tokens
// (1 for a decoding request, a chunk of the prompt for a prefilling one),
// already appended, so its cache holds context_lens[s] tokens and new token i
// sits at position p_i = context_lens[s] - n_s + i.  Token i attends to the
// cached tokens at positions 0 .. p_i (causal), read through the block table.
//
// Work split: one CTA per (tile of 16 new tokens of one sequence, KV head).
// Warp 0 streams that head's K and V tiles of the blocks the tile needs
// (positions up to the tile's last p_i) into a ring of shared-memory stages
// with TMA (128-byte swizzle, as the decode kernel); warp 1 + w computes query
// head h*G + w for the 16 tokens, in the usual flash-attention register layout:
//   S[16 tok x 16 keys] = Q[16 x D] . K^T     (m16n8k16, Q in registers, K by ldmatrix)
//   causal mask, online softmax per row (fp32, base 2)
//   O[16 x D] += P[16 x 16] . V[16 x D]       (P from the S registers as the A
//                                             operand, high + low halves; V by ldmatrix.trans)
// The tile index -> (sequence, tile) map comes from a small plan kernel
// (prefix of tiles per sequence in the workspace).
#include "decode_kernel.cuh"
#include "mma_frag.cuh"

namespace pkv {

namespace {

constexpr int kQT = 16;  // new tokens per tile

// cum[s] = sum_{s' < s} ceil(n_s' / tile_tokens); cum[B] = tiles.  One block; flags
// a chunk longer than its context or a decreasing query_start.
__global__ void __launch_bounds__(1024) prefill_plan_kernel(const PrefillArgs a) {
    pdl_allow_next();
    pdl_wait();
    __shared__ int32_t warp_sum[32];
    __shared__ int32_t carry_s;
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) carry_s = 0;
    __syncthreads();
    for (int base = 0; base < a.num_seqs; base += blockDim.x) {
        const int s = base + tid;
        int v = 0;
        if (s < a.num_seqs) {
            const int n = a.query_start[s + 1] - a.query_start[s];
            const int c = a.context_lens[s];
            if (n < 0 || n > c || c > a.max_blocks * a.block_size) raise_flag(a.status, kFlagBadContext);
            v = n > 0 && n <= c && c <= a.max_blocks * a.block_size ? (n + a.tile_tokens - 1) / a.tile_tokens : 0;
        }
        int x = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_sum[wid] = x;
        __syncthreads();
        if (wid == 0) {
            const int nw = blockDim.x >> 5;
            int t = lane < nw ? warp_sum[lane] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, t, o);
                if (lane >= o) t += y;
            }
            warp_sum[lane] = t;
        }
        __syncthreads();
        const int before = carry_s + (wid > 0 ? warp_sum[wid - 1] : 0);
        if (s < a.num_seqs) a.tile_cum[s] = before + x - v;
        __syncthreads();
        if (tid == 0) carry_s += warp_sum[(blockDim.x >> 5) - 1];
        __syncthreads();
    }
    if (tid == 0) a.tile_cum[a.num_seqs] = carry_s;
}

template <int DT, int D>
struct PrefillTile {
    using T = typename Elem<DT>::T;
    static constexpr int KS = D / 16;  // k-steps of QK
    static constexpr int ND = D / 8;   // 8-dim column groups of O

    uint32_t qa[KS][4];  // A fragments of Q: rows g / g+8, dims 16ks + 2c (+8)
    float o[ND][4];      // O: rows g / g+8, dims 8nd + 2c, 2c+1
    float m[2], l[2];    // rows g and g+8
    int qpos[2];         // positions of rows g and g+8

    // q rows of tokens t0 .. t0+15 of head `head` (rows past n repeat the last token).
    __device__ __forceinline__ void begin(const PrefillArgs& a, int64_t tok0, int rows, int head,
                                          int pos0) {
        const int lane = threadIdx.x & 31;
        const int g = lane >> 2, c = lane & 3;
        const int r0 = g < rows ? g : rows - 1, r1 = g + 8 < rows ? g + 8 : rows - 1;
        const T* q0 = static_cast<const T*>(a.q) + ((tok0 + r0) * a.num_q_heads + head) * D;
        const T* q1 = static_cast<const T*>(a.q) + ((tok0 + r1) * a.num_q_heads + head) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qa[ks][0] = *reinterpret_cast<const uint32_t*>(q0 + 16 * ks + 2 * c);
            qa[ks][1] = *reinterpret_cast<const uint32_t*>(q1 + 16 * ks + 2 * c);
            qa[ks][2] = *reinterpret_cast<const uint32_t*>(q0 + 16 * ks + 2 * c + 8);
            qa[ks][3] = *reinterpret_cast<const uint32_t*>(q1 + 16 * ks + 2 * c + 8);
        }
#pragma unroll
        for (int nd = 0; nd < ND; ++nd)
#pragma unroll
            for (int r = 0; r < 4; ++r) o[nd][r] = 0.f;
        m[0] = m[1] = -INFINITY;
        l[0] = l[1] = 0.f;
        qpos[0] = pos0 + r0;
        qpos[1] = pos0 + r1;
    }

    // 16 keys at positions kpos0 .. kpos0+15 in rows row0 .. row0+15 of a
    // stage ([64-element slice][bs rows][128 B], 128-byte swizzled).
    __device__ __forceinline__ void slice(const PrefillArgs& a, uint32_t kbase, uint32_t vbase,
                                          uint32_t slice_bytes, int row0, int kpos0) {
        const int lane = threadIdx.x & 31;
        const int c = lane & 3;
        const uint32_t sw = lane & 7;
        // ---- S = Q . K^T: n-group 0 = keys 0-7, 1 = keys 8-15; two chains each
        float s[2][2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int e = 0; e < 2; ++e)
#pragma unroll
                for (int r = 0; r < 4; ++r) s[n][e][r] = 0.f;
        {
            // lanes 0-7 / 8-15 / 16-23 / 24-31: keys 0-7 chunk 2j / keys 0-7 chunk 2j+1 /
            // keys 8-15 chunk 2j / keys 8-15 chunk 2j+1
            const uint32_t row = static_cast<uint32_t>(row0 + (lane & 7) + ((lane >> 4) << 3));
            const uint32_t csel = (lane >> 3) & 1;
#pragma unroll
            for (int ks = 0; ks < KS; ++ks) {
                const uint32_t chunk = ((ks & 3) << 1) | csel;
                uint32_t b[4];
                ldsm_x4(b, kbase + (ks >> 2) * slice_bytes + row * 128u + ((chunk ^ sw) << 4));
                mma16816<DT>(s[0][ks & 1], qa[ks], b[0], b[1]);
                mma16816<DT>(s[1][ks & 1], qa[ks], b[2], b[3]);
            }
        }
        // ---- causal mask and online softmax (rows g, g+8; 4 keys each per lane)
        float x[2][4];  // [n-group][c0..c3]: (row g, key 2c), (row g, 2c+1), (row g+8, 2c), (row g+8, 2c+1)
#pragma unroll
        for (int n = 0; n < 2; ++n)
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                const int key = kpos0 + 8 * n + 2 * c + (r & 1);
                const int qp = qpos[r >> 1];
                const float v = (s[n][0][r] + s[n][1][r]) * a.scale_log2;
                x[n][r] = key <= qp ? v : -INFINITY;
            }
        float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(m[0], mx0), mn1 = fmaxf(m[1], mx1);
        // A row whose keys are all masked so far keeps m = -inf; its weights are 0.
        const float al0 = mn0 == -INFINITY ? 1.f : fast_exp2(m[0] - mn0);
        const float al1 = mn1 == -INFINITY ? 1.f : fast_exp2(m[1] - mn1);
        m[0] = mn0;
        m[1] = mn1;
        float p[2][4];
#pragma unroll
        for (int n = 0; n < 2; ++n) {
            p[n][0] = mn0 == -INFINITY ? 0.f : fast_exp2(x[n][0] - mn0);
            p[n][1] = mn0 == -INFINITY ? 0.f : fast_exp2(x[n][1] - mn0);
            p[n][2] = mn1 == -INFINITY ? 0.f : fast_exp2(x[n][2] - mn1);
            p[n][3] = mn1 == -INFINITY ? 0.f : fast_exp2(x[n][3] - mn1);
        }
        l[0] = l[0] * al0 + (p[0][0] + p[0][1] + p[1][0] + p[1][1]);
        l[1] = l[1] * al1 + (p[0][2] + p[0][3] + p[1][2] + p[1][3]);
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int nd = 0; nd < ND; ++nd) {
                o[nd][0] *= al0;
                o[nd][1] *= al0;
                o[nd][2] *= al1;
                o[nd][3] *= al1;
            }
        }
        // ---- P as A fragments (rows g / g+8, keys 2c.. / 8+2c..), high + low parts
        uint32_t ph[4], pl[4];
        pack_split<DT>(p[0][0], p[0][1], ph[0], pl[0]);  // row g,   keys 2c, 2c+1
        pack_split<DT>(p[0][2], p[0][3], ph[1], pl[1]);  // row g+8, keys 2c, 2c+1
        pack_split<DT>(p[1][0], p[1][1], ph[2], pl[2]);  // row g,   keys 8+2c, 9+2c
        pack_split<DT>(p[1][2], p[1][3], ph[3], pl[3]);  // row g+8, keys 8+2c, 9+2c
        // ---- O += P . V: ldmatrix.trans gives the B fragments (keys 2c.., dim g)
        {
            // lanes 0-7 / 8-15 / 16-23 / 24-31: keys 0-7 chunk q / keys 8-15 chunk q /
            // keys 0-7 chunk q+1 / keys 8-15 chunk q+1
            const uint32_t row = static_cast<uint32_t>(row0 + (lane & 7) + (lane & 8));
            const uint32_t csel = static_cast<uint32_t>(lane >> 4);
#pragma unroll
            for (int qc = 0; qc < ND / 2; ++qc) {  // pairs of 8-dim chunks
                const uint32_t chunk = ((2 * qc) & 7) | csel;
                uint32_t b[4];
                ldsm_x4_trans(b, vbase + ((2 * qc) >> 3) * slice_bytes + row * 128u + ((chunk ^ sw) << 4));
                mma16816<DT>(o[2 * qc], ph, b[0], b[1]);
                mma16816<DT>(o[2 * qc], pl, b[0], b[1]);
                mma16816<DT>(o[2 * qc + 1], ph, b[2], b[3]);
                mma16816<DT>(o[2 * qc + 1], pl, b[2], b[3]);
            }
        }
    }

    // vs: the V scale of an E4M3 cache (the stage holds the codes' values).
    template <bool kScaled>
    __device__ __forceinline__ void finish(const PrefillArgs& a, int64_t tok0, int rows, int head) const {
        const int lane = threadIdx.x & 31;
        const int g = lane >> 2, c = lane & 3;
        float l0 = l[0], l1 = l[1];
#pragma unroll
        for (int off = 1; off <= 2; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
        float i0 = 1.f / l0, i1 = 1.f / l1;
        if constexpr (kScaled) {
            i0 *= a.v_scale;
            i1 *= a.v_scale;
        }
        const int64_t o0 = ((tok0 + g) * a.num_q_heads + head) * D;
        const int64_t o1 = ((tok0 + g + 8) * a.num_q_heads + head) * D;
#pragma unroll
        for (int nd = 0; nd < ND; ++nd) {
            const int d = 8 * nd + 2 * c;
            if (g < rows) {
                store_out(a.out, o0 + d, o[nd][0] * i0, a.out_dtype);
                store_out(a.out, o0 + d + 1, o[nd][1] * i0, a.out_dtype);
            }
            if (g + 8 < rows) {
                store_out(a.out, o1 + d, o[nd][2] * i1, a.out_dtype);
                store_out(a.out, o1 + d + 1, o[nd][3] * i1, a.out_dtype);
            }
        }
    }
};

// E4M3 cache (kFP8, head_dim 128): the producer brings each block's codes
// (a contiguous [bs][128] byte tile of K and one of V) into one of two raw
// slots with a bulk copy, converts them exactly to q's type (every E4M3 value
// is an f16 and a bf16) into the stage in the layout the tensor copies give
// the other types (128-byte swizzle, rows of 64-element slices), and
// completes the stage with a plain arrival.  The consumers are unchanged:
// the K scale is folded into the score multiplier, the V scale into the
// output.
template <int DT>
__device__ __forceinline__ void convert_e4m3_tile(const uint8_t* raw, uint8_t* stage, int bs) {
    using T = typename Elem<DT>::T;
    const int lane = threadIdx.x & 31;
    const uint32_t slice_bytes = static_cast<uint32_t>(bs) * 128u;
    for (int e = lane; e < bs * 16; e += 32) {  // (row, 8-code chunk) of a 128-code row
        const int r = e >> 4, q = e & 15;        // q: the 8-dim chunk, dims 8q .. 8q + 7
        const uint2 codes = *reinterpret_cast<const uint2*>(raw + r * 128 + q * 8);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t word = k < 2 ? codes.x : codes.y;
            const uint32_t h2 = e4m3x2_to_half2(static_cast<uint16_t>(word >> (16 * (k & 1))));
            if constexpr (DT == kF16) {
                w[k] = h2;
            } else {
                const __half2 hh = *reinterpret_cast<const __half2*>(&h2);
                const __nv_bfloat162 b2 = __floats2bfloat162_rn(__low2float(hh), __high2float(hh));
                w[k] = *reinterpret_cast<const uint32_t*>(&b2);
            }
        }
        const int sl = q >> 3, c = q & 7;  // 64-dim slice and chunk within the 128-byte row
        *reinterpret_cast<uint4*>(stage + sl * slice_bytes + r * 128 + ((c ^ (r & 7)) << 4)) =
            make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// G consumer warps (one per query head of the group) + the producer warp;
// the register budget leaves room for several CTAs per SM.
template <int DT, int D, int G, bool kFP8 = false>
__global__ void __launch_bounds__(32 * (1 + G), G <= 4 ? 2 : 1) paged_prefill_kernel(const PrefillArgs a,
                                                                const __grid_constant__ CUtensorMap tmk,
                                                                const __grid_constant__ CUtensorMap tmv) {
    static_assert(!kFP8 || D == 128, "E4M3 rows of 128 codes");
    extern __shared__ uint8_t smem_raw[];
    pdl_allow_next();
    pdl_wait();
    uint8_t* base = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int h = blockIdx.y;
    const int x = blockIdx.x;
    const int tiles = a.tile_cum[a.num_seqs];
    if (x >= tiles) return;
    const int s = find_sequence(a.tile_cum, a.num_seqs, x);
    const int qt = x - a.tile_cum[s];
    const int n = a.query_start[s + 1] - a.query_start[s];
    const int ctx = a.context_lens[s];
    const int rows = min(kQT, n - qt * kQT);
    const int pos0 = ctx - n + qt * kQT;  // position of the tile's first token
    const int last = pos0 + rows - 1;     // the last position any row reads
    const int nblocks = last / a.block_size + 1;
    const int bs = a.block_size;
    const int half = bs * D * static_cast<int>(sizeof(typename Elem<DT>::T));
    const int stage_bytes = 2 * half;
    uint64_t* full = reinterpret_cast<uint64_t*>(base + a.stages * stage_bytes);
    uint64_t* empty = full + a.stages;
    uint64_t* raw_full = empty + a.stages;  // kFP8: the two raw slots' copies
    volatile int* abort = reinterpret_cast<volatile int*>(raw_full + 2);
    uint8_t* raw = base + a.stages * stage_bytes + 1024;  // kFP8: 2 slots x (K, V) x bs x 128 codes
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int st = 0; st < a.stages; ++st) {
            mbar_init(&full[st], 1);
            mbar_init(&empty[st], G);
        }
        mbar_init(&raw_full[0], 1);
        mbar_init(&raw_full[1], 1);
        *abort = 0;
        fence_barrier_init();
        if constexpr (!kFP8) {
            prefetch_tensor_map(&tmk);
            prefetch_tensor_map(&tmv);
        }
    }
    __syncthreads();
    if (kFP8 && warp == 0) {
        // ---- producer (E4M3): bulk copies into the raw slots, conversion into the stages
        const uint64_t policy = policy_evict_last();
        const uint32_t tile = static_cast<uint32_t>(bs) * 128u;  // one (block, head) tile of codes
        auto block_of = [&](int j) {
            int blk = a.block_tables[static_cast<int64_t>(s) * a.max_blocks + j];
            if (blk < 0 || blk >= a.num_blocks) {
                raise_flag(a.status, kFlagBadBlock);
                blk = 0;
            }
            return blk;
        };
        auto fetch = [&](int j) {  // block j's K and V codes into raw slot j % 2 (lane 0)
            uint8_t* dst = raw + (j & 1) * 2 * tile;
            fence_proxy_async_smem();  // the slot's last reads (generic) before the copy (async)
            const int64_t off = (static_cast<int64_t>(block_of(j)) * a.num_kv_heads + h) * tile;
            mbar_arrive_expect_tx(&raw_full[j & 1], 2 * tile);
            bulk_load(dst, static_cast<const uint8_t*>(a.k_cache) + off, tile, &raw_full[j & 1], policy);
            bulk_load(dst + tile, static_cast<const uint8_t*>(a.v_cache) + off, tile, &raw_full[j & 1], policy);
        };
        int fetched = 0;  // raw copies issued (lane 0)
        if (lane == 0 && nblocks > 0) {
            fetch(0);
            fetched = 1;
        }
        for (int j = 0; j < nblocks; ++j) {
            const int stage = j % a.stages;
            int good = 1;
            if (lane == 0) {
                if (j + 1 < nblocks) {  // the next block's codes, into the slot block j - 1 left
                    fetch(j + 1);
                    ++fetched;
                }
                if (j >= a.stages)
                    good = mbar_wait_bounded(&empty[stage], ((j / a.stages) - 1) & 1, abort, a.status);
                if (good) good = mbar_wait_bounded(&raw_full[j & 1], (j >> 1) & 1, abort, a.status);
            }
            good = __shfl_sync(0xffffffffu, good, 0);
            if (!good) break;
            uint8_t* kd = base + stage * stage_bytes;
            convert_e4m3_tile<DT>(raw + (j & 1) * 2 * tile, kd, bs);
            convert_e4m3_tile<DT>(raw + (j & 1) * 2 * tile + tile, kd + half, bs);
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[stage]);
        }
        // Every raw copy issued must land before the CTA exits (bounded).
        if (lane == 0) {
            for (int sl = 0; sl < 2 && sl < fetched; ++sl) {
                const int lastj = sl + ((fetched - 1 - sl) / 2) * 2;
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&raw_full[sl], (lastj >> 1) & 1)) {
                    if (global_timer_ns() - t0 > kWaitLimitNs) {
                        raise_flag(a.status, kFlagTimeout);
                        break;
                    }
                }
            }
        }
        return;
    }
    if (warp == 0) {
        // ---- producer: K and V tiles of blocks 0 .. nblocks-1 of head h
        const uint64_t policy = policy_evict_last();
        int issued = 0;
        bool ok = true;
        for (int jb = 0; jb < nblocks && ok; jb += 32) {
            int blk = 0;
            if (jb + lane < nblocks) {
                blk = __ldg(a.block_tables + static_cast<int64_t>(s) * a.max_blocks + jb + lane);
                if (blk < 0 || blk >= a.num_blocks) {
                    raise_flag(a.status, kFlagBadBlock);
                    blk = 0;
                }
            }
            const int cnt = min(32, nblocks - jb);
            for (int k = 0; k < cnt; ++k) {
                const int bk = __shfl_sync(0xffffffffu, blk, k);
                int good = 1;
                if (lane == 0) {
                    const int j = jb + k;
                    const int stage = j % a.stages;
                    if (j >= a.stages)
                        good = mbar_wait_bounded(&empty[stage], ((j / a.stages) - 1) & 1, abort, a.status);
                    if (good) {
                        uint8_t* kd = base + stage * stage_bytes;
                        uint8_t* vd = kd + half;
                        mbar_arrive_expect_tx(&full[stage], stage_bytes);
                        const int rowk = (bk * a.num_kv_heads + h) * bs;
                        for (int sl = 0; sl < D / 64; ++sl) {
                            tensor_load_2d(kd + sl * (half / (D / 64)), &tmk, sl * 64, rowk, &full[stage], policy);
                            tensor_load_2d(vd + sl * (half / (D / 64)), &tmv, sl * 64, rowk, &full[stage], policy);
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
        // Wait (bounded) for every copy issued, so none outlives the CTA.
        if (lane == 0) {
            for (int st = 0; st < a.stages && st < issued; ++st) {
                const int lastj = st + ((issued - 1 - st) / a.stages) * a.stages;
                const uint64_t t0 = global_timer_ns();
                while (!mbar_try_wait(&full[st], (lastj / a.stages) & 1)) {
                    if (global_timer_ns() - t0 > kWaitLimitNs) {
                        raise_flag(a.status, kFlagTimeout);
                        break;
                    }
                }
            }
        }
        return;
    }
    // ---- consumers: warp 1 + w computes query head h*G + w
    const int w = warp - 1;
    const int head = h * G + w;
    const int64_t tok0 = a.query_start[s] + static_cast<int64_t>(qt) * kQT;
    PrefillTile<DT, D> t;
    t.begin(a, tok0, rows, head, pos0);
    const uint32_t slice_bytes = static_cast<uint32_t>(bs) * 128u;
    for (int j = 0; j < nblocks; ++j) {
        const int stage = j % a.stages;
        const bool ok = mbar_wait_bounded(&full[stage], (j / a.stages) & 1, abort, a.status);
        if (ok) {
            uint8_t* kt = base + stage * stage_bytes;
            const uint32_t kb = smem_addr(kt);
            const uint32_t vb = kb + half;
            const int kvalid = min(bs, ctx - j * bs);
            // Rows past the sequence's last token may hold any value (even
            // NaN): zero them in V so that 0 * V stays 0.  Every consumer
            // warp writes the same zeros before reading.
            const bool tail = kvalid < bs;
            if (tail) {
                for (int e = lane; e < (bs - kvalid) * (D / 8); e += 32) {
                    const int r = kvalid + e / (D / 8), q = e % (D / 8);  // 16-byte chunk q of row r
                    *reinterpret_cast<uint4*>(kt + half + (q >> 3) * bs * 128 + r * 128 +
                                              (((q & 7) ^ (r & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                }
                __syncwarp();
            }
            for (int sl = 0; sl * 16 < kvalid; ++sl) {
                const int kpos0 = j * bs + sl * 16;
                if (kpos0 > last) break;
                t.slice(a, kb, vb, slice_bytes, sl * 16, kpos0);
            }
            if (tail) fence_proxy_async_smem();  // generic writes before the next TMA fill
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[stage]);
    }
    if (!*abort) t.template finish<kFP8>(a, tok0, rows, head);
}

template <int DT, int D, int G, bool kFP8>
cudaError_t launch_prefill_g(const PrefillArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                             cudaStream_t stream) {
    static std::atomic<int> configured[64];
    auto kern = paged_prefill_kernel<DT, D, G, kFP8>;
    const bool cacheable = a.device >= 0 && a.device < 64;
    if (!cacheable || configured[a.device].load() < a.smem_bytes) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, a.smem_bytes);
        if (e != cudaSuccess) return e;
        if (cacheable) configured[a.device].store(a.smem_bytes);
    }
    return launch_kernel(kern, dim3(a.grid_tiles, a.num_kv_heads), dim3(32 * (1 + G)),
                         static_cast<size_t>(a.smem_bytes), stream, a.pdl != 0, a, tmk, tmv);
}

template <int DT, int D, bool kFP8 = false>
cudaError_t launch_prefill_t(const PrefillArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                             cudaStream_t stream) {
    switch (a.num_q_heads / a.num_kv_heads) {
        case 1: return launch_prefill_g<DT, D, 1, kFP8>(a, tmk, tmv, stream);
        case 2: return launch_prefill_g<DT, D, 2, kFP8>(a, tmk, tmv, stream);
        case 4: return launch_prefill_g<DT, D, 4, kFP8>(a, tmk, tmv, stream);
        case 8: return launch_prefill_g<DT, D, 8, kFP8>(a, tmk, tmv, stream);
    }
    return cudaErrorInvalidValue;
}

// f32 q and cache: one warp per (new token, query head), the token's causal
// prefix one key at a time on the CUDA cores (lane l holds dims VD*l ..
// VD*l + VD - 1; the dot product reduced across the warp), online softmax in
// base 2.  A sequence whose chunk is longer than its context, or whose context
// exceeds its table, writes nothing (the plan kernel flags it).
template <int D>
__global__ void __launch_bounds__(256) paged_prefill_f32_kernel(const PrefillArgs a) {
    constexpr int VD = D / 32;
    pdl_allow_next();
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (row >= static_cast<int64_t>(a.num_tokens) * a.num_q_heads) return;
    const int64_t tok = row / a.num_q_heads;
    const int g = static_cast<int>(row - tok * a.num_q_heads);
    const int h = g / (a.num_q_heads / a.num_kv_heads);
    int lo = 0, hi = a.num_seqs;  // the sequence of the token: largest s with query_start[s] <= tok
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (a.query_start[mid] <= tok) lo = mid; else hi = mid;
    }
    const int s = lo;
    const int n = a.query_start[s + 1] - a.query_start[s];
    const int ctx = a.context_lens[s];
    if (n <= 0 || n > ctx || ctx > a.max_blocks * a.block_size) return;
    const int pos = ctx - n + static_cast<int>(tok - a.query_start[s]);
    const float* qrow = static_cast<const float*>(a.q) + row * D + VD * lane;
    float q[VD], o[VD];
#pragma unroll
    for (int i = 0; i < VD; ++i) {
        q[i] = qrow[i] * a.scale_log2;
        o[i] = 0.f;
    }
    float m = -INFINITY, l = 0.f;
    const float* kc = static_cast<const float*>(a.k_cache);
    const float* vc = static_cast<const float*>(a.v_cache);
    for (int t = 0; t <= pos; ++t) {
        int blk = a.block_tables[static_cast<int64_t>(s) * a.max_blocks + t / a.block_size];
        if (blk < 0 || blk >= a.num_blocks) {
            if (lane == 0) raise_flag(a.status, kFlagBadBlock);
            blk = 0;
        }
        const int64_t r = (static_cast<int64_t>(blk) * a.num_kv_heads + h) * a.block_size + t % a.block_size;
        const float* k = kc + r * D + VD * lane;
        const float* v = vc + r * D + VD * lane;
        float x = 0.f;
#pragma unroll
        for (int i = 0; i < VD; ++i) x = fmaf(q[i], __ldg(k + i), x);
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
        const float mn = fmaxf(m, x);
        const float al = fast_exp2(m - mn);  // 0 while m is -inf
        const float p = fast_exp2(x - mn);
        l = fmaf(l, al, p);
#pragma unroll
        for (int i = 0; i < VD; ++i) o[i] = fmaf(o[i], al, p * __ldg(v + i));
        m = mn;
    }
    const float inv = 1.f / l;
    float* out = static_cast<float*>(a.out) + row * D + VD * lane;
#pragma unroll
    for (int i = 0; i < VD; ++i) out[i] = o[i] * inv;
}

cudaError_t launch_prefill_f32(const PrefillArgs& a, cudaStream_t stream) {
    const int64_t warps = static_cast<int64_t>(a.num_tokens) * a.num_q_heads;
    const int blocks = static_cast<int>((warps + 7) / 8);
    if (a.head_dim == 64) return launch_kernel(paged_prefill_f32_kernel<64>, dim3(blocks), dim3(256), 0, stream,
                                               a.pdl != 0, a);
    if (a.head_dim == 128) return launch_kernel(paged_prefill_f32_kernel<128>, dim3(blocks), dim3(256), 0, stream,
                                                a.pdl != 0, a);
    return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                           cudaStream_t stream) {
    if (a.num_seqs == 0 || a.num_tokens == 0) return cudaSuccess;
    cudaError_t e = launch_kernel(prefill_plan_kernel, dim3(1), dim3(1024), 0, stream, a.pdl != 0, a);
    if (e != cudaSuccess) return e;
    if (a.kv_dtype == kFP8) {
        if (a.head_dim != 128) return cudaErrorInvalidValue;
        if (a.dtype == kF16) return launch_prefill_t<kF16, 128, true>(a, tmk, tmv, stream);
        if (a.dtype == kBF16) return launch_prefill_t<kBF16, 128, true>(a, tmk, tmv, stream);
        return cudaErrorInvalidValue;
    }
    if (a.dtype == kF32) return launch_prefill_f32(a, stream);
    if (a.tensor_cores) return launch_prefill_tc(a, tmk, tmv, stream);
    if (a.dtype == kF16) {
        if (a.head_dim == 64) return launch_prefill_t<kF16, 64>(a, tmk, tmv, stream);
        if (a.head_dim == 128) return launch_prefill_t<kF16, 128>(a, tmk, tmv, stream);
    } else if (a.dtype == kBF16) {
        if (a.head_dim == 64) return launch_prefill_t<kBF16, 64>(a, tmk, tmv, stream);
        if (a.head_dim == 128) return launch_prefill_t<kBF16, 128>(a, tmk, tmv, stream);
    }
    return cudaErrorInvalidValue;
}

// Slot of every new token: token i of sequence s at position context_lens[s] - n_s + i.
__global__ void __launch_bounds__(128) kv_slot_mapping_varlen_kernel(const PrefillArgs a, int32_t* slots) {
    pdl_allow_next();
    pdl_wait();
    const int s = blockIdx.x;
    if (s >= a.num_seqs) return;
    const int q0 = a.query_start[s], q1 = a.query_start[s + 1];
    const int n = q1 - q0, ctx = a.context_lens[s];
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int pos = ctx - n + i;
        int32_t slot = -1;
        const int j = pos >= 0 ? pos / a.block_size : -1;
        if (pos < 0 || j >= a.max_blocks) {
            raise_flag(a.status, kFlagBadContext);
        } else {
            const int blk = a.block_tables[static_cast<int64_t>(s) * a.max_blocks + j];
            if (blk < 0 || blk >= a.num_blocks)
                raise_flag(a.status, kFlagBadBlock);
            else
                slot = blk * a.block_size + (pos - j * a.block_size);
        }
        if (q0 + i < a.num_tokens) slots[q0 + i] = slot;
    }
}

cudaError_t launch_slot_mapping_varlen(const PrefillArgs& a, int32_t* slots, cudaStream_t stream) {
    if (a.num_seqs == 0) return cudaSuccess;
    return launch_kernel(kv_slot_mapping_varlen_kernel, dim3(a.num_seqs), dim3(128), 0, stream,
                         a.pdl != 0, a, slots);
}

}  // namespace pkv
