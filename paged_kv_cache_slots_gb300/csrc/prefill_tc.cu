// Multi-token queries over the paged cache on the fifth-generation tensor
// cores (tcgen05): the same operation as prefill.cu ("Batching and
// Scheduling", Example 5; "vLLM Architecture and Installation", Example 5),
// for head_dim 128.
//
// A CTA takes 128 rows: 128/G new tokens of one sequence times the G query
// heads that share KV head h (row r = token r / G, head h*G + r % G), and
// walks the keys 0 .. (its last token's position) in tiles of 64:
//   warp 4      streams the tile's K rows into a ring of 3 stages and its V
//               rows into a ring of 2 (128-byte swizzle; TMA boxes for
//               blocks of 64 tokens or more, per-lane 16-byte copies for
//               shorter blocks);
//   warp 5      (one lane) issues S = Q . K^T (M 128, N 64, K 128) into one of
//               two tensor-memory buffers, and O += P . V (M 128, N 128,
//               K 64) into tensor memory with P read from tensor memory (a
//               high and a low half-precision part written over the S buffer
//               it came from) and V read MN-major from its stage;
//   warps 0-3   one row each: load the row of S from tensor memory, causal
//               mask, online softmax (base 2) with a lazy rescale of O (only
//               when the row's maximum grows by more than 2^8; the exponent
//               reference stays fixed otherwise, so P <= 256), write P, and
//               at the end O / l.
// Shared memory (112 KiB) and tensor memory (256 columns) are sized so that
// two CTAs share an SM: each SM sub-partition then runs two softmax warps.
// Every hand-off is an mbarrier with a bounded wait; the ones that recur per
// tile are doubled per buffer so that a wait can never see a phase two steps
// old.
#include "decode_kernel.cuh"
#include "mma_frag.cuh"
#include "tc_utils.cuh"

namespace pkv {

namespace {

constexpr int kBM = 128;                        // rows per CTA
constexpr int kNK = 64;                         // keys per key tile
constexpr int kDim = 128;
constexpr int kKRing = 3;                       // K stages
constexpr int kVRing = 2;                       // V stages
constexpr uint32_t kHalf = 2 * kNK * 128;       // K (or V) of a key tile: 2 slices of 64 dims, 16 KiB
constexpr uint32_t kQOff = 0;                   // Q: 2 slices x 128 rows x 128 B
constexpr uint32_t kKOff = 2 * kBM * 128;       // 32 KiB
constexpr uint32_t kVOff = kKOff + kKRing * kHalf;   // 80 KiB
constexpr uint32_t kBarOff = kVOff + kVRing * kHalf; // 112 KiB
constexpr uint32_t kTmemCols = 256;             // S / P buffers (2 x 64) + O (128)
constexpr float kLazy = 8.f;

struct Bars {
    uint64_t kfull[kKRing], kempty[kKRing], vfull[kVRing], vempty[kVRing];
    uint64_t s_full[2], p_full[2], pv_done[2];
    uint32_t tmem;
    int abort;
};

__device__ __forceinline__ bool wait(uint64_t* bar, uint32_t parity, volatile int* abort, uint32_t* status) {
    return mbar_wait_bounded(bar, parity & 1u, abort, status);
}

// kBS 16 or 32: blocks shorter than a key tile, loaded by the producer warp's
// lanes with 16-byte cp.async copies (one TMA box per (block, 64-dim slice)
// would cost 16 boxes per 64-key tile at 16-token blocks); kBS 0: blocks of a
// multiple of 64 tokens, loaded by TMA.
template <int DT, int G, int kBS>
__global__ void __launch_bounds__(192, 2) paged_prefill_tc_kernel(const PrefillArgs a,
                                                                   const __grid_constant__ CUtensorMap tmk,
                                                                   const __grid_constant__ CUtensorMap tmv) {
    using T = typename Elem<DT>::T;
    constexpr int TPT = kBM / G;  // new tokens per CTA
    constexpr bool kLanes = kBS != 0;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    pdl_allow_next();
    pdl_wait();
    // The swizzled layouts need a 1024-byte aligned base; the launch reserves
    // no slack for re-alignment (two CTAs per SM), so a misaligned window is
    // reported rather than overrun.
    if (smem_addr(smem_raw) & 1023u) {
        if (threadIdx.x == 0) raise_flag(a.status, kFlagBadPlan);
        return;
    }
    uint8_t* base = smem_raw;
    Bars* B = reinterpret_cast<Bars*>(base + kBarOff);
    volatile int* abort = &B->abort;
    const int h = blockIdx.y;
    const int x = blockIdx.x;
    if (x >= a.tile_cum[a.num_seqs]) return;
    const int s = find_sequence(a.tile_cum, a.num_seqs, x);
    const int qt = x - a.tile_cum[s];
    const int n = a.query_start[s + 1] - a.query_start[s];
    const int ctx = a.context_lens[s];
    const int ntok = min(TPT, n - qt * TPT);
    const int pos0 = ctx - n + qt * TPT;
    const int last = pos0 + ntok - 1;
    const int nkt = last / kNK + 1;
    const int64_t tok0 = a.query_start[s] + static_cast<int64_t>(qt) * TPT;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    if (tid == 0) {
        // one arrival per producer lane (cp.async), or the TMA byte count
        for (int i = 0; i < kKRing; ++i) {
            mbar_init(&B->kfull[i], kLanes ? 32 : 1);
            mbar_init(&B->kempty[i], 1);
        }
        for (int i = 0; i < kVRing; ++i) {
            mbar_init(&B->vfull[i], kLanes ? 32 : 1);
            mbar_init(&B->vempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&B->s_full[i], 1);
            mbar_init(&B->p_full[i], 4);
            mbar_init(&B->pv_done[i], 1);
        }
        B->abort = 0;
        fence_barrier_init();
        if constexpr (!kLanes) {
            prefetch_tensor_map(&tmk);
            prefetch_tensor_map(&tmv);
        }
    }
    if (warp == 0) tc_alloc(&B->tmem, kTmemCols);
    if (warp < 4) {  // Q rows into shared memory, 128-byte swizzled K-major
        const int r = tid;
        const int tr = min(r / G, ntok - 1);
        const T* qrow = static_cast<const T*>(a.q) + ((tok0 + tr) * a.num_q_heads + h * G + r % G) * kDim;
        // A negative scale is applied as |scale| to the scores of -q (a sign
        // flip is exact), so the row maximum is taken on unscaled scores.
        const uint32_t flip = a.scale_log2 < 0.f ? 0x80008000u : 0u;
#pragma unroll
        for (int q16 = 0; q16 < 16; ++q16) {
            uint4 v = *reinterpret_cast<const uint4*>(qrow + 8 * q16);
            v.x ^= flip;
            v.y ^= flip;
            v.z ^= flip;
            v.w ^= flip;
            *reinterpret_cast<uint4*>(base + kQOff + (q16 >> 3) * (kBM * 128) + r * 128 +
                                      (((q16 & 7) ^ (r & 7)) << 4)) = v;
        }
        fence_proxy_async_smem();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t taddr = B->tmem;

    if (warp == 4) {
        // ---- producer: K rows of key tile i, then V rows of tile i - 1 (K runs
        // one tile ahead: S of a tile is issued before its PV).
        const int bs = a.block_size;
        const int nblk = (ctx + bs - 1) / bs;
        auto block_of = [&](int lb) -> int {
            int blk = a.block_tables[static_cast<int64_t>(s) * a.max_blocks + (lb < nblk ? lb : 0)];
            if (blk < 0 || blk >= a.num_blocks) {
                raise_flag(a.status, kFlagBadBlock);
                blk = 0;
            }
            return blk;
        };
        int kiss = 0, viss = 0;
        if constexpr (kLanes) {
            // Blocks of kBS = 16 or 32 tokens.  Lane e copies the 16-byte chunk
            // e % 8 of the tile's rows e / 8 + 4 q (both 64-dim slices) into the
            // 128-byte swizzled layout the tensor copies produce; row e / 8 + 4 q
            // lies in block q / (kBS / 4), so every address is a per-lane base
            // plus a constant.
            constexpr int kBlk = kNK / kBS;
            constexpr int kRows = kBS / 4;  // this lane's rows per block
            const int ch = lane & 7, l8 = lane >> 3;
            const int64_t lane_src = l8 * (kDim * 2) + ch * 16;
            const uint32_t lane_dst = l8 * 128;
            const uint32_t sw0 = static_cast<uint32_t>(ch ^ l8) << 4, sw1 = static_cast<uint32_t>(ch ^ (l8 + 4)) << 4;
            auto load = [&](int j, const void* cache, uint32_t dst, uint64_t* bar) {
                const char* c0 = static_cast<const char*>(cache) + lane_src;
#pragma unroll
                for (int bb = 0; bb < kBlk; ++bb) {
                    const char* src =
                        c0 + (static_cast<int64_t>(block_of(j * kBlk + bb)) * a.num_kv_heads + h) * (kBS * kDim * 2);
#pragma unroll
                    for (int q = 0; q < kRows; ++q) {
                        const int r = bb * kRows + q;
                        const uint32_t d = dst + lane_dst + r * 512 + ((r & 1) ? sw1 : sw0);
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d), "l"(src + q * 1024)
                                     : "memory");
                        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(d + kNK * 128),
                                     "l"(src + q * 1024 + 128)
                                     : "memory");
                    }
                }
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
            };
            for (int i = 0; i <= nkt; ++i) {
                if (i < nkt) {
                    if (i >= kKRing &&
                        !__all_sync(0xffffffffu, wait(&B->kempty[i % kKRing], i / kKRing - 1, abort, a.status)))
                        break;
                    load(i, a.k_cache, smem_addr(base + kKOff + (i % kKRing) * kHalf), &B->kfull[i % kKRing]);
                    ++kiss;
                }
                if (i >= 1) {
                    const int j = i - 1;
                    if (j >= kVRing &&
                        !__all_sync(0xffffffffu, wait(&B->vempty[j % kVRing], j / kVRing - 1, abort, a.status)))
                        break;
                    load(j, a.v_cache, smem_addr(base + kVOff + (j % kVRing) * kHalf), &B->vfull[j % kVRing]);
                    ++viss;
                }
            }
            // Every copy issued must land before the CTA can exit.
            asm volatile("cp.async.wait_all;" ::: "memory");
        } else if (lane == 0) {
            const uint64_t policy = policy_evict_last();
            auto load = [&](int j, const CUtensorMap* map, uint8_t* dst, uint64_t* bar) {
                // Blocks of a multiple of 64 tokens: one block holds the whole tile.
                mbar_arrive_expect_tx(bar, kHalf);
                const int key0 = j * kNK;
                const int lb = key0 / bs;
                const int y = (block_of(lb) * a.num_kv_heads + h) * bs + (key0 - lb * bs);
                for (int sl = 0; sl < 2; ++sl) tensor_load_2d(dst + sl * (kNK * 128), map, sl * 64, y, bar, policy);
            };
            for (int i = 0; i <= nkt; ++i) {
                if (i < nkt) {
                    if (i >= kKRing && !wait(&B->kempty[i % kKRing], i / kKRing - 1, abort, a.status)) break;
                    load(i, &tmk, base + kKOff + (i % kKRing) * kHalf, &B->kfull[i % kKRing]);
                    ++kiss;
                }
                if (i >= 1) {
                    const int j = i - 1;
                    if (j >= kVRing && !wait(&B->vempty[j % kVRing], j / kVRing - 1, abort, a.status)) break;
                    load(j, &tmv, base + kVOff + (j % kVRing) * kHalf, &B->vfull[j % kVRing]);
                    ++viss;
                }
            }
            // Every copy issued must land before the CTA can exit.
            auto drain = [&](uint64_t* bars, int ring, int issued) {
                for (int st = 0; st < ring && st < issued; ++st) {
                    const int lastj = st + ((issued - 1 - st) / ring) * ring;
                    const uint64_t t0 = global_timer_ns();
                    while (!mbar_try_wait(&bars[st], (lastj / ring) & 1)) {
                        if (global_timer_ns() - t0 > kWaitLimitNs) {
                            raise_flag(a.status, kFlagTimeout);
                            break;
                        }
                    }
                }
            };
            drain(B->kfull, kKRing, kiss);
            drain(B->vfull, kVRing, viss);
        }
        __syncwarp();
    } else if (warp == 5) {
        // ---- MMA issue (one lane)
        if (lane == 0) {
            constexpr int bf = DT == kBF16 ? 1 : 0;
            constexpr uint32_t idS = tc_idesc_f16(bf, false, kNK, kBM);
            constexpr uint32_t idPV = tc_idesc_f16(bf, true, kDim, kBM);
            const uint32_t qa = smem_addr(base + kQOff);
            auto pv = [&](int t) -> bool {
                const int sv = t % kVRing, bt = t & 1;
                if (!wait(&B->p_full[bt], t >> 1, abort, a.status)) return false;
                if (!wait(&B->vfull[sv], t / kVRing, abort, a.status)) return false;
                if constexpr (kLanes) fence_proxy_async_smem();  // lane copies before the tensor cores read them
                tc_fence_after();
                const uint32_t va = smem_addr(base + kVOff + sv * kHalf);
#pragma unroll
                for (int part = 0; part < 2; ++part)
#pragma unroll
                    for (int kk = 0; kk < kNK / 16; ++kk)
                        tc_mma_ts(taddr + 128, taddr + bt * kNK + part * 32 + kk * 8,
                                  tc_sdesc(va + kk * 16 * 128, kNK * 128, 1024), idPV,
                                  !(t == 0 && part == 0 && kk == 0));
                tc_commit(&B->pv_done[bt]);
                tc_commit(&B->vempty[sv]);
                return true;
            };
            bool ok = true;
            for (int j = 0; j < nkt && ok; ++j) {
                const int sk = j % kKRing, b = j & 1;
                ok = wait(&B->kfull[sk], j / kKRing, abort, a.status);
                // S buffer b holds P of tile j - 2 until that PV has completed.
                if (ok && j >= 2) ok = wait(&B->pv_done[b], (j >> 1) - 1, abort, a.status);
                if (!ok) break;
                if constexpr (kLanes) fence_proxy_async_smem();
                tc_fence_after();
                const uint32_t ka = smem_addr(base + kKOff + sk * kHalf);
#pragma unroll
                for (int ks = 0; ks < kDim / 16; ++ks)
                    tc_mma(taddr + b * kNK, tc_sdesc(qa + (ks >> 2) * (kBM * 128) + (ks & 3) * 32, 16, 1024),
                           tc_sdesc(ka + (ks >> 2) * (kNK * 128) + (ks & 3) * 32, 16, 1024), idS, ks > 0);
                tc_commit(&B->s_full[b]);
                tc_commit(&B->kempty[sk]);
                if (j >= 1) ok = pv(j - 1);
            }
            if (ok) pv(nkt - 1);
        }
        __syncwarp();
    } else {
        // ---- softmax: thread r owns row r (tensor-memory lane r)
        const int r = tid;
        const int tr = r / G;
        const int qpos = pos0 + min(tr, ntok - 1);
        const uint32_t lane_base = taddr + (static_cast<uint32_t>(32 * warp) << 16);
        float m_ref = -INFINITY, l = 0.f;
        // |scale| in log2 units; a zero scale is taken as 1e-30, which leaves
        // every finite score's exponent at 0 while masked scores stay -inf.
        const float sc = fmaxf(fabsf(a.scale_log2), 1e-30f);
        bool ok = true;
        for (int j = 0; j < nkt && ok; ++j) {
            const int b = j & 1;
            ok = __all_sync(0xffffffffu, wait(&B->s_full[b], j >> 1, abort, a.status));
            if (!ok) break;
            tc_fence_after();
            float sv[kNK];
            {
                float t0[32], t1[32];
                tc_ld32(lane_base + b * kNK, t0);
                tc_ld32(lane_base + b * kNK + 32, t1);
                tc_wait_ld();
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    sv[c] = t0[c];
                    sv[32 + c] = t1[c];
                }
            }
            const int kbase = j * kNK;
            if (kbase + kNK - 1 > pos0) {  // a key of this tile lies past some row's position
#pragma unroll
                for (int c = 0; c < kNK; ++c) sv[c] = kbase + c <= qpos ? sv[c] : -INFINITY;
            }
            // Row maximum as eight independent chains (short dependency path).
            float mx[8];
#pragma unroll
            for (int c = 0; c < 8; ++c) mx[c] = sv[c];
#pragma unroll
            for (int c = 8; c < kNK; ++c) mx[c & 7] = fmaxf(mx[c & 7], sv[c]);
            const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                                   fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) *
                             sc;
            bool need = false;
            if (j == 0) {
                m_ref = mt;  // key 0 is visible to every row
            } else {
                need = mt > m_ref + kLazy;
            }
            if (__any_sync(0xffffffffu, need)) {
                // O must be complete up to tile j-1 before it is rescaled.
                ok = __all_sync(0xffffffffu, wait(&B->pv_done[(j - 1) & 1], (j - 1) >> 1, abort, a.status));
                if (!ok) break;
                tc_fence_after();
                const float f = need ? fast_exp2(m_ref - mt) : 1.f;
                if (need) {
                    l *= f;
                    m_ref = mt;
                }
#pragma unroll
                for (int cb = 0; cb < kDim / 32; ++cb) {
                    float o[32];
                    tc_ld32(lane_base + 128 + 32 * cb, o);
                    tc_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] *= f;
                    tc_st32(lane_base + 128 + 32 * cb, o);
                }
                tc_wait_st();
            }
            // P over the S buffer it came from: columns 0-31 the high part,
            // 32-63 the low part, keys 2c and 2c + 1 in column c.
            float ps[4] = {0.f, 0.f, 0.f, 0.f};
            {
                uint32_t hi[32], lo[32];
#pragma unroll
                for (int c = 0; c < kNK / 2; ++c) {
                    const float p0 = fast_exp2(fmaf(sv[2 * c], sc, -m_ref));
                    const float p1 = fast_exp2(fmaf(sv[2 * c + 1], sc, -m_ref));
                    ps[c & 3] += p0 + p1;
                    pack_split<DT>(p0, p1, hi[c], lo[c]);
                }
                tc_st32u(lane_base + b * kNK, hi);
                tc_st32u(lane_base + b * kNK + 32, lo);
            }
            l += (ps[0] + ps[1]) + (ps[2] + ps[3]);
            // Keys past the sequence's last token may hold any value in V (even
            // NaN): zero those rows of the last tile's V so that 0 * V stays 0.
            if (kbase + kNK > ctx) {
                ok = __all_sync(0xffffffffu, wait(&B->vfull[j % kVRing], j / kVRing, abort, a.status));
                if (!ok) break;
                const int from = ctx - kbase;
                uint8_t* vd = base + kVOff + (j % kVRing) * kHalf;
                for (int e = r; e < (kNK - from) * 16; e += kBM) {
                    const int row = from + e / 16, q16 = e % 16;
                    *reinterpret_cast<uint4*>(vd + (q16 >> 3) * (kNK * 128) + row * 128 +
                                              (((q16 & 7) ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            tc_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&B->p_full[b]);  // one arrival per warp (count 4)
        }
        if (__all_sync(0xffffffffu, ok && !*abort)) {
            ok = __all_sync(0xffffffffu, wait(&B->pv_done[(nkt - 1) & 1], (nkt - 1) >> 1, abort, a.status));
            tc_fence_after();
            const float inv = 1.f / l;
            const bool row_ok = ok && tr < ntok;
            const int64_t o0 = ((tok0 + tr) * a.num_q_heads + h * G + r % G) * kDim;
#pragma unroll
            for (int cb = 0; cb < kDim / 32; ++cb) {
                float o[32];
                tc_ld32(lane_base + 128 + 32 * cb, o);
                tc_wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int c = 0; c < 32; ++c) store_out(a.out, o0 + 32 * cb + c, o[c] * inv, a.out_dtype);
                }
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tc_dealloc(taddr, kTmemCols);
    }
}

template <int DT, int G, int kBS>
cudaError_t launch_tc_l(const PrefillArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t stream) {
    static std::atomic<int> configured[64];
    auto kern = paged_prefill_tc_kernel<DT, G, kBS>;
    const bool cacheable = a.device >= 0 && a.device < 64;
    if (!cacheable || configured[a.device].load() < a.smem_bytes) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, a.smem_bytes);
        if (e != cudaSuccess) return e;
        if (cacheable) configured[a.device].store(a.smem_bytes);
    }
    return launch_kernel(kern, dim3(a.grid_tiles, a.num_kv_heads), dim3(192), static_cast<size_t>(a.smem_bytes),
                         stream, a.pdl != 0, a, tmk, tmv);
}

template <int DT, int G>
cudaError_t launch_tc_g(const PrefillArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t stream) {
    if (a.block_size == 16) return launch_tc_l<DT, G, 16>(a, tmk, tmv, stream);
    if (a.block_size == 32) return launch_tc_l<DT, G, 32>(a, tmk, tmv, stream);
    if (a.block_size % kNK == 0) return launch_tc_l<DT, G, 0>(a, tmk, tmv, stream);
    return cudaErrorInvalidValue;
}

template <int DT>
cudaError_t launch_tc_t(const PrefillArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv, cudaStream_t stream) {
    switch (a.num_q_heads / a.num_kv_heads) {
        case 1: return launch_tc_g<DT, 1>(a, tmk, tmv, stream);
        case 2: return launch_tc_g<DT, 2>(a, tmk, tmv, stream);
        case 4: return launch_tc_g<DT, 4>(a, tmk, tmv, stream);
        case 8: return launch_tc_g<DT, 8>(a, tmk, tmv, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace

int prefill_tc_smem_bytes() { return static_cast<int>(kBarOff + sizeof(Bars)); }

cudaError_t launch_prefill_tc(const PrefillArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              cudaStream_t stream) {
    if (a.head_dim != kDim) return cudaErrorInvalidValue;
    if (a.dtype == kBF16) return launch_tc_t<kBF16>(a, tmk, tmv, stream);
    if (a.dtype == kF16) return launch_tc_t<kF16>(a, tmk, tmv, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
