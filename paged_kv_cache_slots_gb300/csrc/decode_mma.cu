// Warp-level tensor-core consumer of the split-context decode kernel
// (f16/bf16 K/V, head_dim 64 or 128, block_size a multiple of 16, up to 8
// query heads per KV head).
//
// Per 16-token slice of a tile:
//   S^T[16 tok x 8 heads] = K[16 x D] . Q^T[D x 8]      (mma m16n8k16, fp32 acc)
//   online softmax per head on the fp32 scores (base-2 units)
//   O^T[D x 8 heads]     += V^T[D x 16 tok] . P^T[16 x 8]
// Tokens are the M dimension, so one tile of K feeds the MMA A operand
// straight from shared memory (ldmatrix), the G <= 8 heads of the group are
// the N dimension (padded to 8) and q stays in registers as B fragments.
// P^T is formed from the score accumulators with movmatrix (transpose in
// registers) and split into a high and a low half-precision part, so the
// probabilities carry ~16 significant bits into the PV product.  With up to
// 4 query heads per KV head the low parts travel in the padding columns 4-7
// of the same MMA (one PV MMA per slice instead of two).
// K and V tiles arrive through 2-D tensor maps with a 128-byte swizzle, which
// makes the eight 16-byte rows of every ldmatrix fall in distinct banks.
#include "decode_kernel.cuh"
#include "mma_frag.cuh"

namespace pkv {

template <int DT, int D, int kMaxT = 32 * 16>
struct MmaPolicy {
    static constexpr int kMaxThreads = kMaxT;
    static constexpr bool kTensor = true;
    static constexpr bool kScratch = false;
    static constexpr bool kPairs = false;
    static constexpr int KS = D / 16;  // k-steps of QK, m-tiles of PV
    static constexpr int kD = D;
    using T = typename Elem<DT>::T;

    struct State {
        uint32_t qb[KS][2];  // B fragments of Q^T: head lane/4, dims 16ks + 2(lane%4) (+8)
        float o[KS][4];      // O^T accumulators: dims 16mi + lane/4 (+8), heads 2(lane%4) (+1)
        float m[2];          // running max of heads 2(lane%4), 2(lane%4)+1
        float l[2];          // this lane's share of the running sum
    };

    __device__ __forceinline__ void begin(State& st, const DecodeArgs& a, int s, int h, int G) {
        const int lane = threadIdx.x & 31;
        const int g = lane >> 2, c = lane & 3;
        // Columns g >= G (padding of the MMA's 8 columns) repeat head g % G,
        // so their scores and probabilities equal that head's (see tile()).
        const T* q = static_cast<const T*>(a.q) +
                     (static_cast<int64_t>(s) * a.num_q_heads + h * G + g % G) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            st.qb[ks][0] = *reinterpret_cast<const uint32_t*>(q + 16 * ks + 2 * c);
            st.qb[ks][1] = *reinterpret_cast<const uint32_t*>(q + 16 * ks + 2 * c + 8);
#pragma unroll
            for (int r = 0; r < 4; ++r) st.o[ks][r] = 0.f;
        }
        st.m[0] = st.m[1] = -INFINITY;
        st.l[0] = st.l[1] = 0.f;
    }

    // One head's part of a stage: kt/vt point at the stage's K/V, laid out as
    // [64-element slice][Hc*bs rows][128 B] (128-byte swizzled by the tensor
    // copy); this warp's head owns rows hw*bs .. hw*bs+bs-1 of every slice.
    __device__ __forceinline__ void tile(State& st, const DecodeArgs& a, uint8_t* kt, uint8_t* vt,
                                         int hw, int n_valid, int G, float*) {
        const int lane = threadIdx.x & 31;
        const int bs = a.block_size;
        const uint32_t slice_bytes = static_cast<uint32_t>(a.heads_per_stage * bs) * 128u;
        uint8_t* kh = kt + hw * bs * 128;
        uint8_t* vh = vt + hw * bs * 128;
        // Rows past the valid tokens may hold anything (even NaN): zero this
        // head's V rows there so that 0 * V stays 0 in the PV product.
        if (n_valid < bs) {
            const int per_slice = (bs - n_valid) * 8;  // 16-byte chunks per slice
            for (int e = lane; e < per_slice * (D / 64); e += 32) {
                const int sl = e / per_slice;
                const int r = e - sl * per_slice;
                uint4* p = reinterpret_cast<uint4*>(vh + sl * slice_bytes + (n_valid + (r >> 3)) * 128 +
                                                    ((r & 7) << 4));
                *p = make_uint4(0u, 0u, 0u, 0u);
            }
            __syncwarp();
        }
        const uint32_t kb = smem_addr(kh), vb = smem_addr(vh);
        const uint32_t sw = lane & 7;  // 128-byte swizzle key of the rows this lane addresses
        const float sl = a.scale_log2;
        for (int mt = 0; mt < bs / 16; ++mt) {
            // ---- S^T = K . Q^T for tokens 16mt .. 16mt+15.  The warp-level MMA
            // has a long latency: the k-steps accumulate into up to 4
            // independent chains, summed at the end.
            constexpr int NC = KS < 4 ? KS : 4;
            float part[NC][4];
#pragma unroll
            for (int k = 0; k < NC; ++k)
#pragma unroll
                for (int r = 0; r < 4; ++r) part[k][r] = 0.f;
            {
                const uint32_t row = static_cast<uint32_t>(mt * 16 + (lane & 7) + (lane & 8));
#pragma unroll
                for (int ks = 0; ks < KS; ++ks) {
                    const uint32_t chunk = ((ks & 3) << 1) | (lane >> 4);
                    uint32_t af[4];
                    ldsm_x4(af, kb + (ks >> 2) * slice_bytes + row * 128u + ((chunk ^ sw) << 4));
                    mma16816<DT>(part[ks % NC], af, st.qb[ks][0], st.qb[ks][1]);
                }
            }
            float acc[4];
#pragma unroll
            for (int r = 0; r < 4; ++r) {
                acc[r] = part[0][r];
#pragma unroll
                for (int k = 1; k < NC; ++k) acc[r] += part[k][r];
            }
            // ---- online softmax (heads 2c, 2c+1; tokens g and g+8 of the slice)
            const int t0 = mt * 16 + (lane >> 2);
            const bool v0 = t0 < n_valid, v1 = t0 + 8 < n_valid;
            const float x0 = v0 ? acc[0] * sl : -INFINITY;
            const float x1 = v0 ? acc[1] * sl : -INFINITY;
            const float x2 = v1 ? acc[2] * sl : -INFINITY;
            const float x3 = v1 ? acc[3] * sl : -INFINITY;
            float mx0 = fmaxf(x0, x2), mx1 = fmaxf(x1, x3);
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
            const float al0 = fast_exp2(st.m[0] - mn0), al1 = fast_exp2(st.m[1] - mn1);
            st.m[0] = mn0;
            st.m[1] = mn1;
            const float p0 = fast_exp2(x0 - mn0), p1 = fast_exp2(x1 - mn1);
            const float p2 = fast_exp2(x2 - mn0), p3 = fast_exp2(x3 - mn1);
            st.l[0] = st.l[0] * al0 + (p0 + p2);
            st.l[1] = st.l[1] * al1 + (p1 + p3);
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                for (int mi = 0; mi < KS; ++mi) {
                    st.o[mi][0] *= al0;
                    st.o[mi][1] *= al1;
                    st.o[mi][2] *= al0;
                    st.o[mi][3] *= al1;
                }
            }
            // ---- P^T fragments (k = token, n = head), high + low parts.  With
            // G <= 4 the low parts ride in columns 4-7 (which repeat heads 0-3,
            // so this lane's probabilities there are those of head col % G):
            // one MMA per slice; O of head h is then column h + column h + 4.
            uint32_t h01, l01, h23, l23;
            pack_split<DT>(p0, p1, h01, l01);
            pack_split<DT>(p2, p3, h23, l23);
            const bool packed = G <= 4;
            const bool lo_cols = (lane & 3) >= 2;  // this lane's columns 2c, 2c+1 are >= 4
            const uint32_t bh0 = movmatrix_trans(packed && lo_cols ? l01 : h01);
            const uint32_t bh1 = movmatrix_trans(packed && lo_cols ? l23 : h23);
            uint32_t bl0 = 0u, bl1 = 0u;
            if (!packed) {
                bl0 = movmatrix_trans(l01);
                bl1 = movmatrix_trans(l23);
            }
            // ---- O^T += V^T . P^T
            {
                const uint32_t row = static_cast<uint32_t>(mt * 16 + (lane & 7) + ((lane >> 4) << 3));
                const uint32_t csel = (lane >> 3) & 1;
#pragma unroll
                for (int mi = 0; mi < KS; ++mi) {
                    const uint32_t chunk = ((mi & 3) << 1) | csel;
                    uint32_t af[4];
                    ldsm_x4_trans(af, vb + (mi >> 2) * slice_bytes + row * 128u + ((chunk ^ sw) << 4));
                    mma16816<DT>(st.o[mi], af, bh0, bh1);
                    if (!packed) mma16816<DT>(st.o[mi], af, bl0, bl1);
                }
            }
        }
        if (n_valid < bs) fence_proxy_async_smem();  // generic writes before the next TMA fill
    }

    // 16-byte chunk q of row r of head hw's tile (the stage's 128-byte
    // swizzled layout: chunk c of a row lands at c ^ (row % 8)).
    __device__ __forceinline__ void patch_chunk(const DecodeArgs& a, uint8_t* t, int hw, int r, int q,
                                                uint4 val) const {
        const int bs = a.block_size;
        const int slice_bytes = a.heads_per_stage * bs * 128;
        const int row = hw * bs + r;
        *reinterpret_cast<uint4*>(t + (q >> 3) * slice_bytes + row * 128 + (((q & 7) ^ (row & 7)) << 4)) = val;
    }

    // Accumulators of slice mi with the low-part columns (4-7, G <= 4) added
    // to the columns of their heads; valid in lanes whose columns are < 4.
    __device__ __forceinline__ void fold(const State& st, int mi, int G, float (&v)[4]) const {
#pragma unroll
        for (int r = 0; r < 4; ++r) {
            const float other = __shfl_down_sync(0xffffffffu, st.o[mi][r], 2);
            v[r] = st.o[mi][r] + (G <= 4 ? other : 0.f);
        }
    }

    // Row sums of heads 2c, 2c+1 over the whole warp.
    __device__ __forceinline__ void row_sums(const State& st, float& l0, float& l1) const {
        l0 = st.l[0];
        l1 = st.l[1];
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
    }

    // O (unnormalised) to o[g*os + d], (max, sum) to ml[g*ms], ml[g*ms + 1].
    __device__ __forceinline__ void emit(const State& st, float* o, int os, float* ml, int ms,
                                         int G) const {
        const int lane = threadIdx.x & 31;
        const int g = lane >> 2, c = lane & 3;
        float l0, l1;
        row_sums(st, l0, l1);
        const int h0 = 2 * c, h1 = 2 * c + 1;
#pragma unroll
        for (int mi = 0; mi < KS; ++mi) {
            float v[4];
            fold(st, mi, G, v);
            const int d0 = 16 * mi + g;
            if (h0 < G) {
                o[h0 * os + d0] = v[0];
                o[h0 * os + d0 + 8] = v[2];
            }
            if (h1 < G) {
                o[h1 * os + d0] = v[1];
                o[h1 * os + d0 + 8] = v[3];
            }
        }
        if (g == 0) {
            if (h0 < G) {
                ml[h0 * ms] = st.m[0];
                ml[h0 * ms + 1] = l0;
            }
            if (h1 < G) {
                ml[h1 * ms] = st.m[1];
                ml[h1 * ms + 1] = l1;
            }
        }
    }

    __device__ __forceinline__ void write_state(const State& st, const DecodeArgs&, float* dst,
                                                int stride, int G) const {
        emit(st, dst, stride, dst + D, stride, G);
    }

    __device__ __forceinline__ void write_partial(const State& st, const DecodeArgs&, float* o,
                                                  float* ml, int G) const {
        emit(st, o, D, ml, 2, G);
    }

    // out[s][h*G + head][d] = O / l in the output type.
    __device__ __forceinline__ void write_final(const State& st, const DecodeArgs& a, int s, int h,
                                                int G) const {
        const int lane = threadIdx.x & 31;
        const int g = lane >> 2, c = lane & 3;
        float l0, l1;
        row_sums(st, l0, l1);
        const float i0 = 1.f / l0, i1 = 1.f / l1;
        const int h0 = 2 * c, h1 = 2 * c + 1;
        const int64_t base = (static_cast<int64_t>(s) * a.num_q_heads + h * G) * D;
#pragma unroll
        for (int mi = 0; mi < KS; ++mi) {
            float v[4];
            fold(st, mi, G, v);
            const int d0 = 16 * mi + g;
            if (h0 < G) {
                store_out(a.out, base + h0 * D + d0, v[0] * i0, a.out_dtype);
                store_out(a.out, base + h0 * D + d0 + 8, v[2] * i0, a.out_dtype);
            }
            if (h1 < G) {
                store_out(a.out, base + h1 * D + d0, v[1] * i1, a.out_dtype);
                store_out(a.out, base + h1 * D + d0 + 8, v[3] * i1, a.out_dtype);
            }
        }
    }
};

// Launches of up to 12 warps (the default is 9) use the instantiation built
// for 384 threads, whose register budget (168 a thread) holds the consumer
// state and the merge of split pairs without spilling.
template <int DT, int D>
static cudaError_t launch_mma_t(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                                cudaStream_t stream) {
    if (32 * (1 + a.consumer_warps) <= 32 * 12) return launch_partial<MmaPolicy<DT, D, 32 * 12>>(a, tmk, tmv, stream);
    return launch_partial<MmaPolicy<DT, D>>(a, tmk, tmv, stream);
}

cudaError_t launch_decode_mma(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              cudaStream_t stream) {
    if (a.dtype == kF16) {
        if (a.head_dim == 64) return launch_mma_t<kF16, 64>(a, tmk, tmv, stream);
        if (a.head_dim == 128) return launch_mma_t<kF16, 128>(a, tmk, tmv, stream);
    } else if (a.dtype == kBF16) {
        if (a.head_dim == 64) return launch_mma_t<kBF16, 64>(a, tmk, tmv, stream);
        if (a.head_dim == 128) return launch_mma_t<kBF16, 128>(a, tmk, tmv, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace pkv
