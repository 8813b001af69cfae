// Tensor-core consumer of the split-context decode kernel for an E4M3 (FP8)
// KV cache ("vLLM Architecture and Installation", Example 6: one byte per
// cached value, so a block and the bytes a decode step reads halve).
//
// A cached byte b stands for scale * e4m3(b), one scale per layer for K and
// one for V.  Every E4M3 value is exactly an f16, so the tile is converted in
// registers (two codes per conversion) and fed to the f16 m16n8k16 MMA:
//   S^T = K8 . Q^T           scores, times scale * log2(e) * k_scale
//   O^T += V8^T . P^T        times v_scale when the state is written out
// P enters the PV product as an f16 high part plus an f16 low part; with up
// to 4 query heads per KV head the low parts ride in the MMA's padding
// columns 4-7 (one PV MMA per 16-dim slice), folded back when written out.
// q (f16 or bf16) becomes f16 B fragments once per (sequence, head).
//
// Fragment layout.  ldmatrix moves 16-bit elements, i.e. pairs of codes.
//  - K (non-transposed): a lane receives four consecutive codes of its row,
//    dims 16j + 4c .. 16j + 4c + 3 of a 16-dim chunk j (c = lane % 4).  The
//    dot product does not care in which order dims are summed, so the MMA's
//    k index is permuted inside each chunk: logical columns 2c, 2c+1 hold
//    dims 4c, 4c+2 (the word's even bytes) and logical columns 2c+8, 2c+9
//    hold dims 4c+1, 4c+3 (its odd bytes), and the q fragments are built
//    with the same permutation.  One ldmatrix.x4 then yields the A fragments
//    of two 16-dim chunks.
//  - V (transposed): a lane receives the code pairs (2g, 2g+1) of tokens 2c
//    and 2c+1 (g = lane / 4): the word's even bytes are the token pair of
//    dim 2g and its odd bytes that of dim 2g+1, each converted in place (no
//    byte permute).  So M row g of a 16-dim chunk is dim 2g and row g+8 is
//    dim 2g+1, and the output accumulators are written back with that
//    mapping.
// Tiles arrive through 2-D tensor maps with a 128-byte swizzle: rows of 128
// codes (head_dim 128), chunk c of row r stored at chunk c ^ (r % 8).
#include "decode_kernel.cuh"
#include "mma_frag.cuh"

namespace pkv {

// f16x2 of p's f16 high part (low half) and the f16 rounding of the rest.
__device__ __forceinline__ uint32_t f16_high_low(float p) {
    const __half h = __float2half_rn(p);
    const __half2 hl = __halves2half2(h, __float2half_rn(p - __half2float(h)));
    return *reinterpret_cast<const uint32_t*>(&hl);
}

// kQ8: QK on the E4M3 tensor path (bf16 q, at most 4 query heads per KV
// head).  The K tile feeds the m16n8k32 E4M3 MMA straight from ldmatrix (a
// lane's four consecutive codes are exactly its A-fragment bytes), so K needs
// no conversion.  q is scaled per head by a power of two 2^kq (largest |q| to
// [128, 256)) and split exactly into two E4M3 parts, hi = RN(q') and
// lo = q' - hi (a bf16 value has 8 significant bits, each part holds 4, and
// the rounding residual of hi is a multiple of hi's last-bit weight / 16 no
// larger than half of it, so it fits 4 bits): column 2j carries hi and column
// 2j+1 lo of head j (heads past G repeat), so lane c's two accumulator columns
// are head c's two halves, added in place; the softmax, P's fragments and the
// output then take one head a lane.  Scores carry
// scale * log2(e) * k_scale * 2^-kq.
// kMaxT: the largest block the instantiation is launched with.  The usual
// launch (1 + 8 warps) takes the 384-thread variant, whose register budget
// (168 per thread) holds the state without spilling.
template <int QT, int D, bool kQ8 = false, int kMaxT = 32 * 16>
struct MmaFp8Policy {
    static constexpr int kMaxThreads = kMaxT;
    static_assert(D == 128, "E4M3 rows of 128 codes: one 128-byte slice per row");
    static_assert(!kQ8 || QT == kBF16, "the E4M3 QK path splits a bf16 q exactly");
    static constexpr bool kTensor = true;
    static constexpr bool kScratch = false;
    static constexpr int KS = D / 16;  // 16-dim chunks: k-slices of QK, m-slices of PV
    static constexpr int K8 = D / 32;  // 32-dim k-slices of the E4M3 QK
    static constexpr int kD = D;
    // V enters the P.V product as its E4M3 value times 2^-8 (see
    // e4m3x2_odd_bytes_to_half2_shifted); the outputs are scaled back by 2^8, exactly.
    static constexpr float kVUnscale = 256.f;
    // Likewise K in the f16 form of Q.K^T (not kQ8, where the MMA takes the codes).
    static constexpr float kKUnscale = 256.f;
    using T = typename Elem<QT>::T;

    struct State {
        // f16 B fragments of Q^T, head lane/4: dims 16ks + 4(lane%4) + {0,1} / {2,3};
        // kQ8: E4M3 B fragments, dims 32j + 4(lane%4) + {0..3} / 16 + ...
        uint32_t qb[kQ8 ? K8 : KS][2];
        float sc[2];         // kQ8: score multipliers of columns 2(lane%4), 2(lane%4)+1 (one head)
        float o[KS][4];      // O^T: dims 16mi + 2(lane/4) (+1 for [2],[3]), heads 2(lane%4) (+1 for [1],[3])
        float m[2];          // running max of heads 2(lane%4), 2(lane%4)+1 (kQ8: [0], head lane%4)
        float l[2];          // this lane's share of the running sum (kQ8: [0])
    };

    // kQ8 begin: B fragments of q's two E4M3 parts and the per-column score scale.
    __device__ __forceinline__ void begin_q8(State& st, const DecodeArgs& a, int s, int h, int G) {
        const int lane = threadIdx.x & 31;
        const int g = lane >> 2, c = lane & 3;
        // Column g carries head g/2 (repeated past G): its high part in even
        // columns, its low part in odd ones.
        const T* q = static_cast<const T*>(a.q) +
                     (static_cast<int64_t>(s) * a.num_q_heads + h * G + (g >> 1) % G) * D;
        float v[K8][8];
        float mx = 0.f;
#pragma unroll
        for (int j = 0; j < K8; ++j) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const uint2 raw = *reinterpret_cast<const uint2*>(q + 32 * j + 16 * half + 4 * c);
                const T* e = reinterpret_cast<const T*>(&raw);
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[j][4 * half + i] = Elem<QT>::to_float(e[i]);
                    mx = fmaxf(mx, fabsf(v[j][4 * half + i]));
                }
            }
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        // 2^kq with mx * 2^kq in [128, 256): kq = 7 - floor(log2 mx).
        int kq = 0;
        if (mx > 0.f) kq = 7 - (((__float_as_int(mx) >> 23) & 0xff) - 127);
        kq = kq < -120 ? -120 : (kq > 120 ? 120 : kq);
        const float up = __int_as_float((127 + kq) << 23);
        const bool lo_part = (g & 1) != 0;
#pragma unroll
        for (int j = 0; j < K8; ++j) {
            uint32_t w[2];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                uint32_t word = 0u;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const float x0 = v[j][4 * half + 2 * p] * up, x1 = v[j][4 * half + 2 * p + 1] * up;
                    const uint16_t hi = e4m3x2_from_floats(x0, x1);
                    const uint32_t hh = e4m3x2_to_half2(hi);
                    const __half2 hd = *reinterpret_cast<const __half2*>(&hh);
                    const uint16_t lo = e4m3x2_from_floats(x0 - __low2float(hd), x1 - __high2float(hd));
                    word |= static_cast<uint32_t>(lo_part ? lo : hi) << (16 * p);
                }
                w[half] = word;
            }
            st.qb[j][0] = w[0];
            st.qb[j][1] = w[1];
        }
        // Columns 2c and 2c+1 (this lane's) are both head c: rows g = 2c, 2c+1.
        const int k0 = __shfl_sync(0xffffffffu, kq, 8 * c);
        const int k1 = __shfl_sync(0xffffffffu, kq, 8 * c + 4);
        st.sc[0] = a.scale_log2 * __int_as_float((127 - k0) << 23);
        st.sc[1] = a.scale_log2 * __int_as_float((127 - k1) << 23);
    }

    __device__ __forceinline__ void begin(State& st, const DecodeArgs& a, int s, int h, int G) {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks)
#pragma unroll
            for (int r = 0; r < 4; ++r) st.o[ks][r] = 0.f;
        st.m[0] = st.m[1] = -INFINITY;
        st.l[0] = st.l[1] = 0.f;
        if constexpr (kQ8) {
            begin_q8(st, a, s, h, G);
            return;
        }
        const int g = lane >> 2, c = lane & 3;
        // Columns g >= G (padding of the MMA's 8 columns) repeat head g % G,
        // so their scores and probabilities equal that head's (see tile()).
        const T* q = static_cast<const T*>(a.q) +
                     (static_cast<int64_t>(s) * a.num_q_heads + h * G + g % G) * D;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            // Dims 4c, 4c+2 (k = 2c, 2c+1) and 4c+1, 4c+3 (k = 2c+8, 2c+9), as K's fragments.
            const uint2 raw = *reinterpret_cast<const uint2*>(q + 16 * ks + 4 * c);
            if constexpr (QT == kF16) {
                st.qb[ks][0] = __byte_perm(raw.x, raw.y, 0x5410u);
                st.qb[ks][1] = __byte_perm(raw.x, raw.y, 0x7632u);
            } else {
                const T* e = reinterpret_cast<const T*>(&raw);
                const __half2 h0 = __floats2half2_rn(Elem<QT>::to_float(e[0]), Elem<QT>::to_float(e[2]));
                const __half2 h1 = __floats2half2_rn(Elem<QT>::to_float(e[1]), Elem<QT>::to_float(e[3]));
                st.qb[ks][0] = *reinterpret_cast<const uint32_t*>(&h0);
                st.qb[ks][1] = *reinterpret_cast<const uint32_t*>(&h1);
            }
        }
    }

    // Rows past the valid tokens may hold any code (even NaN): zero this
    // head's V rows [n_valid, bs) of a stage so that 0 * V stays 0 in PV.
    __device__ __forceinline__ void zero_tail(uint8_t* vh, int n_valid, int bs) const {
        const int lane = threadIdx.x & 31;
        for (int e = lane; e < (bs - n_valid) * 8; e += 32) {
            uint4* p = reinterpret_cast<uint4*>(vh + (n_valid + (e >> 3)) * 128 + ((e & 7) << 4));
            *p = make_uint4(0u, 0u, 0u, 0u);
        }
        __syncwarp();
    }

    // NS 16-token slices at once: kb[n] / vb[n] are the shared addresses of
    // slice n's first K / V row, nv[n] its valid tokens (<= 0: none).  One
    // online-softmax update covers all their tokens, and the independent MMA
    // chains of the slices interleave, which keeps the warp's dependent
    // instruction chains short.
    template <int NS>
    __device__ __forceinline__ void slices(State& st, const DecodeArgs& a, const uint32_t (&kb)[NS],
                                           const uint32_t (&vb)[NS], const int (&nv)[NS], int G) {
        const int lane = threadIdx.x & 31;
        const uint32_t sw = lane & 7;  // swizzle key of the rows this lane addresses
        // Lanes 0-7 / 8-15 / 16-23 / 24-31 address rows 0-7 / 8-15 / 0-7 / 8-15
        // of a slice, in chunk 2p / 2p / 2p+1 / 2p+1.
        const uint32_t rofs = static_cast<uint32_t>((lane & 7) + (lane & 8)) * 128u;
        const uint32_t csel = static_cast<uint32_t>(lane >> 4);
        // ---- S^T = K . Q^T, two accumulation chains per slice
        float acc[NS][4];
#pragma unroll
        for (int n = 0; n < NS; ++n) {
            float part[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
            for (int kp = 0; kp < KS / 2; ++kp) {
                uint32_t r[4];
                ldsm_x4(r, kb[n] + rofs + ((((2u * kp) | csel) ^ sw) << 4));
                if constexpr (kQ8) {
                    // r[0] / r[1]: rows g / g+8, dims 32kp + 4c..; r[2] / r[3]: dims 32kp + 16 + 4c..
                    const uint32_t af[4] = {r[0], r[1], r[2], r[3]};
                    mma16832_e4m3(part[kp & 1], af, st.qb[kp][0], st.qb[kp][1]);
                } else {
#pragma unroll
                    for (int hf = 0; hf < 2; ++hf) {  // chunk 2kp + hf: rows g / g+8 in r[2hf] / r[2hf+1]
                        uint32_t af[4];
                        // K codes as f16 values times 2^-8 (kKUnscale restores the scores):
                        // even bytes are k = 2c, 2c+1, odd bytes k = 2c+8, 2c+9.
                        af[0] = e4m3x2_even_bytes_to_half2_shifted(r[2 * hf]);
                        af[1] = e4m3x2_even_bytes_to_half2_shifted(r[2 * hf + 1]);
                        af[2] = e4m3x2_odd_bytes_to_half2_shifted(r[2 * hf]);
                        af[3] = e4m3x2_odd_bytes_to_half2_shifted(r[2 * hf + 1]);
                        mma16816<kF16>(part[hf], af, st.qb[2 * kp + hf][0], st.qb[2 * kp + hf][1]);
                    }
                }
            }
#pragma unroll
            for (int r = 0; r < 4; ++r) acc[n][r] = part[0][r] + part[1][r];
            if constexpr (kQ8) {  // head c: its high (column 2c) and low (2c+1) parts
                acc[n][0] += acc[n][1];
                acc[n][2] += acc[n][3];
            }
        }
        uint32_t bh[NS][2], bl[NS][2];
        const bool packed = kQ8 || G <= 4;
        if constexpr (kQ8) {
            // ---- online softmax over all NS slices (head c; tokens g, g+8 of each)
            const float sl = st.sc[0];
            float x[NS][2];
            float mx = -INFINITY;
#pragma unroll
            for (int n = 0; n < NS; ++n) {
                const int t0 = lane >> 2;
                x[n][0] = t0 < nv[n] ? acc[n][0] * sl : -INFINITY;
                x[n][1] = t0 + 8 < nv[n] ? acc[n][2] * sl : -INFINITY;
                mx = fmaxf(mx, fmaxf(x[n][0], x[n][1]));
            }
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float mn = fmaxf(st.m[0], mx);
            const float al = fast_exp2(st.m[0] - mn);
            st.m[0] = mn;
            float ls = 0.f;
#pragma unroll
            for (int n = 0; n < NS; ++n) {
                const float p0 = fast_exp2(x[n][0] - mn), p1 = fast_exp2(x[n][1] - mn);
                ls += p0 + p1;
                // P^T fragments: column 2c the f16 high part of head c's p, 2c+1 the low part.
                bh[n][0] = movmatrix_trans(f16_high_low(p0));
                bh[n][1] = movmatrix_trans(f16_high_low(p1));
                bl[n][0] = bl[n][1] = 0u;
            }
            st.l[0] = st.l[0] * al + ls;
            if (__any_sync(0xffffffffu, al != 1.f)) {
#pragma unroll
                for (int mi = 0; mi < KS; ++mi)
#pragma unroll
                    for (int r = 0; r < 4; ++r) st.o[mi][r] *= al;
            }
        } else {
        const float sl0 = a.scale_log2 * kKUnscale;
        const float sl1 = a.scale_log2 * kKUnscale;
        // ---- online softmax over all NS slices (heads 2c, 2c+1; tokens g, g+8 of each)
        float x[NS][4];
        float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
        for (int n = 0; n < NS; ++n) {
            const int t0 = lane >> 2;
            const bool v0 = t0 < nv[n], v1 = t0 + 8 < nv[n];
            x[n][0] = v0 ? acc[n][0] * sl0 : -INFINITY;
            x[n][1] = v0 ? acc[n][1] * sl1 : -INFINITY;
            x[n][2] = v1 ? acc[n][2] * sl0 : -INFINITY;
            x[n][3] = v1 ? acc[n][3] * sl1 : -INFINITY;
            mx0 = fmaxf(mx0, fmaxf(x[n][0], x[n][2]));
            mx1 = fmaxf(mx1, fmaxf(x[n][1], x[n][3]));
        }
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
        }
        const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
        const float al0 = fast_exp2(st.m[0] - mn0), al1 = fast_exp2(st.m[1] - mn1);
        st.m[0] = mn0;
        st.m[1] = mn1;
        float ls0 = 0.f, ls1 = 0.f;
        const bool lo_cols = (lane & 3) >= 2;
#pragma unroll
        for (int n = 0; n < NS; ++n) {
            const float p0 = fast_exp2(x[n][0] - mn0), p1 = fast_exp2(x[n][1] - mn1);
            const float p2 = fast_exp2(x[n][2] - mn0), p3 = fast_exp2(x[n][3] - mn1);
            ls0 += p0 + p2;
            ls1 += p1 + p3;
            // P^T fragments (k = token, n = head), f16 high + low parts; with G <= 4
            // the low parts ride in the padding columns 4-7 (see fold).
            uint32_t h01, l01, h23, l23;
            pack_split<kF16>(p0, p1, h01, l01);
            pack_split<kF16>(p2, p3, h23, l23);
            bh[n][0] = movmatrix_trans(packed && lo_cols ? l01 : h01);
            bh[n][1] = movmatrix_trans(packed && lo_cols ? l23 : h23);
            bl[n][0] = bl[n][1] = 0u;
            if (!packed) {
                bl[n][0] = movmatrix_trans(l01);
                bl[n][1] = movmatrix_trans(l23);
            }
        }
        st.l[0] = st.l[0] * al0 + ls0;
        st.l[1] = st.l[1] * al1 + ls1;
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
            for (int mi = 0; mi < KS; ++mi) {
                st.o[mi][0] *= al0;
                st.o[mi][1] *= al1;
                st.o[mi][2] *= al0;
                st.o[mi][3] *= al1;
            }
        }
        }
        // ---- O^T += V^T . P^T
#pragma unroll
        for (int mp = 0; mp < KS / 2; ++mp) {
#pragma unroll
            for (int n = 0; n < NS; ++n) {
                uint32_t r[4];
                ldsm_x4_trans(r, vb[n] + rofs + ((((2u * mp) | csel) ^ sw) << 4));
                // r[k] bytes: (tok 2c, dim 2g), (tok 2c, dim 2g+1), (tok 2c+1, dim 2g), (tok 2c+1, dim 2g+1);
                // r[2hf] holds tokens 0-7 and r[2hf+1] tokens 8-15 of chunk 2mp + hf.
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t af[4];
                    af[0] = e4m3x2_even_bytes_to_half2_shifted(r[2 * hf]);     // dim 2g,   tokens 2c, 2c+1
                    af[1] = e4m3x2_odd_bytes_to_half2_shifted(r[2 * hf]);      // dim 2g+1, tokens 2c, 2c+1
                    af[2] = e4m3x2_even_bytes_to_half2_shifted(r[2 * hf + 1]); // dim 2g,   tokens 8+2c, 9+2c
                    af[3] = e4m3x2_odd_bytes_to_half2_shifted(r[2 * hf + 1]);  // dim 2g+1, tokens 8+2c, 9+2c
                    mma16816<kF16>(st.o[2 * mp + hf], af, bh[n][0], bh[n][1]);
                    if (!packed) mma16816<kF16>(st.o[2 * mp + hf], af, bl[n][0], bl[n][1]);
                }
            }
        }
    }

    // One head's part of a stage: kt/vt point at the stage's K/V codes,
    // [Hc*bs rows][128 B]; this warp's head owns rows hw*bs .. hw*bs+bs-1,
    // taken two 16-token slices at a time.
    __device__ __forceinline__ void tile(State& st, const DecodeArgs& a, uint8_t* kt, uint8_t* vt,
                                         int hw, int n_valid, int G, float*) {
        const int bs = a.block_size;
        uint8_t* kh = kt + hw * bs * 128;
        uint8_t* vh = vt + hw * bs * 128;
        if (n_valid < bs) zero_tail(vh, n_valid, bs);
        const uint32_t kb = smem_addr(kh), vb = smem_addr(vh);
        int mt = 0;
        for (; mt + 2 <= bs / 16; mt += 2) {
            const uint32_t k2[2] = {kb + mt * 2048u, kb + (mt + 1) * 2048u};
            const uint32_t v2[2] = {vb + mt * 2048u, vb + (mt + 1) * 2048u};
            const int n2[2] = {n_valid - 16 * mt, n_valid - 16 * (mt + 1)};
            slices<2>(st, a, k2, v2, n2, G);
        }
        if (mt < bs / 16) {
            const uint32_t k1[1] = {kb + mt * 2048u};
            const uint32_t v1[1] = {vb + mt * 2048u};
            const int n1[1] = {n_valid - 16 * mt};
            slices<1>(st, a, k1, v1, n1, G);
        }
        if (n_valid < bs) fence_proxy_async_smem();  // generic writes before the next TMA fill
    }

    // Two 16-token blocks (block_size 16) from two stages of one (sequence,
    // head) run, processed together.
    static constexpr bool kPairs = true;
    __device__ __forceinline__ void tile2(State& st, const DecodeArgs& a, uint8_t* kt0, uint8_t* vt0,
                                          int n0, uint8_t* kt1, uint8_t* vt1, int n1, int hw, int G) {
        uint8_t* kh0 = kt0 + hw * 16 * 128;
        uint8_t* vh0 = vt0 + hw * 16 * 128;
        uint8_t* kh1 = kt1 + hw * 16 * 128;
        uint8_t* vh1 = vt1 + hw * 16 * 128;
        if (n0 < 16) zero_tail(vh0, n0, 16);
        if (n1 < 16) zero_tail(vh1, n1, 16);
        const uint32_t k2[2] = {smem_addr(kh0), smem_addr(kh1)};
        const uint32_t v2[2] = {smem_addr(vh0), smem_addr(vh1)};
        const int n2[2] = {n0, n1};
        slices<2>(st, a, k2, v2, n2, G);
        if (n0 < 16 || n1 < 16) fence_proxy_async_smem();
    }

    // 16-byte chunk q of row r of head hw's tile (chunk c of a row lands at c ^ (row % 8)).
    __device__ __forceinline__ void patch_chunk(const DecodeArgs& a, uint8_t* t, int hw, int r, int q,
                                                uint4 val) const {
        const int row = hw * a.block_size + r;
        *reinterpret_cast<uint4*>(t + row * 128 + (((q & 7) ^ (row & 7)) << 4)) = val;
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

    __device__ __forceinline__ void row_sums(const State& st, float& l0, float& l1) const {
        l0 = st.l[0];
        l1 = st.l[1];
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) {
            l0 += __shfl_xor_sync(0xffffffffu, l0, off);
            l1 += __shfl_xor_sync(0xffffffffu, l1, off);
        }
    }

    // v_scale * O (unnormalised) to o[g*os + d], (max, sum) to ml[g*ms], ml[g*ms + 1].
    __device__ __forceinline__ void emit(const State& st, float vs, float* o, int os, float* ml, int ms,
                                         int G) const {
        const int lane = threadIdx.x & 31;
        const int g = lane >> 2, c = lane & 3;
        if constexpr (kQ8) {  // head c: its high and low columns summed
            float l = st.l[0];
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
            if (c >= G) return;
#pragma unroll
            for (int mi = 0; mi < KS; ++mi) {
                const int d0 = 16 * mi + 2 * g;
                o[c * os + d0] = (st.o[mi][0] + st.o[mi][1]) * vs;
                o[c * os + d0 + 1] = (st.o[mi][2] + st.o[mi][3]) * vs;
            }
            if (g == 0) {
                ml[c * ms] = st.m[0];
                ml[c * ms + 1] = l;
            }
            return;
        }
        float l0, l1;
        row_sums(st, l0, l1);
        const int h0 = 2 * c, h1 = 2 * c + 1;
#pragma unroll
        for (int mi = 0; mi < KS; ++mi) {
            float v[4];
            fold(st, mi, G, v);
            const int d0 = 16 * mi + 2 * g;
            if (h0 < G) {
                o[h0 * os + d0] = v[0] * vs;
                o[h0 * os + d0 + 1] = v[2] * vs;
            }
            if (h1 < G) {
                o[h1 * os + d0] = v[1] * vs;
                o[h1 * os + d0 + 1] = v[3] * vs;
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

    __device__ __forceinline__ void write_state(const State& st, const DecodeArgs& a, float* dst,
                                                int stride, int G) const {
        emit(st, a.v_scale * kVUnscale, dst, stride, dst + D, stride, G);
    }

    __device__ __forceinline__ void write_partial(const State& st, const DecodeArgs& a, float* o,
                                                  float* ml, int G) const {
        emit(st, a.v_scale * kVUnscale, o, D, ml, 2, G);
    }

    // out[s][h*G + head][d] = v_scale * O / l in the output type.
    __device__ __forceinline__ void write_final(const State& st, const DecodeArgs& a, int s, int h,
                                                int G) const {
        const int lane = threadIdx.x & 31;
        const int g = lane >> 2, c = lane & 3;
        if constexpr (kQ8) {  // head c: its high and low columns summed
            float l = st.l[0];
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) l += __shfl_xor_sync(0xffffffffu, l, off);
            if (c >= G) return;
            const float inv = a.v_scale * kVUnscale / l;
            const int64_t base = (static_cast<int64_t>(s) * a.num_q_heads + h * G + c) * D;
#pragma unroll
            for (int mi = 0; mi < KS; ++mi) {
                const int d0 = 16 * mi + 2 * g;
                store_out(a.out, base + d0, (st.o[mi][0] + st.o[mi][1]) * inv, a.out_dtype);
                store_out(a.out, base + d0 + 1, (st.o[mi][2] + st.o[mi][3]) * inv, a.out_dtype);
            }
            return;
        }
        float l0, l1;
        row_sums(st, l0, l1);
        const float i0 = a.v_scale * kVUnscale / l0, i1 = a.v_scale * kVUnscale / l1;
        const int h0 = 2 * c, h1 = 2 * c + 1;
        const int64_t base = (static_cast<int64_t>(s) * a.num_q_heads + h * G) * D;
#pragma unroll
        for (int mi = 0; mi < KS; ++mi) {
            float v[4];
            fold(st, mi, G, v);
            const int d0 = 16 * mi + 2 * g;
            if (h0 < G) {
                store_out(a.out, base + h0 * D + d0, v[0] * i0, a.out_dtype);
                store_out(a.out, base + h0 * D + d0 + 1, v[2] * i0, a.out_dtype);
            }
            if (h1 < G) {
                store_out(a.out, base + h1 * D + d0, v[1] * i1, a.out_dtype);
                store_out(a.out, base + h1 * D + d0 + 1, v[3] * i1, a.out_dtype);
            }
        }
    }
};

cudaError_t launch_decode_fp8(const DecodeArgs& a, const CUtensorMap& tmk, const CUtensorMap& tmv,
                              cudaStream_t stream) {
    if (a.kv_dtype != kFP8 || a.head_dim != 128) return cudaErrorInvalidValue;
    const int G = a.num_q_heads / a.num_kv_heads;
    if (a.dtype == kF16) return launch_partial<MmaFp8Policy<kF16, 128>>(a, tmk, tmv, stream);
    if (a.dtype == kBF16 && G <= 4) {
        if (32 * (1 + a.consumer_warps) <= 32 * 12)
            return launch_partial<MmaFp8Policy<kBF16, 128, true, 32 * 12>>(a, tmk, tmv, stream);
        return launch_partial<MmaFp8Policy<kBF16, 128, true>>(a, tmk, tmv, stream);
    }
    if (a.dtype == kBF16) return launch_partial<MmaFp8Policy<kBF16, 128>>(a, tmk, tmv, stream);
    return cudaErrorInvalidValue;
}

}  // namespace pkv
