// CUDA-core (fp32 FMA) consumer of the split-context decode kernel.
//
// Each lane owns head_dim/32 consecutive dimensions: q (pre-multiplied by
// scale*log2(e)) and the output accumulator of all G heads of the group stay
// in registers.  Per token, the lanes' partial dot products for the G heads
// are summed with a reduce-scatter across the warp (G-1 + log2(32/G)
// shuffles), scores go to a per-warp scratch row, the tile's max and sum are
// taken, and the tile's V rows are accumulated with the softmax weights.
// Tiles arrive as plain contiguous bulk copies.
#include "decode_kernel.cuh"

namespace pkv {

template <int DT, int VD>
__device__ __forceinline__ void load_row(const typename Elem<DT>::T* p, float (&x)[VD]) {
    using T = typename Elem<DT>::T;
    if constexpr (sizeof(T) * VD == 16) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int i = 0; i < VD; ++i) x[i] = Elem<DT>::to_float(e[i]);
    } else if constexpr (sizeof(T) * VD == 8) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int i = 0; i < VD; ++i) x[i] = Elem<DT>::to_float(e[i]);
    } else {
        static_assert(sizeof(T) * VD == 4, "row slice must be 4, 8 or 16 bytes");
        const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
        const T* e = reinterpret_cast<const T*>(&u);
#pragma unroll
        for (int i = 0; i < VD; ++i) x[i] = Elem<DT>::to_float(e[i]);
    }
}

// Sum v[0..G) over the 32 lanes so that each lane ends with the total of one
// head; returns that head's index.  Halving exchanges first (each lane keeps
// the half of its values selected by one lane bit), then a plain butterfly.
template <int G>
__device__ __forceinline__ float reduce_scatter(float (&v)[G], int lane, int& head) {
    head = 0;
#pragma unroll
    for (int cnt = G, off = 16; cnt > 1; cnt >>= 1, off >>= 1) {
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < cnt / 2; ++i) {
            const float send = upper ? v[i] : v[i + cnt / 2];
            const float keep = upper ? v[i + cnt / 2] : v[i];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
        }
        if (upper) head += cnt / 2;
    }
    float x = v[0];
#pragma unroll
    for (int off = 16 / G; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, off));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
    return x;
}

template <int DT, int D, int G>
struct FfmaPolicy {
    static constexpr int kMaxThreads = 32 * 16;
    static constexpr bool kTensor = false;
    static constexpr bool kScratch = true;
    static constexpr bool kPairs = false;
    static constexpr int VD = D / 32;
    static constexpr int kD = D;
    using T = typename Elem<DT>::T;

    struct State {
        float q[G][VD];
        float o[G][VD];
        float m[G];
        float l[G];
    };

    __device__ __forceinline__ void begin(State& st, const DecodeArgs& a, int s, int h, int) {
        const int lane = threadIdx.x & 31;
        const T* q = static_cast<const T*>(a.q) +
                     (static_cast<int64_t>(s) * a.num_q_heads + h * G) * D + lane * VD;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float x[VD];
            load_row<DT, VD>(q + g * D, x);
#pragma unroll
            for (int i = 0; i < VD; ++i) {
                st.q[g][i] = x[i] * a.scale_log2;
                st.o[g][i] = 0.f;
            }
            st.m[g] = -INFINITY;
            st.l[g] = 0.f;
        }
    }

    // One head's part of a stage: kt/vt point at the stage's K/V, laid out as
    // [Hc][bs][D]; this warp's head is hw.
    __device__ __forceinline__ void tile(State& st, const DecodeArgs& a, const uint8_t* kt,
                                         const uint8_t* vt, int hw, int n_valid, int, float* sc) {
        const int lane = threadIdx.x & 31;
        const int64_t head_off = static_cast<int64_t>(hw) * a.block_size * D;
        const T* K = reinterpret_cast<const T*>(kt) + head_off + lane * VD;
        const T* V = reinterpret_cast<const T*>(vt) + head_off + lane * VD;
        // Scores (base-2 units) of every valid token, into scratch[t][g].
        for (int t = 0; t < n_valid; ++t) {
            float k[VD];
            load_row<DT, VD>(K + t * D, k);
            float d[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                float acc = 0.f;
#pragma unroll
                for (int i = 0; i < VD; ++i) acc = fmaf(st.q[g][i], k[i], acc);
                d[g] = acc;
            }
            int head;
            const float tot = reduce_scatter<G>(d, lane, head);
            if ((lane & (32 / G - 1)) == 0) sc[t * G + head] = tot;
        }
        __syncwarp();
        // Tile max per head, new running max, rescale, weights.
        float mx[G], alpha[G], ps[G];
#pragma unroll
        for (int g = 0; g < G; ++g) mx[g] = -INFINITY;
        for (int t = lane; t < n_valid; t += 32) {
#pragma unroll
            for (int g = 0; g < G; ++g) mx[g] = fmaxf(mx[g], sc[t * G + g]);
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float mn = fmaxf(st.m[g], warp_max(mx[g]));
            alpha[g] = fast_exp2(st.m[g] - mn);
            st.m[g] = mn;
            ps[g] = 0.f;
        }
        __syncwarp();
        for (int t = lane; t < n_valid; t += 32) {
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float p = fast_exp2(sc[t * G + g] - st.m[g]);
                sc[t * G + g] = p;
                ps[g] += p;
            }
        }
#pragma unroll
        for (int g = 0; g < G; ++g) {
            st.l[g] = st.l[g] * alpha[g] + warp_sum(ps[g]);
#pragma unroll
            for (int i = 0; i < VD; ++i) st.o[g][i] *= alpha[g];
        }
        __syncwarp();
        for (int t = 0; t < n_valid; ++t) {
            float v[VD];
            load_row<DT, VD>(V + t * D, v);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float p = sc[t * G + g];
#pragma unroll
                for (int i = 0; i < VD; ++i) st.o[g][i] = fmaf(p, v[i], st.o[g][i]);
            }
        }
        __syncwarp();
    }

    // 16-byte chunk q of row r of head hw's tile (plain [Hc][bs][D] layout).
    __device__ __forceinline__ void patch_chunk(const DecodeArgs& a, uint8_t* t, int hw, int r, int q,
                                                uint4 val) const {
        *(reinterpret_cast<uint4*>(t + (static_cast<int64_t>(hw) * a.block_size + r) * D * sizeof(T)) + q) = val;
    }

    // O (unnormalised) to o[g*os + d], (max, sum) to ml[g*ms], ml[g*ms + 1].
    __device__ __forceinline__ void emit(const State& st, float* o, int os, float* ml, int ms) const {
        const int lane = threadIdx.x & 31;
#pragma unroll
        for (int g = 0; g < G; ++g) {
#pragma unroll
            for (int i = 0; i < VD; ++i) o[g * os + lane * VD + i] = st.o[g][i];
            if (lane == 0) {
                ml[g * ms] = st.m[g];
                ml[g * ms + 1] = st.l[g];
            }
        }
    }

    __device__ __forceinline__ void write_state(const State& st, const DecodeArgs&, float* dst,
                                                int stride, int) const {
        emit(st, dst, stride, dst + D, stride);
    }

    __device__ __forceinline__ void write_partial(const State& st, const DecodeArgs&, float* o,
                                                  float* ml, int) const {
        emit(st, o, D, ml, 2);
    }

    // out[s][h*G + g][d] = O / l in the output type.
    __device__ __forceinline__ void write_final(const State& st, const DecodeArgs& a, int s, int h,
                                                int) const {
        const int lane = threadIdx.x & 31;
        const int64_t base = (static_cast<int64_t>(s) * a.num_q_heads + h * G) * D + lane * VD;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float inv = 1.f / st.l[g];
#pragma unroll
            for (int i = 0; i < VD; ++i) store_out(a.out, base + g * D + i, st.o[g][i] * inv, a.out_dtype);
        }
    }
};

template <int DT, int D, int G>
static cudaError_t launch_ffma_t(const DecodeArgs& a, cudaStream_t stream) {
    CUtensorMap none{};
    return launch_partial<FfmaPolicy<DT, D, G>>(a, none, none, stream);
}

template <int DT, int D>
static cudaError_t launch_ffma_g(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.num_q_heads / a.num_kv_heads) {
        case 1: return launch_ffma_t<DT, D, 1>(a, stream);
        case 2: return launch_ffma_t<DT, D, 2>(a, stream);
        case 4: return launch_ffma_t<DT, D, 4>(a, stream);
        case 8: return launch_ffma_t<DT, D, 8>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

template <int DT>
static cudaError_t launch_ffma_d(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.head_dim) {
        case 64: return launch_ffma_g<DT, 64>(a, stream);
        case 128: return launch_ffma_g<DT, 128>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_decode_ffma(const DecodeArgs& a, cudaStream_t stream) {
    switch (a.dtype) {
        case kF32: return launch_ffma_d<kF32>(a, stream);
        case kF16: return launch_ffma_d<kF16>(a, stream);
        case kBF16: return launch_ffma_d<kBF16>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pkv
