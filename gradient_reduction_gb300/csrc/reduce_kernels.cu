// Ring-order reduce-scatter (with micro-batch accumulation, averaging and the
// fp32 partition-gradient cast) and the fused all-reduce.
//
// The ring of the pages is a schedule of K-1 message rounds between K
// devices (CMU 11-868 Lecture 14 notes, section 3.2; "Ring All-Reduce
// illustrated", Phase 1).  Its arithmetic result is fixed by the order in
// which the partial sum of chunk j travels: it starts at rank j and collects
// ranks j+1, ..., j-1.  On one GPU all K rank buffers are resident, so the
// kernels do not pass chunks through memory round by round: every thread
// reads the K addends of its elements once and adds them in that same order
// in registers.  The result is bit-identical to the round-by-round ring and
// each input byte crosses HBM once.
//
// Layout: grid.y = chunk j (so the ring's start rank is uniform per block),
// grid.x blocks stride over the chunk's elements.  Vector kernels move 8
// bf16 elements (16 bytes) per rank per step; element-wise kernels serve
// unaligned layouts and chunks that are not a multiple of 8 elements.
#include "dpr_device.cuh"
#include "dpr_kernels.h"

namespace dpr {
namespace {

template <bool NC>
__device__ __forceinline__ uint4 load16(const uint16_t* p) {
    if constexpr (NC) return ld_nc_v4(p);
    else return ld_v4(p);
}

// x_r = bf16(g0_r + g1_r): rank-local accumulation of the micro-batches.
template <int M>
__device__ __forceinline__ uint4 local_accumulate(const uint4 (&v)[M]) {
    if constexpr (M == 1) return v[0];
    else return add_bf16x8(v[0], v[1]);
}

// Folds the next addend (already locally accumulated) into the ring sum.
template <int MODE>
__device__ __forceinline__ void ring_add(bool first, uint4 x, float (&acc)[8], uint4& hop) {
    if constexpr (MODE == DPR_SUM_RING_FP32) {
        float f[8];
        unpack8(x, f);
        if (first) {
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = f[k];
        } else {
#pragma unroll
            for (int k = 0; k < 8; ++k) acc[k] = __fadd_rn(acc[k], f[k]);
        }
    } else {
        hop = first ? x : add_bf16x8(hop, x);
    }
}

// Ring-order sum of elements [e, e+8) of chunk j over K ranks (K a compile-
// time constant).  Loads are issued in groups of G ranks (all micro-batches)
// before the group is added, so up to 16 16-byte loads are in flight per
// thread while the additions keep the exact ring order.
template <int K, int M, int MODE, bool NC>
__device__ __forceinline__ void ring_sum8(const uint16_t* const* in, int j, uint64_t e,
                                          float (&acc)[8]) {
    constexpr int G = (K * M <= 16) ? K : 16 / M;
    static_assert(K % G == 0, "group size must divide K");
    uint4 hop = make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int g0 = 0; g0 < K; g0 += G) {
        uint4 v[G][M];
#pragma unroll
        for (int s = 0; s < G; ++s) {
            int r = j + g0 + s;
            r = (r >= K) ? r - K : r;
#pragma unroll
            for (int m = 0; m < M; ++m) v[s][m] = load16<NC>(in[m * K + r] + e);
        }
#pragma unroll
        for (int s = 0; s < G; ++s) ring_add<MODE>(g0 + s == 0, local_accumulate<M>(v[s]), acc, hop);
    }
    if constexpr (MODE == DPR_SUM_HOP_BF16) unpack8(hop, acc);
}

// Same with K known only at run time (any 2 <= K <= 64).
template <int M, int MODE, bool NC>
__device__ __forceinline__ void ring_sum8_rt(const uint16_t* const* in, int K, int j,
                                             uint64_t e, float (&acc)[8]) {
    constexpr int G = 8;
    uint4 hop = make_uint4(0, 0, 0, 0);
    for (int g0 = 0; g0 < K; g0 += G) {
        uint4 v[G][M];
#pragma unroll
        for (int s = 0; s < G; ++s) {
            if (g0 + s < K) {
                int r = j + g0 + s;
                r = (r >= K) ? r - K : r;
#pragma unroll
                for (int m = 0; m < M; ++m) v[s][m] = load16<NC>(in[m * K + r] + e);
            }
        }
#pragma unroll
        for (int s = 0; s < G; ++s)
            if (g0 + s < K) ring_add<MODE>(g0 + s == 0, local_accumulate<M>(v[s]), acc, hop);
    }
    if constexpr (MODE == DPR_SUM_HOP_BF16) unpack8(hop, acc);
}

// Scaled fp32 shard store: out = acc*scale, or out + acc*scale (two roundings).
__device__ __forceinline__ void store_shard8(float* o, const float (&acc)[8], float scale,
                                             int accumulate) {
    float r[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) r[k] = __fmul_rn(acc[k], scale);
    if (accumulate) {
        const float4 a = *reinterpret_cast<const float4*>(o);
        const float4 b = *reinterpret_cast<const float4*>(o + 4);
        r[0] = __fadd_rn(a.x, r[0]); r[1] = __fadd_rn(a.y, r[1]);
        r[2] = __fadd_rn(a.z, r[2]); r[3] = __fadd_rn(a.w, r[3]);
        r[4] = __fadd_rn(b.x, r[4]); r[5] = __fadd_rn(b.y, r[5]);
        r[6] = __fadd_rn(b.z, r[6]); r[7] = __fadd_rn(b.w, r[7]);
    }
    st_f4(o, r[0], r[1], r[2], r[3]);
    st_f4(o + 4, r[4], r[5], r[6], r[7]);
}

// ---- reduce-scatter ------------------------------------------------------------

// KC > 0: K is the compile-time constant KC; KC == 0: K from the parameters.
template <int KC, int M, int MODE>
__global__ void __launch_bounds__(kThreads) rs_vec(const __grid_constant__ RsParams p) {
    const int j = blockIdx.y;
    const uint64_t base = uint64_t(j) * uint64_t(p.S);
    float* const out = p.out[j];
    for (uint32_t t = blockIdx.x * kThreads + threadIdx.x; t < p.su; t += gridDim.x * kThreads) {
        float acc[8];
        if constexpr (KC > 0) ring_sum8<KC, M, MODE, true>(p.in, j, base + 8ull * t, acc);
        else ring_sum8_rt<M, MODE, true>(p.in, p.K, j, base + 8ull * t, acc);
        store_shard8(out + 8ull * t, acc, p.scale, p.accumulate);
    }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) rs_scalar(const __grid_constant__ RsParams p) {
    const int j = blockIdx.y, K = p.K, M = p.M;
    const uint64_t S = uint64_t(p.S), base = uint64_t(j) * S;
    float* const out = p.out[j];
    for (uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x; t < S;
         t += uint64_t(gridDim.x) * kThreads) {
        const uint64_t e = base + t;
        float acc = 0.0f;
        uint16_t hop = 0;
        for (int s = 0; s < K; ++s) {
            int r = j + s;
            r = (r >= K) ? r - K : r;
            uint16_t x = p.in[r][e];
            if (M == 2) x = add_bf16(x, p.in[K + r][e]);
            if constexpr (MODE == DPR_SUM_RING_FP32) acc = (s == 0) ? bf_1(x) : __fadd_rn(acc, bf_1(x));
            else hop = (s == 0) ? x : add_bf16(hop, x);
        }
        if constexpr (MODE == DPR_SUM_HOP_BF16) acc = bf_1(hop);
        float v = __fmul_rn(acc, p.scale);
        if (p.accumulate) v = __fadd_rn(out[t], v);
        out[t] = v;
    }
}

// ---- all-reduce (fused reduce-scatter + all-gather) -----------------------------

// Inputs may be the outputs (in place): each thread reads all K addends of
// its elements before writing them, no other thread touches those elements,
// and the loads use the coherent path.
template <int KC, int MODE>
__global__ void __launch_bounds__(kThreads) ar_vec(const __grid_constant__ ArParams p) {
    const int j = blockIdx.y;
    const int K = KC > 0 ? KC : p.K;
    const uint64_t base = uint64_t(j) * uint64_t(p.S);
    for (uint32_t t = blockIdx.x * kThreads + threadIdx.x; t < p.su; t += gridDim.x * kThreads) {
        const uint64_t e = base + 8ull * t;
        float acc[8];
        if constexpr (KC > 0) ring_sum8<KC, 1, MODE, false>(p.in, j, e, acc);
        else ring_sum8_rt<1, MODE, false>(p.in, K, j, e, acc);
        const float s = p.scale;
        const uint4 w = make_uint4(pack_bf16x2(__fmul_rn(acc[0], s), __fmul_rn(acc[1], s)),
                                   pack_bf16x2(__fmul_rn(acc[2], s), __fmul_rn(acc[3], s)),
                                   pack_bf16x2(__fmul_rn(acc[4], s), __fmul_rn(acc[5], s)),
                                   pack_bf16x2(__fmul_rn(acc[6], s), __fmul_rn(acc[7], s)));
#pragma unroll 8
        for (int r = 0; r < K; ++r) st_v4(p.out[r] + e, w);
    }
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) ar_scalar(const __grid_constant__ ArParams p) {
    const int j = blockIdx.y, K = p.K;
    const uint64_t S = uint64_t(p.S), base = uint64_t(j) * S;
    for (uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x; t < S;
         t += uint64_t(gridDim.x) * kThreads) {
        const uint64_t e = base + t;
        float acc = 0.0f;
        uint16_t hop = 0;
        for (int s = 0; s < K; ++s) {
            int r = j + s;
            r = (r >= K) ? r - K : r;
            const uint16_t x = p.in[r][e];
            if constexpr (MODE == DPR_SUM_RING_FP32) acc = (s == 0) ? bf_1(x) : __fadd_rn(acc, bf_1(x));
            else hop = (s == 0) ? x : add_bf16(hop, x);
        }
        if constexpr (MODE == DPR_SUM_HOP_BF16) acc = bf_1(hop);
        const uint16_t v = to_bf16(__fmul_rn(acc, p.scale));
        for (int r = 0; r < K; ++r) p.out[r][e] = v;
    }
}

template <int M, int MODE>
const void* rs_vec_for(int K) {
    switch (K) {
        case 2: return reinterpret_cast<const void*>(rs_vec<2, M, MODE>);
        case 4: return reinterpret_cast<const void*>(rs_vec<4, M, MODE>);
        case 8: return reinterpret_cast<const void*>(rs_vec<8, M, MODE>);
        case 16: return reinterpret_cast<const void*>(rs_vec<16, M, MODE>);
        case 32: return reinterpret_cast<const void*>(rs_vec<32, M, MODE>);
        case 64: return reinterpret_cast<const void*>(rs_vec<64, M, MODE>);
        default: return reinterpret_cast<const void*>(rs_vec<0, M, MODE>);
    }
}

template <int MODE>
const void* ar_vec_for(int K) {
    switch (K) {
        case 2: return reinterpret_cast<const void*>(ar_vec<2, MODE>);
        case 4: return reinterpret_cast<const void*>(ar_vec<4, MODE>);
        case 8: return reinterpret_cast<const void*>(ar_vec<8, MODE>);
        case 16: return reinterpret_cast<const void*>(ar_vec<16, MODE>);
        case 32: return reinterpret_cast<const void*>(ar_vec<32, MODE>);
        case 64: return reinterpret_cast<const void*>(ar_vec<64, MODE>);
        default: return reinterpret_cast<const void*>(ar_vec<0, MODE>);
    }
}

}  // namespace

cudaError_t launch_reduce_scatter(const RsParams& p, int mode, bool vec, cudaStream_t s) {
    const void* k;
    if (vec) {
        if (mode == DPR_SUM_RING_FP32) k = (p.M == 1) ? rs_vec_for<1, DPR_SUM_RING_FP32>(p.K)
                                                      : rs_vec_for<2, DPR_SUM_RING_FP32>(p.K);
        else k = (p.M == 1) ? rs_vec_for<1, DPR_SUM_HOP_BF16>(p.K)
                            : rs_vec_for<2, DPR_SUM_HOP_BF16>(p.K);
    } else {
        k = (mode == DPR_SUM_RING_FP32) ? reinterpret_cast<const void*>(rs_scalar<DPR_SUM_RING_FP32>)
                                        : reinterpret_cast<const void*>(rs_scalar<DPR_SUM_HOP_BF16>);
    }
    int gx = 1;
    cudaError_t e = blocks_per_chunk(k, p.K, vec ? uint64_t(p.su) : uint64_t(p.S), &gx);
    if (e != cudaSuccess) return e;
    void* args[] = {const_cast<RsParams*>(&p)};
    return cudaLaunchKernel(k, dim3(gx, p.K), dim3(kThreads), args, 0, s);
}

cudaError_t launch_allreduce(const ArParams& p, int mode, bool vec, cudaStream_t s) {
    const void* k;
    if (vec) k = (mode == DPR_SUM_RING_FP32) ? ar_vec_for<DPR_SUM_RING_FP32>(p.K)
                                             : ar_vec_for<DPR_SUM_HOP_BF16>(p.K);
    else k = (mode == DPR_SUM_RING_FP32) ? reinterpret_cast<const void*>(ar_scalar<DPR_SUM_RING_FP32>)
                                         : reinterpret_cast<const void*>(ar_scalar<DPR_SUM_HOP_BF16>);
    int gx = 1;
    cudaError_t e = blocks_per_chunk(k, p.K, vec ? uint64_t(p.su) : uint64_t(p.S), &gx);
    if (e != cudaSuccess) return e;
    void* args[] = {const_cast<ArParams*>(&p)};
    return cudaLaunchKernel(k, dim3(gx, p.K), dim3(kThreads), args, 0, s);
}

}  // namespace dpr
