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
// Layout: grid.y = chunk j (so the ring's start rank is uniform per block);
// each thread owns one unit of 2W consecutive elements of its chunk (W = 8:
// 32-byte accesses, W = 4: 16-byte accesses), and there are as many blocks
// as units / 256 -- on GB300 this keeps more requests in flight than a
// persistent grid and streams HBM faster.  Element-wise kernels serve layouts
// that are not 16-byte aligned or chunks that are not a multiple of 8.
#include "dpr_device.cuh"
#include "dpr_kernels.h"

namespace dpr {
namespace {

// Folds the next addend (2W elements as W bf16x2 words) into the ring sum.
template <int MODE, int W>
__device__ __forceinline__ void ring_add(bool first, const uint32_t (&x)[W], float (&acc)[2 * W],
                                         uint32_t (&hop)[W]) {
    if constexpr (MODE == DPR_SUM_RING_FP32) {
#pragma unroll
        for (int k = 0; k < W; ++k) {
            if (first) {
                acc[2 * k] = bf_lo(x[k]);
                acc[2 * k + 1] = bf_hi(x[k]);
            } else {
                acc[2 * k] = __fadd_rn(acc[2 * k], bf_lo(x[k]));
                acc[2 * k + 1] = __fadd_rn(acc[2 * k + 1], bf_hi(x[k]));
            }
        }
    } else {
#pragma unroll
        for (int k = 0; k < W; ++k) hop[k] = first ? x[k] : add_bf16x2(hop[k], x[k]);
    }
}

// Ring-order sum of elements [e, e + 2W) of chunk j.  KC > 0: K = KC known at
// compile time; KC == 0: K at run time.  Loads are issued in groups of G
// ranks (all M micro-batches of each) before the group is added, keeping up
// to 256 bytes in flight per thread while the additions follow the ring.
// With M = 2 each rank's addend is first its local accumulation
// bf16(g0 + g1).
template <int KC, int M, int MODE, int W, bool NC>
__device__ __forceinline__ void ring_sum(const uint16_t* const* in, int K, int j, uint64_t e,
                                         float (&acc)[2 * W]) {
    constexpr int LOADS = (W == 8) ? 8 : 16;
    constexpr int G0 = LOADS / M;
    constexpr int G = (KC > 0 && KC < G0) ? KC : G0;
    static_assert(KC == 0 || KC % G == 0, "load groups must tile K");
    uint32_t hop[W];
#pragma unroll
    for (int k = 0; k < W; ++k) hop[k] = 0;
    const int Kr = KC > 0 ? KC : K;
#pragma unroll(KC > 0 ? 64 : 1)
    for (int g0 = 0; g0 < Kr; g0 += G) {
        uint32_t v[G][M][W];
#pragma unroll
        for (int s = 0; s < G; ++s) {
            if (KC > 0 || g0 + s < Kr) {
                int r = j + g0 + s;
                r = (r >= Kr) ? r - Kr : r;
#pragma unroll
                for (int m = 0; m < M; ++m) load_words<W, NC>(in[m * Kr + r] + e, v[s][m]);
            }
        }
#pragma unroll
        for (int s = 0; s < G; ++s) {
            if (KC > 0 || g0 + s < Kr) {
                uint32_t x[W];
#pragma unroll
                for (int k = 0; k < W; ++k)
                    x[k] = (M == 1) ? v[s][0][k] : add_bf16x2(v[s][0][k], v[s][M - 1][k]);
                ring_add<MODE, W>(g0 + s == 0, x, acc, hop);
            }
        }
    }
    if constexpr (MODE == DPR_SUM_HOP_BF16) {
#pragma unroll
        for (int k = 0; k < W; ++k) {
            acc[2 * k] = bf_lo(hop[k]);
            acc[2 * k + 1] = bf_hi(hop[k]);
        }
    }
}

// Scaled fp32 shard store of 2W values: out = acc*scale, or out + acc*scale
// (two roundings, never fused).
template <int W>
__device__ __forceinline__ void store_shard(float* o, const float (&acc)[2 * W], float scale,
                                            int accumulate) {
    float r[2 * W];
#pragma unroll
    for (int k = 0; k < 2 * W; ++k) r[k] = __fmul_rn(acc[k], scale);
    if (accumulate) {
#pragma unroll
        for (int q = 0; q < 2 * W; q += 4) {
            const float4 a = *reinterpret_cast<const float4*>(o + q);
            r[q] = __fadd_rn(a.x, r[q]);
            r[q + 1] = __fadd_rn(a.y, r[q + 1]);
            r[q + 2] = __fadd_rn(a.z, r[q + 2]);
            r[q + 3] = __fadd_rn(a.w, r[q + 3]);
        }
    }
    if constexpr (W == 8) {
        st_f8(o, r);
        st_f8(o + 8, r + 8);
    } else {
        st_f4(o, r[0], r[1], r[2], r[3]);
        st_f4(o + 4, r[4], r[5], r[6], r[7]);
    }
}

// ---- reduce-scatter ------------------------------------------------------------

template <int KC, int M, int MODE, int W>
__global__ void __launch_bounds__(kThreads) rs_vec(const __grid_constant__ RsParams p) {
    const uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x;
    if (t >= p.su) return;
    const int j = blockIdx.y;
    const uint64_t e = uint64_t(j) * uint64_t(p.S) + uint64_t(2 * W) * t;
    float acc[2 * W];
    ring_sum<KC, M, MODE, W, true>(p.in, p.K, j, e, acc);
    store_shard<W>(p.out[j] + uint64_t(2 * W) * t, acc, p.scale, p.accumulate);
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
template <int KC, int MODE, int W>
__global__ void __launch_bounds__(kThreads) ar_vec(const __grid_constant__ ArParams p) {
    const uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x;
    if (t >= p.su) return;
    const int j = blockIdx.y;
    const int K = KC > 0 ? KC : p.K;
    const uint64_t e = uint64_t(j) * uint64_t(p.S) + uint64_t(2 * W) * t;
    float acc[2 * W];
    ring_sum<KC, 1, MODE, W, false>(p.in, K, j, e, acc);
    const float s = p.scale;
    uint32_t w[W];
#pragma unroll
    for (int k = 0; k < W; ++k) w[k] = pack_bf16x2(__fmul_rn(acc[2 * k], s), __fmul_rn(acc[2 * k + 1], s));
#pragma unroll 8
    for (int r = 0; r < K; ++r) store_words<W>(p.out[r] + e, w);
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

// 32-byte kernels are specialised for the configured K; other K (and the
// 16-byte fallback) use the run-time-K form.
template <int M, int MODE>
const void* rs_kernel_for(int K, int W) {
    if (W == 4) return reinterpret_cast<const void*>(rs_vec<0, M, MODE, 4>);
    switch (K) {
        case 2: return reinterpret_cast<const void*>(rs_vec<2, M, MODE, 8>);
        case 4: return reinterpret_cast<const void*>(rs_vec<4, M, MODE, 8>);
        case 8: return reinterpret_cast<const void*>(rs_vec<8, M, MODE, 8>);
        case 16: return reinterpret_cast<const void*>(rs_vec<16, M, MODE, 8>);
        case 32: return reinterpret_cast<const void*>(rs_vec<32, M, MODE, 8>);
        case 64: return reinterpret_cast<const void*>(rs_vec<64, M, MODE, 8>);
        default: return reinterpret_cast<const void*>(rs_vec<0, M, MODE, 8>);
    }
}

template <int MODE>
const void* ar_kernel_for(int K, int W) {
    if (W == 4) return reinterpret_cast<const void*>(ar_vec<0, MODE, 4>);
    switch (K) {
        case 2: return reinterpret_cast<const void*>(ar_vec<2, MODE, 8>);
        case 4: return reinterpret_cast<const void*>(ar_vec<4, MODE, 8>);
        case 8: return reinterpret_cast<const void*>(ar_vec<8, MODE, 8>);
        case 16: return reinterpret_cast<const void*>(ar_vec<16, MODE, 8>);
        case 32: return reinterpret_cast<const void*>(ar_vec<32, MODE, 8>);
        case 64: return reinterpret_cast<const void*>(ar_vec<64, MODE, 8>);
        default: return reinterpret_cast<const void*>(ar_vec<0, MODE, 8>);
    }
}

}  // namespace

cudaError_t launch_reduce_scatter(const RsParams& p, int mode, int width, cudaStream_t s) {
    const void* k;
    dim3 grid;
    if (width > 0) {
        if (mode == DPR_SUM_RING_FP32)
            k = (p.M == 1) ? rs_kernel_for<1, DPR_SUM_RING_FP32>(p.K, width)
                           : rs_kernel_for<2, DPR_SUM_RING_FP32>(p.K, width);
        else
            k = (p.M == 1) ? rs_kernel_for<1, DPR_SUM_HOP_BF16>(p.K, width)
                           : rs_kernel_for<2, DPR_SUM_HOP_BF16>(p.K, width);
        grid = dim3(unsigned((uint64_t(p.su) + kThreads - 1) / kThreads), p.K);
    } else {
        k = (mode == DPR_SUM_RING_FP32) ? reinterpret_cast<const void*>(rs_scalar<DPR_SUM_RING_FP32>)
                                        : reinterpret_cast<const void*>(rs_scalar<DPR_SUM_HOP_BF16>);
        int gx = 1;
        cudaError_t e = blocks_per_chunk(k, p.K, uint64_t(p.S), &gx);
        if (e != cudaSuccess) return e;
        grid = dim3(gx, p.K);
    }
    void* args[] = {const_cast<RsParams*>(&p)};
    return cudaLaunchKernel(k, grid, dim3(kThreads), args, 0, s);
}

cudaError_t launch_allreduce(const ArParams& p, int mode, int width, cudaStream_t s) {
    const void* k;
    dim3 grid;
    if (width > 0) {
        k = (mode == DPR_SUM_RING_FP32) ? ar_kernel_for<DPR_SUM_RING_FP32>(p.K, width)
                                        : ar_kernel_for<DPR_SUM_HOP_BF16>(p.K, width);
        grid = dim3(unsigned((uint64_t(p.su) + kThreads - 1) / kThreads), p.K);
    } else {
        k = (mode == DPR_SUM_RING_FP32) ? reinterpret_cast<const void*>(ar_scalar<DPR_SUM_RING_FP32>)
                                        : reinterpret_cast<const void*>(ar_scalar<DPR_SUM_HOP_BF16>);
        int gx = 1;
        cudaError_t e = blocks_per_chunk(k, p.K, uint64_t(p.S), &gx);
        if (e != cudaSuccess) return e;
        grid = dim3(gx, p.K);
    }
    void* args[] = {const_cast<ArParams*>(&p)};
    return cudaLaunchKernel(k, grid, dim3(kThreads), args, 0, s);
}

}  // namespace dpr
