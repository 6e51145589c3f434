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
#include "dpr_ring.cuh"

namespace dpr {
namespace {

// ---- reduce-scatter ------------------------------------------------------------

// One unit per thread when the grid covers the chunk (the default launch);
// with a capped grid (a block budget, e.g. to leave SMs to concurrent
// compute) the same blocks stride over the remaining units.
template <int KC, int M, int MODE, int W>
__global__ void __launch_bounds__(kThreads) rs_vec(const __grid_constant__ RsParams p) {
    const int j = blockIdx.y;
    order_start(p.order);
    order_enter(p.order);
    for (uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x; t < p.su;
         t += uint64_t(gridDim.x) * kThreads) {
        const uint64_t e = uint64_t(j) * uint64_t(p.S) + uint64_t(2 * W) * t;
        float acc[2 * W];
        ring_sum<KC, M, MODE, W, true>(p.in, p.K, j, e, acc);
        store_shard<W>(p.out[j] + uint64_t(2 * W) * t, acc, p.scale, p.accumulate);
    }
    order_exit(p.order);
}

// bf16 partition shards (the ZeRO-3 partition buffer): the shard is rounded
// once to bf16, bf16(fp32(acc) * scale); with accumulate it is added in bf16
// to the existing shard, bf16(old + shard) (copy_ / add_ of the walkthrough's
// section 5.3).  RsParams::out holds bf16 buffers here.
template <int W>
__device__ __forceinline__ void store_shard_bf16(uint16_t* o, const float (&acc)[2 * W], float scale,
                                                 int accumulate) {
    uint32_t w[W];
#pragma unroll
    for (int k = 0; k < W; ++k)
        w[k] = pack_bf16x2(__fmul_rn(acc[2 * k], scale), __fmul_rn(acc[2 * k + 1], scale));
    if (accumulate) {
        uint32_t old[W];
        load_words<W, false>(o, old);
#pragma unroll
        for (int k = 0; k < W; ++k) w[k] = add_bf16x2(old[k], w[k]);
    }
    store_words<W>(o, w);
}

template <int KC, int M, int MODE, int W>
__global__ void __launch_bounds__(kThreads) rs_bf16_vec(const __grid_constant__ RsParams p) {
    const int j = blockIdx.y;
    uint16_t* const out = reinterpret_cast<uint16_t*>(p.out[j]);
    order_start(p.order);
    order_enter(p.order);
    for (uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x; t < p.su;
         t += uint64_t(gridDim.x) * kThreads) {
        const uint64_t e = uint64_t(j) * uint64_t(p.S) + uint64_t(2 * W) * t;
        float acc[2 * W];
        ring_sum<KC, M, MODE, W, true>(p.in, p.K, j, e, acc);
        store_shard_bf16<W>(out + uint64_t(2 * W) * t, acc, p.scale, p.accumulate);
    }
    order_exit(p.order);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) rs_bf16_scalar(const __grid_constant__ RsParams p) {
    const int j = blockIdx.y, K = p.K, M = p.M;
    const uint64_t S = uint64_t(p.S), base = uint64_t(j) * S;
    uint16_t* const out = reinterpret_cast<uint16_t*>(p.out[j]);
    order_start(p.order);
    order_enter(p.order);
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
        uint16_t v = to_bf16(__fmul_rn(acc, p.scale));
        if (p.accumulate) v = add_bf16(out[t], v);
        out[t] = v;
    }
    order_exit(p.order);
}

// step()-time cast of a bf16 partition to fp32 (exact widening); one unit of
// 16 elements per thread, 32-byte loads and stores when both buffers allow.
__global__ void __launch_bounds__(kThreads) cast_bf16_fp32(const uint16_t* __restrict__ in,
                                                           float* __restrict__ out, uint64_t n,
                                                           int vec) {
    order_enter(kAfterPrevious);
    const uint64_t u = uint64_t(blockIdx.x) * kThreads + threadIdx.x;
    const uint64_t e0 = 16 * u;
    if (e0 >= n) return;
    if (vec && e0 + 16 <= n) {
        uint32_t w[8];
        load_words<8, true>(in + e0, w);
        float f[16];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            f[2 * k] = bf_lo(w[k]);
            f[2 * k + 1] = bf_hi(w[k]);
        }
        st_f8(out + e0, f);
        st_f8(out + e0 + 8, f + 8);
        return;
    }
    for (uint64_t e = e0; e < n && e < e0 + 16; ++e) out[e] = bf_1(in[e]);
}

template <int MODE>
__global__ void __launch_bounds__(kThreads) rs_scalar(const __grid_constant__ RsParams p) {
    const int j = blockIdx.y, K = p.K, M = p.M;
    const uint64_t S = uint64_t(p.S), base = uint64_t(j) * S;
    float* const out = p.out[j];
    order_start(p.order);
    order_enter(p.order);
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
    order_exit(p.order);
}

// ---- all-reduce (fused reduce-scatter + all-gather) -----------------------------

// Inputs may be the outputs (in place): each thread reads all K addends of
// its elements before writing them, no other thread touches those elements,
// and the loads use the coherent path.
template <int KC, int MODE, int W>
__global__ void __launch_bounds__(kThreads) ar_vec(const __grid_constant__ ArParams p) {
    order_enter(p.order);
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
    order_enter(p.order);
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

// The vector kernels are specialised for the configured K (both access
// widths: 16-byte accesses serve chunks whose length is a multiple of 8 but
// not 16, such as 25,000,000 / 8); other K use the run-time-K form.
template <int M, int MODE, int W>
const void* rs_vec_for(int K) {
    switch (K) {
        case 2: return reinterpret_cast<const void*>(rs_vec<2, M, MODE, W>);
        case 4: return reinterpret_cast<const void*>(rs_vec<4, M, MODE, W>);
        case 8: return reinterpret_cast<const void*>(rs_vec<8, M, MODE, W>);
        case 16: return reinterpret_cast<const void*>(rs_vec<16, M, MODE, W>);
        case 32: return reinterpret_cast<const void*>(rs_vec<32, M, MODE, W>);
        case 64: return reinterpret_cast<const void*>(rs_vec<64, M, MODE, W>);
        default: return reinterpret_cast<const void*>(rs_vec<0, M, MODE, W>);
    }
}

template <int M, int MODE>
const void* rs_kernel_for(int K, int W) {
    return (W == 4) ? rs_vec_for<M, MODE, 4>(K) : rs_vec_for<M, MODE, 8>(K);
}

template <int M, int MODE>
const void* rs_bf16_kernel_for(int K, int W) {
    if (W == 4)
        return (K == 8) ? reinterpret_cast<const void*>(rs_bf16_vec<8, M, MODE, 4>)
                        : reinterpret_cast<const void*>(rs_bf16_vec<0, M, MODE, 4>);
    return (K == 8) ? reinterpret_cast<const void*>(rs_bf16_vec<8, M, MODE, 8>)
                    : reinterpret_cast<const void*>(rs_bf16_vec<0, M, MODE, 8>);
}

template <int MODE, int W>
const void* ar_vec_for(int K) {
    switch (K) {
        case 2: return reinterpret_cast<const void*>(ar_vec<2, MODE, W>);
        case 4: return reinterpret_cast<const void*>(ar_vec<4, MODE, W>);
        case 8: return reinterpret_cast<const void*>(ar_vec<8, MODE, W>);
        case 16: return reinterpret_cast<const void*>(ar_vec<16, MODE, W>);
        case 32: return reinterpret_cast<const void*>(ar_vec<32, MODE, W>);
        case 64: return reinterpret_cast<const void*>(ar_vec<64, MODE, W>);
        default: return reinterpret_cast<const void*>(ar_vec<0, MODE, W>);
    }
}

template <int MODE>
const void* ar_kernel_for(int K, int W) {
    return (W == 4) ? ar_vec_for<MODE, 4>(K) : ar_vec_for<MODE, 8>(K);
}

}  // namespace

cudaError_t launch_reduce_scatter(const RsParams& p, int mode, int width, cudaStream_t s,
                                  int max_blocks, bool programmatic) {
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
    if (max_blocks > 0) {
        const unsigned cap = unsigned(max_blocks / p.K > 0 ? max_blocks / p.K : 1);
        if (grid.x > cap) grid.x = cap;
    }
    void* args[] = {const_cast<RsParams*>(&p)};
    return launch_kernel(k, grid, args, s, programmatic);
}

cudaError_t launch_reduce_scatter_bf16(const RsParams& p, int mode, int width, cudaStream_t s) {
    const void* k;
    dim3 grid;
    if (width > 0) {
        if (mode == DPR_SUM_RING_FP32)
            k = (p.M == 1) ? rs_bf16_kernel_for<1, DPR_SUM_RING_FP32>(p.K, width)
                           : rs_bf16_kernel_for<2, DPR_SUM_RING_FP32>(p.K, width);
        else
            k = (p.M == 1) ? rs_bf16_kernel_for<1, DPR_SUM_HOP_BF16>(p.K, width)
                           : rs_bf16_kernel_for<2, DPR_SUM_HOP_BF16>(p.K, width);
        grid = dim3(unsigned((uint64_t(p.su) + kThreads - 1) / kThreads), p.K);
    } else {
        k = (mode == DPR_SUM_RING_FP32)
                ? reinterpret_cast<const void*>(rs_bf16_scalar<DPR_SUM_RING_FP32>)
                : reinterpret_cast<const void*>(rs_bf16_scalar<DPR_SUM_HOP_BF16>);
        int gx = 1;
        cudaError_t e = blocks_per_chunk(k, p.K, uint64_t(p.S), &gx);
        if (e != cudaSuccess) return e;
        grid = dim3(gx, p.K);
    }
    void* args[] = {const_cast<RsParams*>(&p)};
    return launch_kernel(k, grid, args, s);
}

cudaError_t launch_cast(const uint16_t* in, float* out, uint64_t n, bool vec, cudaStream_t s) {
    const uint64_t units = (n + 15) / 16;
    const unsigned blocks = unsigned((units + kThreads - 1) / kThreads);
    int v = vec ? 1 : 0;
    void* args[] = {&in, &out, &n, &v};
    return launch_kernel(reinterpret_cast<const void*>(cast_bf16_fp32), dim3(blocks), args, s);
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
    return launch_kernel(k, grid, args, s);
}

}  // namespace dpr
