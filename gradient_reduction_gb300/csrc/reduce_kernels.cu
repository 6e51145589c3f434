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
// 32-byte accesses, W = 4: 16-byte accesses; with W = 8 a chunk whose length
// is 8 more than a multiple of 16 has one 8-element unit at its unaligned
// end), and there are as many blocks as units / 256 -- on GB300 this keeps
// more requests in flight than a persistent grid and streams HBM faster.
// Element-wise kernels serve layouts that are not 16-byte aligned or chunks
// that are not a multiple of 8.
#include "dpr_device.cuh"
#include "dpr_kernels.h"
#include "dpr_ring.cuh"

namespace dpr {
namespace {

// ---- reduce-scatter ------------------------------------------------------------

// One unit per thread when the grid covers the chunk (the default launch);
// with a capped grid (a block budget, e.g. to leave SMs to concurrent
// compute) the same blocks stride over the remaining units.
//
// EDGE (rs_vec_edge; p.edge, see edge_unit(): S % 16 == 8, 32-byte aligned
// buffers, K even): chunk j starts 8 elements past a 32-byte boundary when j
// is odd, so its 32-byte units start 8 elements in, and the chunk's last unit
// is a 32-byte window around the 8 elements left over -- the head of an odd
// chunk, [c0 - 8, c0 + 8), or the tail of an even one, [c0 + S - 8,
// c0 + S + 8).  The window's other 8 elements belong to the neighbouring
// chunk, inside the buffer (an odd chunk has a chunk before it; with K even
// an even chunk has one after it); the inputs are read-only here, those 8
// sums are dropped and only the chunk's own 8 are stored.  The edge unit thus
// runs the same 32-byte code as every other unit.  The kernel is capped at 64
// registers (4 blocks per SM); for the K it is built for it spills at most 4
// bytes.
template <int KC, int M, int MODE, int W, bool EDGE>
__device__ __forceinline__ void rs_units(const RsParams& p) {
    static_assert(!EDGE || W == 8, "the edge layout has 32-byte units");
    const int j = blockIdx.y;
    order_start(p.order);
    order_enter(p.order);
    if constexpr (EDGE) {
        const uint64_t c0 = uint64_t(j) * uint64_t(p.S);
        const bool odd = (c0 & 15) != 0;
        const uint64_t body = uint64_t(p.su) - 1;
        for (uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x; t < p.su;
             t += uint64_t(gridDim.x) * kThreads) {
            const bool edge = t == body;
            // one summation per unit (a second call site would double the registers)
            const uint64_t win = edge ? (odd ? c0 - 8 : c0 + uint64_t(p.S) - 8)
                                      : c0 + (odd ? 8 : 0) + 16 * t;
            float acc[16];
            ring_sum<KC, M, MODE, 8, true>(p.in, p.K, j, win, acc);
            if (edge) {
                float mine[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mine[k] = odd ? acc[8 + k] : acc[k];
                store_shard<4>(p.out[j] + (odd ? 0 : uint64_t(p.S) - 8), mine, p.scale,
                               p.accumulate);
            } else {
                store_shard<8>(p.out[j] + (win - c0), acc, p.scale, p.accumulate);
            }
        }
    } else {
        for (uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x; t < p.su;
             t += uint64_t(gridDim.x) * kThreads) {
            const uint64_t e = uint64_t(j) * uint64_t(p.S) + uint64_t(2 * W) * t;
            float acc[2 * W];
            ring_sum<KC, M, MODE, W, true>(p.in, p.K, j, e, acc);
            store_shard<W>(p.out[j] + uint64_t(2 * W) * t, acc, p.scale, p.accumulate);
        }
    }
    order_exit(p.order);
}

template <int KC, int M, int MODE, int W>
__global__ void __launch_bounds__(kThreads) rs_vec(const __grid_constant__ RsParams p) {
    rs_units<KC, M, MODE, W, false>(p);
}

template <int KC, int M, int MODE>
__global__ void __launch_bounds__(kThreads, 4) rs_vec_edge(const __grid_constant__ RsParams p) {
    rs_units<KC, M, MODE, 8, true>(p);
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
// The all-reduce of 16 elements from e: ring sum, scale, bf16.
template <int KC, int MODE>
__device__ __forceinline__ void ar_words(const ArParams& p, int K, int j, uint64_t e,
                                         uint32_t (&w)[8]) {
    float acc[16];
    ring_sum<KC, 1, MODE, 8, false>(p.in, K, j, e, acc);
    const float s = p.scale;
#pragma unroll
    for (int k = 0; k < 8; ++k) w[k] = pack_bf16x2(__fmul_rn(acc[2 * k], s), __fmul_rn(acc[2 * k + 1], s));
}

// EDGE as in rs_vec, for out-of-place calls only (an in-place call writes the
// inputs, so no unit may read a neighbouring chunk's elements): the window's
// own 8 elements are stored, with 16-byte stores.
template <int KC, int MODE, int W, bool EDGE>
__device__ __forceinline__ void ar_units(const ArParams& p) {
    static_assert(!EDGE || W == 8, "the edge layout has 32-byte units");
    order_enter(p.order);
    const uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x;
    if (t >= p.su) return;
    const int j = blockIdx.y;
    const int K = KC > 0 ? KC : p.K;
    const uint64_t c0 = uint64_t(j) * uint64_t(p.S);
    if constexpr (EDGE) {
        const bool odd = (c0 & 15) != 0;
        const bool edge = t + 1 == uint64_t(p.su);
        const uint64_t win = edge ? (odd ? c0 - 8 : c0 + uint64_t(p.S) - 8)
                                  : c0 + (odd ? 8 : 0) + 16 * t;
        uint32_t w[8];
        ar_words<KC, MODE>(p, K, j, win, w);
        if (edge) {
            uint32_t mine[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) mine[k] = odd ? w[4 + k] : w[k];
            const uint64_t e = odd ? c0 : c0 + uint64_t(p.S) - 8;
#pragma unroll 8
            for (int r = 0; r < K; ++r) store_words<4>(p.out[r] + e, mine);
            return;
        }
#pragma unroll 8
        for (int r = 0; r < K; ++r) store_words<8>(p.out[r] + win, w);
        return;
    }
    const uint64_t e = c0 + uint64_t(2 * W) * t;
    float acc[2 * W];
    ring_sum<KC, 1, MODE, W, false>(p.in, K, j, e, acc);
    const float s = p.scale;
    uint32_t w[W];
#pragma unroll
    for (int k = 0; k < W; ++k) w[k] = pack_bf16x2(__fmul_rn(acc[2 * k], s), __fmul_rn(acc[2 * k + 1], s));
#pragma unroll 8
    for (int r = 0; r < K; ++r) store_words<W>(p.out[r] + e, w);
}

template <int KC, int MODE, int W>
__global__ void __launch_bounds__(kThreads) ar_vec(const __grid_constant__ ArParams p) {
    ar_units<KC, MODE, W, false>(p);
}

template <int KC, int MODE>
__global__ void __launch_bounds__(kThreads, 4) ar_vec_edge(const __grid_constant__ ArParams p) {
    ar_units<KC, MODE, 8, true>(p);
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
// widths: 16-byte accesses serve buffers that are 16- but not 32-byte
// aligned); other K use the run-time-K form.
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

// The edge layout exists for the K that edge_unit() admits for the
// reduce-scatter (2-32); other K never set RsParams::edge.
template <int M, int MODE>
const void* rs_edge_for(int K) {
    switch (K) {
        case 2: return reinterpret_cast<const void*>(rs_vec_edge<2, M, MODE>);
        case 4: return reinterpret_cast<const void*>(rs_vec_edge<4, M, MODE>);
        case 8: return reinterpret_cast<const void*>(rs_vec_edge<8, M, MODE>);
        case 16: return reinterpret_cast<const void*>(rs_vec_edge<16, M, MODE>);
        case 32: return reinterpret_cast<const void*>(rs_vec_edge<32, M, MODE>);
        default: return nullptr;
    }
}

template <int M, int MODE>
const void* rs_kernel_for(int K, int W, bool edge) {
    if (edge) return rs_edge_for<M, MODE>(K);
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

// The all-reduce's edge layout exists for K = 2, 4, 8 (edge_unit()).
template <int MODE>
const void* ar_edge_for(int K) {
    switch (K) {
        case 2: return reinterpret_cast<const void*>(ar_vec_edge<2, MODE>);
        case 4: return reinterpret_cast<const void*>(ar_vec_edge<4, MODE>);
        case 8: return reinterpret_cast<const void*>(ar_vec_edge<8, MODE>);
        default: return nullptr;
    }
}

template <int MODE>
const void* ar_kernel_for(int K, int W, bool edge) {
    if (edge) return ar_edge_for<MODE>(K);
    return (W == 4) ? ar_vec_for<MODE, 4>(K) : ar_vec_for<MODE, 8>(K);
}

}  // namespace

cudaError_t launch_reduce_scatter(const RsParams& p, int mode, int width, cudaStream_t s,
                                  int max_blocks, bool programmatic) {
    const void* k;
    dim3 grid;
    if (width > 0) {
        const bool edge = p.edge != 0;
        if (mode == DPR_SUM_RING_FP32)
            k = (p.M == 1) ? rs_kernel_for<1, DPR_SUM_RING_FP32>(p.K, width, edge)
                           : rs_kernel_for<2, DPR_SUM_RING_FP32>(p.K, width, edge);
        else
            k = (p.M == 1) ? rs_kernel_for<1, DPR_SUM_HOP_BF16>(p.K, width, edge)
                           : rs_kernel_for<2, DPR_SUM_HOP_BF16>(p.K, width, edge);
        if (!k) return cudaErrorInvalidDeviceFunction;   // an edge layout edge_unit() never sets
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
        k = (mode == DPR_SUM_RING_FP32) ? ar_kernel_for<DPR_SUM_RING_FP32>(p.K, width, p.edge != 0)
                                        : ar_kernel_for<DPR_SUM_HOP_BF16>(p.K, width, p.edge != 0);
        if (!k) return cudaErrorInvalidDeviceFunction;   // an edge layout edge_unit() never sets
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
