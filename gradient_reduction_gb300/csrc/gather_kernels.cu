// All-gather (K shards -> K full replicas) and the flat-bucket gather of
// fragmented per-parameter gradients.  Both are bit copies bounded by HBM
// bandwidth: each source byte is read once, each destination byte written once.
#include "dpr_device.cuh"
#include "dpr_kernels.h"

namespace dpr {
namespace {

// ---- all-gather --------------------------------------------------------------
// Ring all-gather result (CMU 11-868 Lecture 14 notes, section 3.2; "Ring
// All-Reduce illustrated", Phase 2): every replica r receives every complete
// chunk j at position j*S.  grid.y = source shard j.  The in-place form
// shard[j] == out[j] + j*S is allowed, so loads use the coherent path.
__global__ void __launch_bounds__(kThreads) ag_vec(const __grid_constant__ AgParams p) {
    const int j = blockIdx.y, K = p.K;
    const uint16_t* const src = p.shard[j];
    const uint64_t base = uint64_t(j) * uint64_t(p.S);
    for (uint32_t t = blockIdx.x * kThreads + threadIdx.x; t < p.su; t += gridDim.x * kThreads) {
        const uint4 v = ld_v4(src + 8ull * t);
        const uint64_t e = base + 8ull * t;
#pragma unroll 8
        for (int r = 0; r < K; ++r) st_v4(p.out[r] + e, v);
    }
}

__global__ void __launch_bounds__(kThreads) ag_scalar(const __grid_constant__ AgParams p) {
    const int j = blockIdx.y, K = p.K;
    const uint64_t S = uint64_t(p.S), base = uint64_t(j) * S;
    const uint16_t* const src = p.shard[j];
    for (uint64_t t = uint64_t(blockIdx.x) * kThreads + threadIdx.x; t < S;
         t += uint64_t(gridDim.x) * kThreads) {
        const uint16_t v = src[t];
        for (int r = 0; r < K; ++r) p.out[r][base + t] = v;
    }
}

// ---- flat-bucket gather ----------------------------------------------------------
// DeepSpeed ZeRO-3 source walkthrough, sections 3.2 and 5.1: gradient p of a
// rank occupies [offset_p, offset_p + numel_p) of that rank's flat bucket.
// The plan cuts every (rank, gradient) segment into tiles of kFlatTile
// elements; blocks stride over the global tile index and find their segment
// by binary search over the segments' first-tile indices.

// Copies n elements of one tile.  When source and destination share their
// offset modulo 16 bytes the bulk moves as 16-byte vectors (a scalar head
// reaches the boundary, a scalar tail finishes), four vectors in flight per
// thread; otherwise element by element.
__device__ __forceinline__ void copy_tile(const uint16_t* src, uint16_t* dst, int64_t n) {
    const uintptr_t sa = reinterpret_cast<uintptr_t>(src);
    const uintptr_t da = reinterpret_cast<uintptr_t>(dst);
    if (((sa ^ da) & 15u) != 0) {
        for (int64_t i = threadIdx.x; i < n; i += kThreads) dst[i] = src[i];
        return;
    }
    int64_t h = int64_t(((16u - (sa & 15u)) & 15u) >> 1);
    if (h > n) h = n;
    if (threadIdx.x < h) dst[threadIdx.x] = src[threadIdx.x];
    const int64_t nv = (n - h) >> 3;
    const uint4* s4 = reinterpret_cast<const uint4*>(src + h);
    uint4* d4 = reinterpret_cast<uint4*>(dst + h);
    constexpr int U = 4;
    for (int64_t v0 = threadIdx.x; v0 < nv; v0 += U * kThreads) {
        uint4 x[U];
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v0 + u * kThreads < nv) x[u] = ld_nc_v4(s4 + v0 + u * kThreads);
#pragma unroll
        for (int u = 0; u < U; ++u)
            if (v0 + u * kThreads < nv) st_v4(d4 + v0 + u * kThreads, x[u]);
    }
    const int64_t done = h + nv * 8;
    if (threadIdx.x < n - done) dst[done + threadIdx.x] = src[done + threadIdx.x];
}

__global__ void __launch_bounds__(kThreads) flatten_kernel(const __grid_constant__ FlatParams p) {
    for (int64_t tile = blockIdx.x; tile < p.n_tiles; tile += gridDim.x) {
        int64_t lo = 0, hi = p.n_seg - 1;
        while (lo < hi) {
            const int64_t mid = (lo + hi + 1) >> 1;
            if (p.segs[mid].tile0 <= tile) lo = mid;
            else hi = mid - 1;
        }
        const FlatSeg sg = p.segs[lo];
        const int64_t t0 = (tile - sg.tile0) * kFlatTile;
        const int64_t rem = sg.numel - t0;
        const int64_t n = rem < kFlatTile ? rem : kFlatTile;
        copy_tile(sg.src + t0, p.dst[sg.rank] + sg.dst_off + t0, n);
    }
}

}  // namespace

cudaError_t launch_allgather(const AgParams& p, bool vec, cudaStream_t s) {
    const void* k = vec ? reinterpret_cast<const void*>(ag_vec)
                        : reinterpret_cast<const void*>(ag_scalar);
    int gx = 1;
    cudaError_t e = blocks_per_chunk(k, p.K, vec ? uint64_t(p.su) : uint64_t(p.S), &gx);
    if (e != cudaSuccess) return e;
    void* args[] = {const_cast<AgParams*>(&p)};
    return cudaLaunchKernel(k, dim3(gx, p.K), dim3(kThreads), args, 0, s);
}

cudaError_t launch_flatten(const FlatParams& p, cudaStream_t s) {
    const void* k = reinterpret_cast<const void*>(flatten_kernel);
    int g = 1;
    // one "chunk": blocks stride over all tiles
    cudaError_t e = blocks_per_chunk(k, 1, uint64_t(p.n_tiles) * kThreads, &g);
    if (e != cudaSuccess) return e;
    void* args[] = {const_cast<FlatParams*>(&p)};
    return cudaLaunchKernel(k, dim3(g), dim3(kThreads), args, 0, s);
}

}  // namespace dpr
