// Per-parameter (ZeRO-3) partitioning: reduce-scatter of fragmented
// per-parameter gradients into per-parameter shards, and the all-gather that
// rebuilds full parameters from them.
//
// DeepSpeed ZeRO-3 source walkthrough, section 1: each parameter lives as a
// 1/N shard per rank; section 5.2: the discrete path reduce-scatters the
// list of fragmented gradients (no flat bucket).  Parameter p of numel n_p is
// treated as zero-padded to K * s_p, s_p = ceil(n_p / K); rank j owns
// elements [j*s_p, (j+1)*s_p); rank j's partition buffer holds its shards of
// every parameter in parameter order (offset_p = sum_{q<p} s_q).  Each shard
// is the ring-order sum of section 3.2 of the CMU 11-868 Lecture 14 notes,
// starting at rank j.
//
// Work is cut into (parameter, shard) segments and tiles of kCoalTile
// elements; one block handles one tile (and, for the all-gather, one
// replica).  A per-tile map gives each block its segment and parameter in one
// load, so the segment record and the tensor pointers arrive together, two
// dependent loads before the first data load.
#include <algorithm>
#include <cstring>
#include <new>
#include <vector>

#include "dpr_device.cuh"
#include "dpr_kernels.h"
#include "dpr_ring.cuh"
#include "host_checks.h"

namespace dpr {
namespace {

#ifndef DPR_COAL_TILE
#define DPR_COAL_TILE 4096
#endif
constexpr int64_t kCoalTile = DPR_COAL_TILE;   // reduce-scatter tile: K * 2 * kCoalTile bytes read per block
constexpr int64_t kCoalAgTile = 8192;   // all-gather tile: 16 KB written per block

struct CoalSeg {
    int64_t s;        // shard length of the parameter, ceil(n / K)
    int64_t valid;    // elements of this shard inside the parameter (<= s)
    int64_t off;      // offset of the parameter's shard in every partition
    int64_t tile0;    // first reduce-scatter tile of this segment
    int64_t ag_tile0; // first all-gather tile of this segment
    int32_t p;        // parameter
    int32_t j;        // shard (= partition / owning rank)
    int32_t vec;      // every rank's tensor at j*s is 32-byte aligned, s and off % 16 == 0
    int32_t pad;
};

struct TileRef {
    int32_t seg;      // segment of the tile
    int32_t p;        // its parameter (= segs[seg].p, here so the pointer load need not wait)
};

struct CoalParams {
    const CoalSeg* segs;
    const TileRef* tiles;           // reduce-scatter tiles, or all-gather tiles
    uint16_t* const* ptrs;          // device table [K * P]: tensors[r * P + p]
    int64_t n_tiles;
    float* out[DPR_MAX_RANKS];      // reduce-scatter: fp32 partitions
    const uint16_t* shard[DPR_MAX_RANKS];   // all-gather: bf16 partitions
    int K;
    int P;
    float scale;
    int accumulate;
    int bases_aligned32;            // every out / shard base is 32-byte aligned
    int order;                      // kAfterPrevious
};

// KC > 0: K = KC fixed at compile time (the ring's loads and adds unrolled,
// about half the registers of the run-time-K form); KC == 0: any K.
template <int KC, int MODE>
__global__ void __launch_bounds__(kThreads) rs_coalesced(const __grid_constant__ CoalParams p) {
    __shared__ const uint16_t* base[DPR_MAX_RANKS];
    const int64_t tile = blockIdx.x;
    const TileRef tr = p.tiles[tile];
    const int K = KC > 0 ? KC : p.K;
    const uint16_t* t = (threadIdx.x < K) ? p.ptrs[int64_t(threadIdx.x) * p.P + tr.p] : nullptr;
    const CoalSeg sg = p.segs[tr.seg];
    if (threadIdx.x < K) base[threadIdx.x] = t + sg.j * sg.s;
    __syncthreads();
    order_enter(p.order);           // the plan's tables above are fixed; the buffers are not
    const int64_t t0 = (tile - sg.tile0) * kCoalTile;
    const int64_t n = (sg.s - t0 < kCoalTile) ? sg.s - t0 : kCoalTile;
    float* out = p.out[sg.j] + sg.off + t0;
    if (sg.vec && p.bases_aligned32 && t0 + n <= sg.valid) {
        // whole tile inside the parameter: 16 elements per thread and access
        for (int64_t u = threadIdx.x; u < n / 16; u += kThreads) {
            float acc[16];
            ring_sum<KC, 1, MODE, 8, true>(base, K, sg.j, uint64_t(t0 + 16 * u), acc);
            store_shard<8>(out + 16 * u, acc, p.scale, p.accumulate);
        }
        return;
    }
    // element-wise, with the zero padding past the end of the parameter
    for (int64_t i = threadIdx.x; i < n; i += kThreads) {
        const int64_t e = t0 + i;
        const bool in = e < sg.valid;
        float acc = 0.0f;
        uint16_t hop = 0;
        for (int k = 0; k < K; ++k) {
            int r = sg.j + k;
            r = (r >= K) ? r - K : r;
            const uint16_t x = in ? base[r][e] : uint16_t(0);
            if constexpr (MODE == DPR_SUM_RING_FP32) acc = (k == 0) ? bf_1(x) : __fadd_rn(acc, bf_1(x));
            else hop = (k == 0) ? x : add_bf16(hop, x);
        }
        if constexpr (MODE == DPR_SUM_HOP_BF16) acc = bf_1(hop);
        float v = __fmul_rn(acc, p.scale);
        if (p.accumulate) v = __fadd_rn(out[i], v);
        out[i] = v;
    }
}

// One block per (tile, replica r); the K replicas of a tile are adjacent so
// the shard tile is read from HBM once.  Only the shard's elements inside the
// parameter are written (padding is dropped).
__global__ void __launch_bounds__(kThreads) ag_coalesced(const __grid_constant__ CoalParams p) {
    const uint64_t b = blockIdx.x;
    const int r = int(b % uint64_t(p.K));
    const int64_t tile = int64_t(b / uint64_t(p.K));
    const TileRef tr = p.tiles[tile];
    uint16_t* const t = p.ptrs[int64_t(r) * p.P + tr.p];
    const CoalSeg sg = p.segs[tr.seg];
    order_enter(p.order);
    const int64_t t0 = (tile - sg.ag_tile0) * kCoalAgTile;
    const int64_t n = (sg.valid - t0 < kCoalAgTile) ? sg.valid - t0 : kCoalAgTile;
    if (n <= 0) return;
    const uint16_t* src = p.shard[sg.j] + sg.off + t0;
    uint16_t* dst = t + sg.j * sg.s + t0;
    if (sg.vec && p.bases_aligned32 && n == kCoalAgTile) {
#pragma unroll
        for (int u = 0; u < int(kCoalAgTile) / 16 / kThreads; ++u) {
            const int i = (u * kThreads + int(threadIdx.x)) * 16;
            uint32_t w[8];
            load_words<8, true>(src + i, w);
            store_words<8>(dst + i, w);
        }
        return;
    }
    for (int64_t i = threadIdx.x; i < n; i += kThreads) dst[i] = src[i];
}

template <int MODE>
const void* rs_coalesced_for(int K) {
    switch (K) {
        case 2: return reinterpret_cast<const void*>(rs_coalesced<2, MODE>);
        case 4: return reinterpret_cast<const void*>(rs_coalesced<4, MODE>);
        case 8: return reinterpret_cast<const void*>(rs_coalesced<8, MODE>);
        case 16: return reinterpret_cast<const void*>(rs_coalesced<16, MODE>);
        case 32: return reinterpret_cast<const void*>(rs_coalesced<32, MODE>);
        case 64: return reinterpret_cast<const void*>(rs_coalesced<64, MODE>);
        default: return reinterpret_cast<const void*>(rs_coalesced<0, MODE>);
    }
}

dpr_status coal_cuda(cudaError_t e) { return record_cuda_status(e); }

}  // namespace
}  // namespace dpr

using namespace dpr;

struct dpr_coalesced_plan {
    int K = 0;
    int P = 0;
    int device = 0;
    int64_t partition_numel = 0;
    int64_t n_tiles = 0;
    int64_t n_ag_tiles = 0;
    std::vector<int64_t> numel;
    std::vector<CoalSeg> segs;
    std::vector<Span> tensor_spans;
    CoalSeg* d_segs = nullptr;
    TileRef* d_tiles = nullptr;      // [n_tiles]
    TileRef* d_ag_tiles = nullptr;   // [n_ag_tiles]
    uint16_t** d_ptrs = nullptr;
};

namespace {

void free_plan(dpr_coalesced_plan* pl) {
    if (pl->d_segs) cudaFree(pl->d_segs);
    if (pl->d_tiles) cudaFree(pl->d_tiles);
    if (pl->d_ag_tiles) cudaFree(pl->d_ag_tiles);
    if (pl->d_ptrs) cudaFree(pl->d_ptrs);
    delete pl;
}

}  // namespace

extern "C" {

dpr_status dpr_coalesced_plan_create(dpr_coalesced_plan** plan, int K, int P,
                                     void* const* tensors, const int64_t* numel, void* stream) {
    if (!plan) return DPR_ERR_INVALID_ARG;
    *plan = nullptr;
    if (K < 2 || K > DPR_MAX_RANKS || P < 0) return DPR_ERR_INVALID_ARG;
    if (P > 0 && (!tensors || !numel)) return DPR_ERR_INVALID_ARG;
    std::vector<Span> spans;
    for (int p = 0; p < P; ++p) {
        if (numel[p] < 0) return DPR_ERR_INVALID_ARG;
        if (numel[p] > DPR_MAX_ELEMS) return DPR_ERR_UNSUPPORTED;
        for (int r = 0; r < K; ++r) {
            const void* t = tensors[size_t(r) * P + p];
            if (numel[p] == 0) continue;
            if (!t) return DPR_ERR_INVALID_ARG;
            if (!aligned(t, 2)) return DPR_ERR_ALIGNMENT;
            const uintptr_t a = reinterpret_cast<uintptr_t>(t);
            spans.push_back(Span{a, a + uintptr_t(numel[p]) * 2});
        }
    }
    // the all-gather writes these tensors: they must not overlap
    std::vector<Span> sorted = spans;
    std::sort(sorted.begin(), sorted.end(), [](const Span& a, const Span& b) { return a.lo < b.lo; });
    for (size_t i = 1; i < sorted.size(); ++i)
        if (sorted[i].lo < sorted[i - 1].hi) return DPR_ERR_ALIAS;

    dpr_coalesced_plan* pl = new (std::nothrow) dpr_coalesced_plan();
    if (!pl) return DPR_ERR_CUDA;
    pl->K = K;
    pl->P = P;
    pl->numel.assign(numel, numel + P);
    pl->tensor_spans = spans;
    int64_t off = 0, tiles = 0, ag_tiles = 0;
    for (int p = 0; p < P; ++p) {
        const int64_t s = (numel[p] + K - 1) / K;
        if (s == 0) continue;
        for (int j = 0; j < K; ++j) {
            CoalSeg g;
            g.s = s;
            g.valid = std::max<int64_t>(0, std::min<int64_t>(s, numel[p] - int64_t(j) * s));
            g.off = off;
            g.tile0 = tiles;
            g.ag_tile0 = ag_tiles;
            g.p = p;
            g.j = j;
            bool vec = (s % 16 == 0) && (off % 16 == 0);
            for (int r = 0; r < K && vec; ++r)
                vec = aligned(static_cast<const uint16_t*>(tensors[size_t(r) * P + p]) + j * s, 32);
            g.vec = vec ? 1 : 0;
            g.pad = 0;
            tiles += (s + kCoalTile - 1) / kCoalTile;
            ag_tiles += (s + kCoalAgTile - 1) / kCoalAgTile;
            pl->segs.push_back(g);
        }
        off += s;
    }
    pl->partition_numel = off;
    pl->n_tiles = tiles;
    pl->n_ag_tiles = ag_tiles;
    // one block per reduce-scatter tile and per (all-gather tile, replica):
    // both must fit a 1-D grid
    if (tiles > int64_t(0x7FFFFFFF) || ag_tiles * K > int64_t(0x7FFFFFFF)) {
        free_plan(pl);
        return DPR_ERR_UNSUPPORTED;
    }
    cudaError_t e = cudaGetDevice(&pl->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (e == cudaSuccess && !pl->segs.empty()) {
        std::vector<TileRef> map(static_cast<size_t>(tiles)), ag_map(static_cast<size_t>(ag_tiles));
        for (size_t g = 0; g < pl->segs.size(); ++g) {
            const CoalSeg& sg = pl->segs[g];
            const TileRef ref{int32_t(g), sg.p};
            std::fill_n(map.begin() + sg.tile0, (sg.s + kCoalTile - 1) / kCoalTile, ref);
            std::fill_n(ag_map.begin() + sg.ag_tile0, (sg.s + kCoalAgTile - 1) / kCoalAgTile, ref);
        }
        std::vector<uint16_t*> ptrs(size_t(K) * P);
        for (size_t i = 0; i < ptrs.size(); ++i) ptrs[i] = static_cast<uint16_t*>(tensors[i]);
        e = upload(&pl->d_segs, pl->segs, st);
        if (e == cudaSuccess) e = upload(&pl->d_tiles, map, st);
        if (e == cudaSuccess) e = upload(&pl->d_ag_tiles, ag_map, st);
        if (e == cudaSuccess) e = upload(&pl->d_ptrs, ptrs, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    if (e != cudaSuccess) {
        free_plan(pl);
        return coal_cuda(e);
    }
    *plan = pl;
    return DPR_OK;
}

dpr_status dpr_coalesced_partition_numel(const dpr_coalesced_plan* plan, int64_t* numel) {
    if (!plan || !numel) return DPR_ERR_INVALID_ARG;
    *numel = plan->partition_numel;
    return DPR_OK;
}

dpr_status dpr_reduce_scatter_coalesced(const dpr_coalesced_plan* plan, float* const* out,
                                        int mode, float scale, int accumulate, void* stream) {
    if (!plan || !out) return DPR_ERR_INVALID_ARG;
    if (mode != DPR_SUM_RING_FP32 && mode != DPR_SUM_HOP_BF16) return DPR_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return coal_cuda(e);
    if (dev != plan->device) return DPR_ERR_INVALID_ARG;
    const int K = plan->K;
    bool a32 = true;
    std::vector<Span> outs;
    for (int j = 0; j < K; ++j) {
        if (!out[j]) return DPR_ERR_INVALID_ARG;
        if (!aligned(out[j], 4)) return DPR_ERR_ALIGNMENT;
        a32 = a32 && aligned(out[j], 32);
        const uintptr_t a = reinterpret_cast<uintptr_t>(out[j]);
        outs.push_back(Span{a, a + uintptr_t(plan->partition_numel) * 4});
    }
    for (int j = 0; j < K; ++j)
        for (int q = j + 1; q < K; ++q)
            if (overlaps(outs[j], outs[q])) return DPR_ERR_ALIAS;
    for (const Span& t : plan->tensor_spans)
        for (const Span& o : outs)
            if (overlaps(t, o)) return DPR_ERR_ALIAS;
    if (plan->n_tiles == 0) return DPR_OK;
    CoalParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.segs = plan->d_segs;
    prm.tiles = plan->d_tiles;
    prm.ptrs = plan->d_ptrs;
    prm.n_tiles = plan->n_tiles;
    for (int j = 0; j < K; ++j) prm.out[j] = out[j];
    prm.K = K;
    prm.P = plan->P;
    prm.scale = scale;
    prm.accumulate = accumulate ? 1 : 0;
    prm.bases_aligned32 = a32 ? 1 : 0;
    const void* k = (mode == DPR_SUM_RING_FP32) ? rs_coalesced_for<DPR_SUM_RING_FP32>(K)
                                                : rs_coalesced_for<DPR_SUM_HOP_BF16>(K);
    void* args[] = {&prm};
    return coal_cuda(launch_kernel(k, dim3(unsigned(plan->n_tiles)), args,
                                   static_cast<cudaStream_t>(stream)));
}

dpr_status dpr_allgather_coalesced(const dpr_coalesced_plan* plan, const void* const* shards,
                                   void* stream) {
    if (!plan || !shards) return DPR_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return coal_cuda(e);
    if (dev != plan->device) return DPR_ERR_INVALID_ARG;
    const int K = plan->K;
    bool a32 = true;
    for (int j = 0; j < K; ++j) {
        if (!shards[j]) return DPR_ERR_INVALID_ARG;
        if (!aligned(shards[j], 2)) return DPR_ERR_ALIGNMENT;
        a32 = a32 && aligned(shards[j], 32);
        const uintptr_t a = reinterpret_cast<uintptr_t>(shards[j]);
        const Span sp{a, a + uintptr_t(plan->partition_numel) * 2};
        for (const Span& t : plan->tensor_spans)
            if (overlaps(t, sp)) return DPR_ERR_ALIAS;
    }
    if (plan->n_tiles == 0) return DPR_OK;
    CoalParams prm;
    std::memset(&prm, 0, sizeof(prm));
    prm.segs = plan->d_segs;
    prm.tiles = plan->d_ag_tiles;
    prm.ptrs = plan->d_ptrs;
    prm.n_tiles = plan->n_ag_tiles;
    for (int j = 0; j < K; ++j) prm.shard[j] = static_cast<const uint16_t*>(shards[j]);
    prm.K = K;
    prm.P = plan->P;
    prm.bases_aligned32 = a32 ? 1 : 0;
    const uint64_t blocks = uint64_t(plan->n_ag_tiles) * uint64_t(K);
    void* args[] = {&prm};
    return coal_cuda(launch_kernel(reinterpret_cast<const void*>(ag_coalesced),
                                   dim3(unsigned(blocks)), args, static_cast<cudaStream_t>(stream)));
}

dpr_status dpr_coalesced_plan_destroy(dpr_coalesced_plan* plan) {
    if (!plan) return DPR_OK;
    cudaError_t e = cudaSuccess;
    for (void* q : {static_cast<void*>(plan->d_segs), static_cast<void*>(plan->d_tiles),
                    static_cast<void*>(plan->d_ag_tiles), static_cast<void*>(plan->d_ptrs)}) {
        if (!q) continue;
        const cudaError_t e2 = cudaFree(q);
        if (e == cudaSuccess) e = e2;
    }
    plan->d_segs = nullptr;
    plan->d_tiles = plan->d_ag_tiles = nullptr;
    plan->d_ptrs = nullptr;
    delete plan;
    return coal_cuda(e);
}

}  // extern "C"
