// Reduce-scatter of a flat gradient bucket straight from its fragments.
//
// ZeRO-2 gathers a bucket's gradients into the IPG buffer at fixed offsets
// and reduce-scatters the buffer (DeepSpeed ZeRO-3 source walkthrough,
// sections 3.2 and 5.1); in DeepSpeed the gradients are written into the
// bucket in the first place, so the gather costs nothing.  Here the per-rank
// gradients already exist as separate buffers.  Gathering them first costs a
// full write and re-read of the bucket, so this path reads each element of a
// chunk from the gradient that covers it and adds the K ranks in ring order
// (CMU 11-868 Lecture 14 notes, section 3.2), exactly as the reduce-scatter
// of the gathered bucket would.  Positions no gradient covers add zeros.
//
// The bucket's chunks are cut into tiles of kFragTile elements that never
// cross a chunk boundary; one block handles one tile.  Each tile is split
// into pieces, runs of elements that lie inside one gradient or inside one gap
// between gradients.  A tile that is one piece inside one gradient, with every
// rank's source 32-byte aligned, takes the 32-byte ring-sum path; any other
// tile is summed element by element, piece by piece.
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

#ifndef DPR_FRAG_TILE
#define DPR_FRAG_TILE 4096
#endif
constexpr int64_t kFragTile = DPR_FRAG_TILE;     // elements per chunk tile, one block each
// Minimum blocks per SM the fragments kernels are compiled for, for K <= 8
// (larger K keeps the compiler's choice, which a cap would make spill).  1
// leaves the register count to the compiler: with the packed tile record and
// its L2 prefetch, a cap of 48 registers (5 blocks per SM) measured slower.
#ifndef DPR_FRAG_MIN_BLOCKS
#define DPR_FRAG_MIN_BLOCKS 1
#endif
constexpr int frag_min_blocks(int KC) { return (KC > 0 && KC <= 8) ? DPR_FRAG_MIN_BLOCKS : 1; }

// 24 bytes, so that the record each block reads before its first data load
// shares a DRAM sector with its neighbours'.
struct FragTile {
    int64_t src_off;    // vec tiles: offset of the tile inside gradient p
    int32_t t0_tiles;   // first element of the tile inside its chunk, / kFragTile
    int32_t first;      // vec tiles: the gradient p; otherwise the first piece
    int32_t n_pieces;
    uint16_t n;         // elements in the tile (<= kFragTile)
    uint8_t j;          // chunk
    uint8_t vec;        // one aligned piece inside a gradient, n % 16 == 0
};
static_assert(sizeof(FragTile) == 24, "packed tile record");
static_assert(kFragTile <= 65535 && DPR_MAX_RANKS <= 255, "tile record field widths");

struct FragPiece {
    int64_t tile_off;   // first element of the piece inside its tile
    int64_t len;
    int64_t src_off;    // element offset inside gradient p (unused for a gap)
    int32_t p;          // gradient, or -1 for a gap
    int32_t pad;
};

struct FragParams {
    const FragTile* tiles;
    int64_t n_tiles;
    const FragPiece* pieces;
    uint16_t* const* ptrs;      // device table [K * P]: src[r * P + p]
    float* out[DPR_MAX_RANKS];
    int64_t S;
    int K;
    int P;
    float scale;
    int accumulate;
    int out_aligned32;
    int order;                  // kAfterPrevious / kBesidePrevious
};

// One tile of one bucket (the body of both kernels below).  `ptrs` is the
// plan's [K * P] gradient table, `outs` the bucket's K fp32 shards, `base`
// K shared-memory slots.  Everything before order_enter reads only the plan's
// fixed tables.
template <int KC, int MODE>
__device__ __forceinline__ void fragments_tile(const FragTile& tl, const FragPiece* pieces,
                                               uint16_t* const* ptrs, int P, float* const* outs,
                                               int K_rt, float scale, int accumulate,
                                               int out_aligned32, int order,
                                               const uint16_t** base) {
    const int K = KC > 0 ? KC : K_rt;
    const int j = tl.j;
    float* const out = outs[j] + int64_t(tl.t0_tiles) * kFragTile;
    if (tl.vec && out_aligned32) {
        if (threadIdx.x < K) base[threadIdx.x] = ptrs[int64_t(threadIdx.x) * P + tl.first] + tl.src_off;
        __syncthreads();
        order_enter(order);             // the plan's tables above are fixed; the buffers are not
        for (int64_t u = threadIdx.x; u < tl.n / 16; u += kThreads) {
            float acc[16];
            ring_sum<KC, 1, MODE, 8, true>(base, K, j, uint64_t(16 * u), acc);
            store_shard<8>(out + 16 * u, acc, scale, accumulate);
        }
        order_exit(order);
        return;
    }
    order_enter(order);
    for (int q = 0; q < tl.n_pieces; ++q) {
        __syncthreads();                       // the previous piece is done with base[]
        const FragPiece pc = pieces[tl.first + q];
        if (threadIdx.x < K)
            base[threadIdx.x] = pc.p >= 0 ? ptrs[int64_t(threadIdx.x) * P + pc.p] + pc.src_off
                                          : nullptr;
        __syncthreads();
        for (int64_t i = threadIdx.x; i < pc.len; i += kThreads) {
            float acc = 0.0f;
            uint16_t hop = 0;
            for (int s = 0; s < K; ++s) {
                int r = j + s;
                r = (r >= K) ? r - K : r;
                const uint16_t x = pc.p >= 0 ? base[r][i] : uint16_t(0);
                if constexpr (MODE == DPR_SUM_RING_FP32) acc = (s == 0) ? bf_1(x) : __fadd_rn(acc, bf_1(x));
                else hop = (s == 0) ? x : add_bf16(hop, x);
            }
            if constexpr (MODE == DPR_SUM_HOP_BF16) acc = bf_1(hop);
            float v = __fmul_rn(acc, scale);
            float* o = out + pc.tile_off + i;
            if (accumulate) v = __fadd_rn(*o, v);
            *o = v;
        }
    }
    order_exit(order);
}

// Blocks ahead whose tile record a block asks L2 to fetch (a little more
// than one wave of resident blocks), so that the record a block reads first
// is an L2 hit rather than a DRAM miss.
#ifndef DPR_FRAG_PREFETCH_AHEAD
#define DPR_FRAG_PREFETCH_AHEAD 1024
#endif

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

template <int KC, int MODE>
__global__ void __launch_bounds__(kThreads, frag_min_blocks(KC)) rs_fragments(const __grid_constant__ FragParams p) {
    __shared__ const uint16_t* base[DPR_MAX_RANKS];
    order_start(p.order);
    if (DPR_FRAG_PREFETCH_AHEAD > 0 && threadIdx.x == 0 &&
        int64_t(blockIdx.x) + DPR_FRAG_PREFETCH_AHEAD < p.n_tiles)
        prefetch_l2(p.tiles + blockIdx.x + DPR_FRAG_PREFETCH_AHEAD);
    const FragTile tl = p.tiles[blockIdx.x];
    fragments_tile<KC, MODE>(tl, p.pieces, p.ptrs, p.P, p.out, p.K, p.scale, p.accumulate,
                             p.out_aligned32, p.order, base);
}

// Several buckets in one grid: the blocks of member m are
// [tile0[m], tile0[m + 1]); each block finds its member by binary search over
// tile0 (uniform across the block, in the parameter block) and runs the
// member's tile.  Members share K, mode, scale and accumulate.
constexpr int kMultiMembers = 128;     // members per launch
constexpr int kMultiOuts = 2048;       // shard pointers per launch

struct FragMember {
    const FragTile* tiles;
    const FragPiece* pieces;
    uint16_t* const* ptrs;
    int32_t P;
    int32_t out0;           // the member's first shard pointer in out[]
    int32_t out_aligned32;
    int32_t pad;
};

struct FragMultiParams {
    int64_t tile0[kMultiMembers + 1];
    FragMember m[kMultiMembers];
    float* out[kMultiOuts];
    int n;
    int K;
    float scale;
    int accumulate;
    int order;
};

template <int KC, int MODE>
__global__ void __launch_bounds__(kThreads, frag_min_blocks(KC)) rs_fragments_multi(const __grid_constant__ FragMultiParams p) {
    __shared__ const uint16_t* base[DPR_MAX_RANKS];
    order_start(p.order);
    const int64_t b = blockIdx.x;
    int lo = 0, hi = p.n - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (p.tile0[mid] <= b) lo = mid;
        else hi = mid - 1;
    }
    const FragMember& mb = p.m[lo];
    if (DPR_FRAG_PREFETCH_AHEAD > 0 && threadIdx.x == 0 &&
        b + DPR_FRAG_PREFETCH_AHEAD < p.tile0[lo + 1])
        prefetch_l2(mb.tiles + (b - p.tile0[lo]) + DPR_FRAG_PREFETCH_AHEAD);
    const FragTile tl = mb.tiles[b - p.tile0[lo]];
    fragments_tile<KC, MODE>(tl, mb.pieces, mb.ptrs, mb.P, p.out + mb.out0, p.K, p.scale,
                             p.accumulate, mb.out_aligned32, p.order, base);
}

template <int MODE>
const void* rs_fragments_multi_for(int K) {
    switch (K) {
        case 2: return reinterpret_cast<const void*>(rs_fragments_multi<2, MODE>);
        case 4: return reinterpret_cast<const void*>(rs_fragments_multi<4, MODE>);
        case 8: return reinterpret_cast<const void*>(rs_fragments_multi<8, MODE>);
        case 16: return reinterpret_cast<const void*>(rs_fragments_multi<16, MODE>);
        case 32: return reinterpret_cast<const void*>(rs_fragments_multi<32, MODE>);
        case 64: return reinterpret_cast<const void*>(rs_fragments_multi<64, MODE>);
        default: return reinterpret_cast<const void*>(rs_fragments_multi<0, MODE>);
    }
}

template <int MODE>
const void* rs_fragments_for(int K) {
    switch (K) {
        case 2: return reinterpret_cast<const void*>(rs_fragments<2, MODE>);
        case 4: return reinterpret_cast<const void*>(rs_fragments<4, MODE>);
        case 8: return reinterpret_cast<const void*>(rs_fragments<8, MODE>);
        case 16: return reinterpret_cast<const void*>(rs_fragments<16, MODE>);
        case 32: return reinterpret_cast<const void*>(rs_fragments<32, MODE>);
        case 64: return reinterpret_cast<const void*>(rs_fragments<64, MODE>);
        default: return reinterpret_cast<const void*>(rs_fragments<0, MODE>);
    }
}

}  // namespace
}  // namespace dpr

using namespace dpr;

struct dpr_fragments_plan {
    int K = 0;
    int P = 0;
    int device = 0;
    int64_t bucket_numel = 0;
    std::vector<Span> src_spans;
    std::vector<FragTile> tiles;
    FragTile* d_tiles = nullptr;
    FragPiece* d_pieces = nullptr;
    uint16_t** d_ptrs = nullptr;
};

namespace {

void free_fragments_plan(dpr_fragments_plan* pl) {
    if (pl->d_tiles) cudaFree(pl->d_tiles);
    if (pl->d_pieces) cudaFree(pl->d_pieces);
    if (pl->d_ptrs) cudaFree(pl->d_ptrs);
    delete pl;
}

}  // namespace

extern "C" {

dpr_status dpr_fragments_plan_create(dpr_fragments_plan** plan, int K, int P, const void* const* src,
                                     const int64_t* numel, const int64_t* offset,
                                     int64_t bucket_numel, void* stream) {
    if (!plan) return DPR_ERR_INVALID_ARG;
    *plan = nullptr;
    if (K < 2 || K > DPR_MAX_RANKS || P < 0 || bucket_numel < 0) return DPR_ERR_INVALID_ARG;
    if (bucket_numel > DPR_MAX_ELEMS) return DPR_ERR_UNSUPPORTED;
    if (bucket_numel % K != 0) return DPR_ERR_INVALID_ARG;
    if (P > 0 && (!src || !numel || !offset)) return DPR_ERR_INVALID_ARG;
    // gradients in bucket order; every span inside the bucket, none overlapping
    std::vector<int> order;
    for (int p = 0; p < P; ++p) {
        if (numel[p] < 0 || offset[p] < 0) return DPR_ERR_INVALID_ARG;
        if (numel[p] == 0) continue;
        if (offset[p] > bucket_numel - numel[p]) return DPR_ERR_INVALID_ARG;
        order.push_back(p);
    }
    std::sort(order.begin(), order.end(), [&](int a, int b) { return offset[a] < offset[b]; });
    for (size_t i = 1; i < order.size(); ++i)
        if (offset[order[i]] < offset[order[i - 1]] + numel[order[i - 1]]) return DPR_ERR_ALIAS;
    std::vector<Span> spans;
    for (int p : order)
        for (int r = 0; r < K; ++r) {
            const void* t = src[size_t(r) * P + p];
            if (!t) return DPR_ERR_INVALID_ARG;
            if (!aligned(t, 2)) return DPR_ERR_ALIGNMENT;
            const uintptr_t a = reinterpret_cast<uintptr_t>(t);
            spans.push_back(Span{a, a + uintptr_t(numel[p]) * 2});
        }
    const int64_t S = bucket_numel / K;
    const int64_t tiles_per_chunk = (S + kFragTile - 1) / kFragTile;
    if (int64_t(K) * tiles_per_chunk > int64_t(0x7FFFFFFF)) return DPR_ERR_UNSUPPORTED;

    dpr_fragments_plan* pl = new (std::nothrow) dpr_fragments_plan();
    if (!pl) return DPR_ERR_CUDA;
    pl->K = K;
    pl->P = P;
    pl->bucket_numel = bucket_numel;
    pl->src_spans = spans;
    std::vector<FragPiece> pieces;
    size_t g = 0;      // first gradient (in bucket order) that may overlap the current tile
    for (int j = 0; j < K && S > 0; ++j) {
        for (int64_t t0 = 0; t0 < S; t0 += kFragTile) {
            const int64_t a = int64_t(j) * S + t0;
            const int64_t n = std::min(kFragTile, S - t0);
            FragTile tl;
            tl.t0_tiles = int32_t(t0 / kFragTile);
            tl.n = uint16_t(n);
            tl.j = uint8_t(j);
            const int64_t piece0 = int64_t(pieces.size());
            while (g < order.size() && offset[order[g]] + numel[order[g]] <= a) ++g;
            int64_t at = a;
            for (size_t h = g; at < a + n; ++h) {
                const bool have = h < order.size() && offset[order[h]] < a + n;
                const int64_t next = have ? std::max(offset[order[h]], at) : a + n;
                if (next > at)       // a gap before the next gradient
                    pieces.push_back(FragPiece{at - a, next - at, 0, -1, 0});
                at = next;
                if (!have) break;
                const int p = order[h];
                const int64_t end = std::min(offset[p] + numel[p], a + n);
                pieces.push_back(FragPiece{at - a, end - at, at - offset[p], p, 0});
                at = end;
            }
            if (int64_t(pieces.size()) > int64_t(0x7FFFFFFF)) {
                free_fragments_plan(pl);
                return DPR_ERR_UNSUPPORTED;
            }
            tl.n_pieces = int32_t(int64_t(pieces.size()) - piece0);
            const FragPiece& first = pieces[size_t(piece0)];
            bool vec = tl.n_pieces == 1 && first.p >= 0 && n % 16 == 0;
            for (int r = 0; r < K && vec; ++r)
                vec = aligned(static_cast<const uint16_t*>(src[size_t(r) * P + first.p]) + first.src_off, 32);
            tl.vec = vec ? 1 : 0;
            tl.first = vec ? first.p : int32_t(piece0);
            tl.src_off = vec ? first.src_off : 0;
            pl->tiles.push_back(tl);
        }
    }
    if (pieces.size() > size_t(0x7FFFFFFF)) {
        free_fragments_plan(pl);
        return DPR_ERR_UNSUPPORTED;
    }
    cudaError_t e = cudaGetDevice(&pl->device);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (e == cudaSuccess && !pl->tiles.empty()) {
        std::vector<uint16_t*> ptrs(size_t(K) * P);
        for (size_t i = 0; i < ptrs.size(); ++i)
            ptrs[i] = static_cast<uint16_t*>(const_cast<void*>(src[i]));
        e = upload(&pl->d_tiles, pl->tiles, st);
        if (e == cudaSuccess) e = upload(&pl->d_pieces, pieces, st);
        if (e == cudaSuccess && !ptrs.empty()) e = upload(&pl->d_ptrs, ptrs, st);
        if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    }
    if (e != cudaSuccess) {
        free_fragments_plan(pl);
        return record_cuda_status(e);
    }
    *plan = pl;
    return DPR_OK;
}

}  // extern "C"

namespace {

// The checks of dpr_reduce_scatter_fragments; on success fills the parameter
// block and the kernel and appends the output spans to `outs` (nothing is
// launched).  *empty is set when the plan has no tiles.
dpr_status prepare_fragments(const dpr_fragments_plan* plan, float* const* out, int mode,
                             float scale, int accumulate, FragParams* prm, const void** kernel,
                             std::vector<Span>* outs, bool* empty) {
    if (!plan || !out) return DPR_ERR_INVALID_ARG;
    if (mode != DPR_SUM_RING_FP32 && mode != DPR_SUM_HOP_BF16) return DPR_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_status(e);
    if (dev != plan->device) return DPR_ERR_INVALID_ARG;
    const int K = plan->K;
    const int64_t S = plan->bucket_numel / K;
    bool a32 = true;
    std::vector<Span> mine;
    for (int j = 0; j < K; ++j) {
        if (!out[j]) return DPR_ERR_INVALID_ARG;
        if (!aligned(out[j], 4)) return DPR_ERR_ALIGNMENT;
        a32 = a32 && aligned(out[j], 32);
        mine.push_back(span_of(out[j], uint64_t(S) * 4));
    }
    if (!pairwise_disjoint(mine)) return DPR_ERR_ALIAS;
    for (const Span& t : plan->src_spans)
        for (const Span& o : mine)
            if (overlaps(t, o)) return DPR_ERR_ALIAS;
    *empty = plan->tiles.empty();
    std::memset(prm, 0, sizeof(*prm));
    prm->tiles = plan->d_tiles;
    prm->n_tiles = int64_t(plan->tiles.size());
    prm->pieces = plan->d_pieces;
    prm->ptrs = plan->d_ptrs;
    for (int j = 0; j < K; ++j) prm->out[j] = out[j];
    prm->S = S;
    prm->K = K;
    prm->P = plan->P;
    prm->scale = scale;
    prm->accumulate = accumulate ? 1 : 0;
    prm->out_aligned32 = a32 ? 1 : 0;
    prm->order = kAfterPrevious;
    *kernel = (mode == DPR_SUM_RING_FP32) ? rs_fragments_for<DPR_SUM_RING_FP32>(K)
                                          : rs_fragments_for<DPR_SUM_HOP_BF16>(K);
    outs->insert(outs->end(), mine.begin(), mine.end());
    return DPR_OK;
}

cudaError_t launch_fragments(const dpr_fragments_plan* plan, FragParams& prm, const void* kernel,
                             cudaStream_t stream) {
    void* args[] = {&prm};
    return launch_kernel(kernel, dim3(unsigned(plan->tiles.size())), args, stream);
}

}  // namespace

extern "C" {

dpr_status dpr_reduce_scatter_fragments(const dpr_fragments_plan* plan, float* const* out, int mode,
                                        float scale, int accumulate, void* stream) {
    FragParams prm;
    const void* k = nullptr;
    std::vector<Span> outs;
    bool empty = false;
    dpr_status st = prepare_fragments(plan, out, mode, scale, accumulate, &prm, &k, &outs, &empty);
    if (st != DPR_OK || empty) return st;
    return record_cuda_status(launch_fragments(plan, prm, k, static_cast<cudaStream_t>(stream)));
}

dpr_status dpr_reduce_scatter_fragments_batch(int n, const dpr_fragments_plan* const* plans,
                                              float* const* out, int mode, float scale,
                                              int accumulate, void* stream) {
    if (n < 0 || n > DPR_MAX_BATCH) return n < 0 ? DPR_ERR_INVALID_ARG : DPR_ERR_UNSUPPORTED;
    if (n == 0) return DPR_OK;
    if (!plans || !out) return DPR_ERR_INVALID_ARG;
    std::vector<FragParams> prm(static_cast<size_t>(n));
    std::vector<const void*> kern(static_cast<size_t>(n), nullptr);
    std::vector<char> skip(static_cast<size_t>(n), 0);
    std::vector<Span> outs, srcs;
    size_t o = 0;
    for (int i = 0; i < n; ++i) {
        if (!plans[i]) return DPR_ERR_INVALID_ARG;
        bool empty = false;
        dpr_status st = prepare_fragments(plans[i], out + o, mode, scale, accumulate, &prm[i],
                                          &kern[i], &outs, &empty);
        if (st != DPR_OK) return st;
        skip[i] = empty ? 1 : 0;
        o += size_t(plans[i]->K);
        srcs.insert(srcs.end(), plans[i]->src_spans.begin(), plans[i]->src_spans.end());
    }
    // members are independent: no output touches another output or any source
    if (!pairwise_disjoint(outs) || any_overlap(outs, srcs)) return DPR_ERR_ALIAS;
    // members with tiles, grouped into launches of one grid each: consecutive
    // members with the same K, up to kMultiMembers members, kMultiOuts shard
    // pointers and a 1-D grid's blocks per launch
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    std::vector<FragMultiParams> launches;
    size_t o_at = 0;
    for (int i = 0; i < n; ++i) {
        const dpr_fragments_plan* pl = plans[i];
        const size_t o_i = o_at;
        o_at += size_t(pl->K);
        if (skip[i]) continue;
        const int64_t t = int64_t(pl->tiles.size());
        FragMultiParams* cur = launches.empty() ? nullptr : &launches.back();
        if (!cur || cur->K != pl->K || cur->n == kMultiMembers ||
            cur->m[cur->n - 1].out0 + 2 * pl->K > kMultiOuts ||
            cur->tile0[cur->n] + t > int64_t(0x7FFFFFFF)) {
            launches.emplace_back();
            cur = &launches.back();
            std::memset(cur, 0, sizeof(*cur));
            cur->K = pl->K;
            cur->scale = scale;
            cur->accumulate = accumulate ? 1 : 0;
        }
        FragMember& mb = cur->m[cur->n];
        mb.tiles = pl->d_tiles;
        mb.pieces = pl->d_pieces;
        mb.ptrs = pl->d_ptrs;
        mb.P = pl->P;
        mb.out0 = cur->n == 0 ? 0 : cur->m[cur->n - 1].out0 + cur->K;
        mb.out_aligned32 = prm[i].out_aligned32;
        for (int j = 0; j < pl->K; ++j) cur->out[mb.out0 + j] = out[o_i + j];
        cur->tile0[cur->n + 1] = cur->tile0[cur->n] + t;
        ++cur->n;
    }
    for (size_t l = 0; l < launches.size(); ++l) {
        FragMultiParams& lp = launches[l];
        lp.order = l == 0 ? kAfterPrevious : kBesidePrevious;
        const void* k = (mode == DPR_SUM_RING_FP32) ? rs_fragments_multi_for<DPR_SUM_RING_FP32>(lp.K)
                                                    : rs_fragments_multi_for<DPR_SUM_HOP_BF16>(lp.K);
        void* args[] = {&lp};
        const cudaError_t e = launch_kernel(k, dim3(unsigned(lp.tile0[lp.n])), args, s);
        if (e != cudaSuccess) return record_cuda_status(e);
    }
    return DPR_OK;
}

dpr_status dpr_fragments_plan_destroy(dpr_fragments_plan* plan) {
    if (!plan) return DPR_OK;
    cudaError_t e = cudaSuccess;
    for (void* q : {static_cast<void*>(plan->d_tiles), static_cast<void*>(plan->d_pieces),
                    static_cast<void*>(plan->d_ptrs)}) {
        if (!q) continue;
        const cudaError_t e2 = cudaFree(q);
        if (e == cudaSuccess) e = e2;
    }
    delete plan;
    return record_cuda_status(e);
}

}  // extern "C"
