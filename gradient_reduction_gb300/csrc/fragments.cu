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

constexpr int64_t kFragTile = 4096;

struct FragTile {
    int64_t t0;         // first element of the tile inside its chunk
    int64_t n;          // elements in the tile
    int64_t src_off;    // vec tiles: offset of the tile inside gradient p
    int32_t piece0;     // first piece
    int32_t n_pieces;
    int32_t j;          // chunk
    int32_t vec;        // one aligned piece inside a gradient, n % 16 == 0
    int32_t p;          // vec tiles: the gradient (so its pointers load with the tile)
    int32_t pad;
};

struct FragPiece {
    int64_t tile_off;   // first element of the piece inside its tile
    int64_t len;
    int64_t src_off;    // element offset inside gradient p (unused for a gap)
    int32_t p;          // gradient, or -1 for a gap
    int32_t pad;
};

struct FragParams {
    const FragTile* tiles;
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

template <int KC, int MODE>
__global__ void __launch_bounds__(kThreads) rs_fragments(const __grid_constant__ FragParams p) {
    __shared__ const uint16_t* base[DPR_MAX_RANKS];
    const FragTile tl = p.tiles[blockIdx.x];
    const int K = KC > 0 ? KC : p.K;
    const int j = tl.j;
    float* const out = p.out[j] + tl.t0;
    if (tl.vec && p.out_aligned32) {
        if (threadIdx.x < K) base[threadIdx.x] = p.ptrs[int64_t(threadIdx.x) * p.P + tl.p] + tl.src_off;
        __syncthreads();
        order_enter(p.order);           // the plan's tables above are fixed; the buffers are not
        for (int64_t u = threadIdx.x; u < tl.n / 16; u += kThreads) {
            float acc[16];
            ring_sum<KC, 1, MODE, 8, true>(base, K, j, uint64_t(16 * u), acc);
            store_shard<8>(out + 16 * u, acc, p.scale, p.accumulate);
        }
        order_exit(p.order);
        return;
    }
    order_enter(p.order);
    for (int q = 0; q < tl.n_pieces; ++q) {
        __syncthreads();                       // the previous piece is done with base[]
        const FragPiece pc = p.pieces[tl.piece0 + q];
        if (threadIdx.x < K)
            base[threadIdx.x] = pc.p >= 0 ? p.ptrs[int64_t(threadIdx.x) * p.P + pc.p] + pc.src_off
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
            float v = __fmul_rn(acc, p.scale);
            float* o = out + pc.tile_off + i;
            if (p.accumulate) v = __fadd_rn(*o, v);
            *o = v;
        }
    }
    order_exit(p.order);
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
            tl.t0 = t0;
            tl.n = n;
            tl.j = j;
            tl.piece0 = int32_t(pieces.size());
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
            tl.n_pieces = int32_t(pieces.size()) - tl.piece0;
            const FragPiece& first = pieces[tl.piece0];
            bool vec = tl.n_pieces == 1 && first.p >= 0 && n % 16 == 0;
            for (int r = 0; r < K && vec; ++r)
                vec = aligned(static_cast<const uint16_t*>(src[size_t(r) * P + first.p]) + first.src_off, 32);
            tl.vec = vec ? 1 : 0;
            tl.p = vec ? first.p : -1;
            tl.src_off = vec ? first.src_off : 0;
            tl.pad = 0;
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
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool first = true;
    for (int i = 0; i < n; ++i) {
        if (skip[i]) continue;
        prm[i].order = first ? kAfterPrevious : kBesidePrevious;
        first = false;
        const cudaError_t e = launch_fragments(plans[i], prm[i], kern[i], s);
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
