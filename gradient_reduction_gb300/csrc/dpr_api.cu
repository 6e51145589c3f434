// Host side of libdpr: argument validation, layout selection and launches.
// Every check runs before anything is enqueued; a rejected call has no effect.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <new>
#include <utility>
#include <vector>

#include "dpr_kernels.h"
#include "host_checks.h"

namespace dpr {
namespace {

thread_local int g_last_cuda_error = 0;
std::atomic<int> g_programmatic{1};

dpr_status cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return DPR_OK;
    g_last_cuda_error = int(e);
    return DPR_ERR_CUDA;
}

}  // namespace

dpr_status record_cuda_status(cudaError_t e) { return cuda_status(e); }

bool programmatic_launch_enabled() { return g_programmatic.load(std::memory_order_relaxed) != 0; }

cudaError_t launch_kernel(const void* kernel, dim3 grid, void** args, cudaStream_t s,
                          bool programmatic) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    // the legacy default stream (and its aliases) keeps plain launches
    const bool legacy = s == nullptr || s == cudaStreamLegacy || s == cudaStreamPerThread;
    cfg.attrs = attr;
    cfg.numAttrs = (programmatic && !legacy && programmatic_launch_enabled()) ? 1 : 0;
    return cudaLaunchKernelExC(&cfg, kernel, args);
}

namespace {

// K, N shared checks.  Returns DPR_OK to proceed.
dpr_status check_kn(int K, int64_t N) {
    if (K < 2 || K > DPR_MAX_RANKS) return DPR_ERR_INVALID_ARG;
    if (N < 0) return DPR_ERR_INVALID_ARG;
    if (N > DPR_MAX_ELEMS) return DPR_ERR_UNSUPPORTED;
    if (N % K != 0) return DPR_ERR_INVALID_ARG;
    return DPR_OK;
}

int sm_count(int dev) {
    static std::mutex mu;
    static std::map<int, int> cache;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it != cache.end()) return it->second;
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        return 0;
    cache[dev] = v;
    return v;
}

}  // namespace

cudaError_t blocks_per_chunk(const void* kernel, int K, uint64_t work_per_chunk, int* gx) {
    static std::mutex mu;
    static std::map<std::pair<const void*, int>, int> occ_cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int sms = sm_count(dev);
    if (sms <= 0) return cudaErrorInvalidDevice;
    int occ = 0;
    {
        std::lock_guard<std::mutex> lock(mu);
        auto it = occ_cache.find({kernel, dev});
        if (it != occ_cache.end()) {
            occ = it->second;
        } else {
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kernel, kThreads, 0);
            if (e != cudaSuccess) return e;
            occ_cache[{kernel, dev}] = occ;
        }
    }
    if (occ < 1) occ = 1;
    // One wave of resident blocks split evenly over the K chunks (rounded
    // down, so no block waits for a second wave), but never more blocks
    // than there are 256-unit slices of work.
    int64_t per_chunk = int64_t(sms) * occ / K;
    if (per_chunk < 1) per_chunk = 1;
    const int64_t need = int64_t((work_per_chunk + kThreads - 1) / kThreads);
    *gx = int(std::max<int64_t>(1, std::min(per_chunk, need)));
    return cudaSuccess;
}

}  // namespace dpr

using namespace dpr;


dpr_status dpr::prepare_reduce_scatter(const void* const* in, int K, int M, int64_t N,
                                       float* const* out, int mode, float scale, int accumulate,
                                       RsParams* p, int* width_out) {
    dpr_status st = check_kn(K, N);
    if (st != DPR_OK) return st;
    if (M < 1 || M > DPR_MAX_MICRO) return DPR_ERR_INVALID_ARG;
    if (mode != DPR_SUM_RING_FP32 && mode != DPR_SUM_HOP_BF16) return DPR_ERR_INVALID_ARG;
    if (N == 0) return DPR_OK;
    if (!in || !out) return DPR_ERR_INVALID_ARG;
    const int64_t S = N / K;
    bool a16 = true, a32 = true;
    std::vector<Span> outs;
    for (int i = 0; i < M * K; ++i) {
        if (!in[i]) return DPR_ERR_INVALID_ARG;
        if (!aligned(in[i], 2)) return DPR_ERR_ALIGNMENT;
        a16 = a16 && aligned(in[i], 16);
        a32 = a32 && aligned(in[i], 32);
    }
    for (int j = 0; j < K; ++j) {
        if (!out[j]) return DPR_ERR_INVALID_ARG;
        if (!aligned(out[j], 4)) return DPR_ERR_ALIGNMENT;
        a16 = a16 && aligned(out[j], 16);
        a32 = a32 && aligned(out[j], 32);
        outs.push_back(span_of(out[j], uint64_t(S) * 4));
    }
    const bool edge = edge_unit(S, K, a32, false);
    const int width = edge ? 8 : access_width(S, a32, a16);
    if (!pairwise_disjoint(outs)) return DPR_ERR_ALIAS;
    for (int i = 0; i < M * K; ++i) {
        const Span a = span_of(in[i], uint64_t(N) * 2);
        for (const Span& o : outs)
            if (overlaps(a, o)) return DPR_ERR_ALIAS;
    }
    std::memset(p, 0, sizeof(*p));
    for (int i = 0; i < M * K; ++i) p->in[i] = static_cast<const uint16_t*>(in[i]);
    for (int j = 0; j < K; ++j) p->out[j] = out[j];
    p->S = S;
    p->su = chunk_units(S, width, edge);
    p->edge = edge ? 1 : 0;
    p->K = K;
    p->M = M;
    p->scale = scale;
    p->accumulate = accumulate ? 1 : 0;
    p->order = kAfterPrevious;
    *width_out = width;
    return DPR_OK;
}

extern "C" {

dpr_status dpr_reduce_scatter(const void* const* in, int K, int M, int64_t N, float* const* out,
                              int mode, float scale, int accumulate, void* stream) {
    return dpr::reduce_scatter_capped(in, K, M, N, out, mode, scale, accumulate,
                                      static_cast<cudaStream_t>(stream), 0);
}

dpr_status dpr_reduce_scatter_batch(int n, const void* const* in, int K, int M, const int64_t* N,
                                    float* const* out, int mode, float scale, int accumulate,
                                    void* stream) {
    if (n < 0) return DPR_ERR_INVALID_ARG;
    if (n > DPR_MAX_BATCH) return DPR_ERR_UNSUPPORTED;
    if (n == 0) return DPR_OK;
    if (!in || !N || !out) return DPR_ERR_INVALID_ARG;
    if (K < 2 || K > DPR_MAX_RANKS || M < 1 || M > DPR_MAX_MICRO) return DPR_ERR_INVALID_ARG;
    std::vector<RsParams> prm(static_cast<size_t>(n));
    std::vector<int> width(static_cast<size_t>(n), 0);
    std::vector<Span> outs, ins;
    for (int i = 0; i < n; ++i) {
        const void* const* in_i = in + size_t(i) * M * K;
        float* const* out_i = out + size_t(i) * K;
        dpr_status st = prepare_reduce_scatter(in_i, K, M, N[i], out_i, mode, scale, accumulate,
                                               &prm[i], &width[i]);
        if (st != DPR_OK) return st;
        if (N[i] == 0) continue;
        for (int j = 0; j < K; ++j) outs.push_back(span_of(out_i[j], uint64_t(N[i] / K) * 4));
        for (int q = 0; q < M * K; ++q) ins.push_back(span_of(in_i[q], uint64_t(N[i]) * 2));
    }
    // members are independent: no output touches another output or any input
    if (!pairwise_disjoint(outs) || any_overlap(outs, ins)) return DPR_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool first = true;
    for (int i = 0; i < n; ++i) {
        if (N[i] == 0) continue;
        prm[i].order = first ? kAfterPrevious : kBesidePrevious;
        first = false;
        const cudaError_t e = launch_reduce_scatter(prm[i], mode, width[i], s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return DPR_OK;
}

dpr_status dpr_set_programmatic_launch(int enable, int* previous) {
    const int old = g_programmatic.exchange(enable ? 1 : 0);
    if (previous) *previous = old;
    return DPR_OK;
}

}  // extern "C"

dpr_status dpr::reduce_scatter_capped(const void* const* in, int K, int M, int64_t N,
                                      float* const* out, int mode, float scale, int accumulate,
                                      cudaStream_t stream, int max_blocks, bool programmatic) {
    RsParams p;
    int width = 0;
    dpr_status st = prepare_reduce_scatter(in, K, M, N, out, mode, scale, accumulate, &p, &width);
    if (st != DPR_OK || N == 0) return st;
    return cuda_status(launch_reduce_scatter(p, mode, width, stream, max_blocks, programmatic));
}

extern "C" {

dpr_status dpr_reduce_scatter_bf16(const void* const* in, int K, int M, int64_t N,
                                   void* const* out, int mode, float scale, int accumulate,
                                   void* stream) {
    dpr_status st = check_kn(K, N);
    if (st != DPR_OK) return st;
    if (M < 1 || M > DPR_MAX_MICRO) return DPR_ERR_INVALID_ARG;
    if (mode != DPR_SUM_RING_FP32 && mode != DPR_SUM_HOP_BF16) return DPR_ERR_INVALID_ARG;
    if (N == 0) return DPR_OK;
    if (!in || !out) return DPR_ERR_INVALID_ARG;
    const int64_t S = N / K;
    bool a16 = true, a32 = true;
    std::vector<Span> outs;
    for (int i = 0; i < M * K; ++i) {
        if (!in[i]) return DPR_ERR_INVALID_ARG;
        if (!aligned(in[i], 2)) return DPR_ERR_ALIGNMENT;
        a16 = a16 && aligned(in[i], 16);
        a32 = a32 && aligned(in[i], 32);
    }
    for (int j = 0; j < K; ++j) {
        if (!out[j]) return DPR_ERR_INVALID_ARG;
        if (!aligned(out[j], 2)) return DPR_ERR_ALIGNMENT;
        a16 = a16 && aligned(out[j], 16);
        a32 = a32 && aligned(out[j], 32);
        outs.push_back(span_of(out[j], uint64_t(S) * 2));
    }
    if (!pairwise_disjoint(outs)) return DPR_ERR_ALIAS;
    for (int i = 0; i < M * K; ++i) {
        const Span a = span_of(in[i], uint64_t(N) * 2);
        for (const Span& o : outs)
            if (overlaps(a, o)) return DPR_ERR_ALIAS;
    }
    const int width = access_width(S, a32, a16);
    RsParams p;
    std::memset(&p, 0, sizeof(p));
    for (int i = 0; i < M * K; ++i) p.in[i] = static_cast<const uint16_t*>(in[i]);
    for (int j = 0; j < K; ++j) p.out[j] = static_cast<float*>(out[j]);
    p.S = S;
    p.su = width > 0 ? uint32_t(S / (2 * width)) : 0;
    p.K = K;
    p.M = M;
    p.scale = scale;
    p.accumulate = accumulate ? 1 : 0;
    return cuda_status(launch_reduce_scatter_bf16(p, mode, width, static_cast<cudaStream_t>(stream)));
}

dpr_status dpr_cast_bf16_to_fp32(const void* in, float* out, int64_t n, void* stream) {
    if (n < 0) return DPR_ERR_INVALID_ARG;
    if (n > DPR_MAX_ELEMS * DPR_MAX_RANKS) return DPR_ERR_UNSUPPORTED;
    if (n == 0) return DPR_OK;
    if (!in || !out) return DPR_ERR_INVALID_ARG;
    if (!aligned(in, 2) || !aligned(out, 4)) return DPR_ERR_ALIGNMENT;
    if (overlaps(span_of(in, uint64_t(n) * 2), span_of(out, uint64_t(n) * 4))) return DPR_ERR_ALIAS;
    const bool vec = aligned(in, 32) && aligned(out, 32);
    return cuda_status(launch_cast(static_cast<const uint16_t*>(in), out, uint64_t(n), vec,
                                   static_cast<cudaStream_t>(stream)));
}

}  // extern "C"

dpr_status dpr::prepare_allreduce(const void* const* in, int K, int64_t N, void* const* out,
                                  int mode, float scale, ArParams* p, int* width_out) {
    dpr_status st = check_kn(K, N);
    if (st != DPR_OK) return st;
    if (mode != DPR_SUM_RING_FP32 && mode != DPR_SUM_HOP_BF16) return DPR_ERR_INVALID_ARG;
    if (N == 0) return DPR_OK;
    if (!in || !out) return DPR_ERR_INVALID_ARG;
    const int64_t S = N / K;
    bool a16 = true, a32 = true;
    std::vector<Span> outs;
    for (int r = 0; r < K; ++r) {
        if (!in[r] || !out[r]) return DPR_ERR_INVALID_ARG;
        if (!aligned(in[r], 2) || !aligned(out[r], 2)) return DPR_ERR_ALIGNMENT;
        a16 = a16 && aligned(in[r], 16) && aligned(out[r], 16);
        a32 = a32 && aligned(in[r], 32) && aligned(out[r], 32);
        outs.push_back(span_of(out[r], uint64_t(N) * 2));
    }
    bool in_place = false;
    if (!pairwise_disjoint(outs)) return DPR_ERR_ALIAS;
    for (int i = 0; i < K; ++i) {
        const Span a = span_of(in[i], uint64_t(N) * 2);
        for (int r = 0; r < K; ++r) {
            if (i == r && in[i] == out[r]) {           // in place
                in_place = true;
                continue;
            }
            if (overlaps(a, outs[r])) return DPR_ERR_ALIAS;
        }
    }
    // the edge unit reads 8 elements of a neighbouring chunk: never over outputs
    const bool edge = !in_place && edge_unit(S, K, a32, true);
    const int width = edge ? 8 : access_width(S, a32, a16);
    std::memset(p, 0, sizeof(*p));
    for (int r = 0; r < K; ++r) {
        p->in[r] = static_cast<const uint16_t*>(in[r]);
        p->out[r] = static_cast<uint16_t*>(out[r]);
    }
    p->S = S;
    p->su = chunk_units(S, width, edge);
    p->edge = edge ? 1 : 0;
    p->K = K;
    p->scale = scale;
    p->order = kAfterPrevious;
    *width_out = width;
    return DPR_OK;
}

// The checks of dpr_allgather, filling the parameter block and the access
// width on success (nothing is launched).
dpr_status dpr::prepare_allgather(const void* const* shard, int K, int64_t N, void* const* out,
                                  AgParams* p, int* width) {
    dpr_status st = check_kn(K, N);
    if (st != DPR_OK) return st;
    if (N == 0) return DPR_OK;
    if (!shard || !out) return DPR_ERR_INVALID_ARG;
    const int64_t S = N / K;
    bool a16 = true, a32 = true;
    std::vector<Span> outs;
    for (int r = 0; r < K; ++r) {
        if (!shard[r] || !out[r]) return DPR_ERR_INVALID_ARG;
        if (!aligned(shard[r], 2) || !aligned(out[r], 2)) return DPR_ERR_ALIGNMENT;
        a16 = a16 && aligned(shard[r], 16) && aligned(out[r], 16);
        a32 = a32 && aligned(shard[r], 32) && aligned(out[r], 32);
        outs.push_back(span_of(out[r], uint64_t(N) * 2));
    }
    if (!pairwise_disjoint(outs)) return DPR_ERR_ALIAS;
    uint64_t in_place_mask = 0;
    for (int j = 0; j < K; ++j) {
        const bool in_place = shard[j] == static_cast<const void*>(
                                             static_cast<const uint16_t*>(out[j]) + j * S);
        if (in_place) in_place_mask |= uint64_t(1) << j;
        const Span a = span_of(shard[j], uint64_t(S) * 2);
        for (int r = 0; r < K; ++r) {
            if (in_place && r == j) continue;
            if (overlaps(a, outs[r])) return DPR_ERR_ALIAS;
        }
    }
    std::memset(p, 0, sizeof(*p));
    for (int r = 0; r < K; ++r) {
        p->shard[r] = static_cast<const uint16_t*>(shard[r]);
        p->out[r] = static_cast<uint16_t*>(out[r]);
    }
    p->S = S;
    p->tiles_per_chunk = uint64_t((S + kAgTile - 1) / kAgTile);
    p->in_place = in_place_mask;
    p->K = K;
    p->order = kAfterPrevious;
    *width = access_width(S, a32, a16);
    return DPR_OK;
}

extern "C" {

dpr_status dpr_allgather(const void* const* shard, int K, int64_t N, void* const* out,
                         void* stream) {
    AgParams p;
    int width = 0;
    dpr_status st = prepare_allgather(shard, K, N, out, &p, &width);
    if (st != DPR_OK || N == 0) return st;
    return cuda_status(launch_allgather(p, width, static_cast<cudaStream_t>(stream)));
}

dpr_status dpr_allgather_batch(int n, const void* const* shard, int K, const int64_t* N,
                               void* const* out, void* stream) {
    if (n < 0) return DPR_ERR_INVALID_ARG;
    if (n > DPR_MAX_BATCH) return DPR_ERR_UNSUPPORTED;
    if (n == 0) return DPR_OK;
    if (!shard || !N || !out) return DPR_ERR_INVALID_ARG;
    if (K < 2 || K > DPR_MAX_RANKS) return DPR_ERR_INVALID_ARG;
    std::vector<AgParams> prm(static_cast<size_t>(n));
    std::vector<int> width(static_cast<size_t>(n), 0);
    std::vector<OwnedSpan> outs;
    std::vector<OwnedSpan> shards;
    for (int i = 0; i < n; ++i) {
        const void* const* sh_i = shard + size_t(i) * K;
        void* const* out_i = out + size_t(i) * K;
        dpr_status st = prepare_allgather(sh_i, K, N[i], out_i, &prm[i], &width[i]);
        if (st != DPR_OK) return st;
        if (N[i] == 0) continue;
        for (int r = 0; r < K; ++r) {
            outs.push_back({span_of(out_i[r], uint64_t(N[i]) * 2), i});
            shards.push_back({span_of(sh_i[r], uint64_t(N[i] / K) * 2), i});
        }
    }
    // members are independent: no output touches another member's output or
    // shard (a member's own in-place shard is checked above)
    std::sort(outs.begin(), outs.end(),
              [](const OwnedSpan& a, const OwnedSpan& b) { return a.s.lo < b.s.lo; });
    for (size_t q = 1; q < outs.size(); ++q)
        if (outs[q].s.lo < outs[q - 1].s.hi) return DPR_ERR_ALIAS;
    for (const OwnedSpan& x : shards)
        if (overlaps_other(outs, x.s, x.owner)) return DPR_ERR_ALIAS;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    bool first = true;
    for (int i = 0; i < n; ++i) {
        if (N[i] == 0) continue;
        prm[i].order = first ? kAfterPrevious : kBesidePrevious;
        first = false;
        const cudaError_t e = launch_allgather(prm[i], width[i], s);
        if (e != cudaSuccess) return cuda_status(e);
    }
    return DPR_OK;
}

dpr_status dpr_allreduce(const void* const* in, int K, int64_t N, void* const* out, int mode,
                         float scale, void* stream) {
    ArParams p;
    int width = 0;
    dpr_status st = prepare_allreduce(in, K, N, out, mode, scale, &p, &width);
    if (st != DPR_OK || N == 0) return st;
    return cuda_status(launch_allreduce(p, mode, width, static_cast<cudaStream_t>(stream)));
}

dpr_status dpr_flatten_plan_create(dpr_flatten_plan** plan, int K, int P, const void* const* src,
                                   const int64_t* numel, const int64_t* offset,
                                   int64_t bucket_numel, void* stream) {
    if (!plan) return DPR_ERR_INVALID_ARG;
    *plan = nullptr;
    if (K < 1 || K > DPR_MAX_RANKS || P < 0) return DPR_ERR_INVALID_ARG;
    if (bucket_numel < 0) return DPR_ERR_INVALID_ARG;
    if (bucket_numel > DPR_MAX_ELEMS) return DPR_ERR_UNSUPPORTED;
    if (P > 0 && (!src || !numel || !offset)) return DPR_ERR_INVALID_ARG;
    std::vector<std::pair<int64_t, int64_t>> spans;
    for (int p = 0; p < P; ++p) {
        if (numel[p] < 0 || offset[p] < 0) return DPR_ERR_INVALID_ARG;
        if (numel[p] == 0) continue;
        if (offset[p] > bucket_numel - numel[p]) return DPR_ERR_INVALID_ARG;
        spans.push_back({offset[p], offset[p] + numel[p]});
    }
    std::sort(spans.begin(), spans.end());
    for (size_t i = 1; i < spans.size(); ++i)
        if (spans[i].first < spans[i - 1].second) return DPR_ERR_ALIAS;
    dpr_flatten_plan* pl = new (std::nothrow) dpr_flatten_plan();
    if (!pl) return DPR_ERR_CUDA;
    pl->K = K;
    pl->P = P;
    pl->bucket_numel = bucket_numel;
    int64_t tiles = 0;
    for (int r = 0; r < K; ++r) {
        for (int p = 0; p < P; ++p) {
            if (numel[p] == 0) continue;
            const void* s = src[size_t(r) * P + p];
            if (!s) { delete pl; return DPR_ERR_INVALID_ARG; }
            if (!aligned(s, 2)) { delete pl; return DPR_ERR_ALIGNMENT; }
            FlatSeg g;
            g.src = static_cast<const uint16_t*>(s);
            g.dst_off = offset[p];
            g.numel = numel[p];
            g.tile0 = tiles;
            g.rank = r;
            g.pad = 0;
            tiles += (numel[p] + kFlatTile - 1) / kFlatTile;
            pl->segs.push_back(g);
        }
    }
    pl->n_tiles = tiles;
    pl->n_data_segs = int64_t(pl->segs.size());
    // zero-fill segments: the ranges of the bucket no gradient covers, per rank
    std::vector<std::pair<int64_t, int64_t>> gaps;
    int64_t at = 0;
    for (const auto& sp : spans) {
        if (sp.first > at) gaps.push_back({at, sp.first});
        at = std::max(at, sp.second);
    }
    if (at < bucket_numel) gaps.push_back({at, bucket_numel});
    for (const auto& gap : gaps) {
        for (int r = 0; r < K; ++r) {
            FlatSeg g;
            g.src = nullptr;
            g.dst_off = gap.first;
            g.numel = gap.second - gap.first;
            g.tile0 = tiles;
            g.rank = r;
            g.pad = 0;
            tiles += (g.numel + kFlatTile - 1) / kFlatTile;
            pl->segs.push_back(g);
        }
    }
    pl->n_tiles_zero = tiles;
    cudaError_t e = cudaGetDevice(&pl->device);
    if (e == cudaSuccess && !pl->segs.empty()) {
        const size_t bytes = pl->segs.size() * sizeof(FlatSeg);
        e = cudaMalloc(reinterpret_cast<void**>(&pl->d_segs), bytes);
        if (e == cudaSuccess)
            e = cudaMemcpyAsync(pl->d_segs, pl->segs.data(), bytes, cudaMemcpyHostToDevice,
                                static_cast<cudaStream_t>(stream));
        // one-time set-up: wait for the upload so the plan is usable on any stream
        if (e == cudaSuccess) e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    }
    if (e != cudaSuccess) {
        if (pl->d_segs) cudaFree(pl->d_segs);
        delete pl;
        return cuda_status(e);
    }
    *plan = pl;
    return DPR_OK;
}

dpr_status dpr_flatten_bucket(const dpr_flatten_plan* plan, void* const* dst, void* stream) {
    if (!plan || !dst) return DPR_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_status(e);
    if (dev != plan->device) return DPR_ERR_INVALID_ARG;
    std::vector<Span> outs;
    for (int r = 0; r < plan->K; ++r) {
        if (!dst[r]) return DPR_ERR_INVALID_ARG;
        if (!aligned(dst[r], 2)) return DPR_ERR_ALIGNMENT;
        outs.push_back(span_of(dst[r], uint64_t(plan->bucket_numel) * 2));
    }
    if (!pairwise_disjoint(outs)) return DPR_ERR_ALIAS;
    for (int64_t i = 0; i < plan->n_data_segs; ++i) {
        const FlatSeg& g = plan->segs[size_t(i)];
        const Span a = span_of(g.src, uint64_t(g.numel) * 2);
        for (const Span& o : outs)
            if (overlaps(a, o)) return DPR_ERR_ALIAS;
    }
    if (plan->n_tiles == 0) return DPR_OK;
    FlatParams p;
    std::memset(&p, 0, sizeof(p));
    p.segs = plan->d_segs;
    p.n_seg = plan->n_data_segs;
    p.n_tiles = plan->n_tiles;
    for (int r = 0; r < plan->K; ++r) p.dst[r] = static_cast<uint16_t*>(dst[r]);
    return cuda_status(launch_flatten(p, static_cast<cudaStream_t>(stream)));
}

dpr_status dpr_flatten_plan_destroy(dpr_flatten_plan* plan) {
    if (!plan) return DPR_OK;
    cudaError_t e = cudaSuccess;
    if (plan->d_segs) e = cudaFree(plan->d_segs);
    delete plan;
    return cuda_status(e);
}

dpr_status dpr_bucket_assign(const int64_t* numel, int P, int64_t cap, int64_t pad_to,
                             int32_t* bucket_of, int64_t* offset, int64_t* bucket_numel,
                             int* n_buckets) {
    if (!n_buckets || P < 0 || cap <= 0 || pad_to <= 0) return DPR_ERR_INVALID_ARG;
    *n_buckets = 0;
    if (P == 0) return DPR_OK;
    if (!numel || !bucket_of || !offset || !bucket_numel) return DPR_ERR_INVALID_ARG;
    for (int p = 0; p < P; ++p)
        if (numel[p] <= 0) return DPR_ERR_INVALID_ARG;
    int nb = 0;
    int64_t used = 0;
    bool open = false;
    auto flush = [&]() {
        if (!open) return;
        bucket_numel[nb] = (used + pad_to - 1) / pad_to * pad_to;
        ++nb;
        used = 0;
        open = false;
    };
    for (int p = 0; p < P; ++p) {
        if (open && used + numel[p] > cap) flush();
        bucket_of[p] = nb;
        offset[p] = used;
        used += numel[p];
        open = true;
    }
    flush();
    *n_buckets = nb;
    return DPR_OK;
}

const char* dpr_strerror(int status) {
    switch (status) {
        case DPR_OK: return "success";
        case DPR_ERR_INVALID_ARG: return "invalid argument";
        case DPR_ERR_ALIGNMENT: return "misaligned buffer";
        case DPR_ERR_UNSUPPORTED: return "size beyond the supported limits";
        case DPR_ERR_CUDA: return "CUDA call failed (see dpr_last_cuda_error)";
        case DPR_ERR_ALIAS: return "buffers overlap";
        default: return "unknown status";
    }
}

int dpr_last_cuda_error(void) { return g_last_cuda_error; }

const char* dpr_version(void) { return "libdpr 0.1 (sm_103a)"; }

}  // extern "C"
