// dpr_flatten_bucket_noalloc: the flat-bucket gather for callers that must
// not allocate device memory.
//
// The plan-based gather keeps its segment table in memory that
// dpr_flatten_plan_create obtains with cudaMalloc.  Some callers cannot do
// that: a process whose device memory is already reserved up front by a
// caching allocator (so a separate cudaMalloc fails or fragments the pool), a
// plug-in that its host forbids from allocating after start-up, or a loop
// that cannot afford cudaMalloc/cudaFree, which may synchronise the whole
// device.  This entry point keeps the table in a fixed array compiled into
// the library instead (DPR_NOALLOC_MAX_SEGMENTS entries, 160 KiB, held by
// every GPU that loads the library until the process exits).  It performs no
// cudaMalloc, cudaFree or other allocating call; the caller still owns the
// source gradients and the destination buckets.
#include <algorithm>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "dpr_kernels.h"

namespace dpr {
namespace {

// Device scratch shared by every call: the segment table of the current call.
// Only the first n_seg entries of a call are read, and the call writes all of
// them, so nothing has to start at zero.  Host code must not take this name's
// address: it is a host-side stand-in.  The device address comes from
// cudaGetSymbolAddress below.
static __device__ __align__(256) FlatSeg g_noalloc_segs[DPR_NOALLOC_MAX_SEGMENTS];

std::mutex g_mu;                                  // guards the two tables below
std::map<int, FlatSeg*> g_table_addr;            // device -> address of g_noalloc_segs
FlatSeg g_host_segs[DPR_NOALLOC_MAX_SEGMENTS];   // host staging of one call's table
std::pair<int64_t, int64_t> g_spans[DPR_NOALLOC_MAX_SEGMENTS];

// Set-up, once per device, with that device current.
cudaError_t table_address(int dev, FlatSeg** out) {
    auto it = g_table_addr.find(dev);
    if (it != g_table_addr.end()) {
        *out = it->second;
        return cudaSuccess;
    }
    void* ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_segs);
    if (e != cudaSuccess) return e;
    g_table_addr[dev] = static_cast<FlatSeg*>(ptr);
    *out = static_cast<FlatSeg*>(ptr);
    return cudaSuccess;
}

bool is_aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

bool span_overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) {
    return a0 < b1 && b0 < a1;
}

}  // namespace
}  // namespace dpr

using namespace dpr;

extern "C" dpr_status dpr_flatten_bucket_noalloc(int K, int P, const void* const* src,
                                                 const int64_t* numel, const int64_t* offset,
                                                 int64_t bucket_numel, void* const* dst,
                                                 void* stream) {
    if (K < 1 || K > DPR_MAX_RANKS || P < 0 || bucket_numel < 0) return DPR_ERR_INVALID_ARG;
    if (bucket_numel > DPR_MAX_ELEMS) return DPR_ERR_UNSUPPORTED;
    if (P > 0 && (!src || !numel || !offset)) return DPR_ERR_INVALID_ARG;
    if (!dst) return DPR_ERR_INVALID_ARG;
    int64_t nonempty = 0;
    for (int p = 0; p < P; ++p) {
        if (numel[p] < 0 || offset[p] < 0) return DPR_ERR_INVALID_ARG;
        if (numel[p] == 0) continue;
        if (offset[p] > bucket_numel - numel[p]) return DPR_ERR_INVALID_ARG;
        ++nonempty;
    }
    // the fixed table holds K * (non-empty gradients) segments at most
    if (nonempty * K > DPR_NOALLOC_MAX_SEGMENTS) return DPR_ERR_UNSUPPORTED;
    for (int r = 0; r < K; ++r) {
        if (!dst[r]) return DPR_ERR_INVALID_ARG;
        if (!is_aligned(dst[r], 2)) return DPR_ERR_ALIGNMENT;
    }

    // A captured copy would re-read the shared host table at replay, after
    // later calls may have rewritten it: refuse capture before enqueueing.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(static_cast<cudaStream_t>(stream), &cap);
    if (e != cudaSuccess) return record_cuda_status(e);
    if (cap != cudaStreamCaptureStatusNone) return DPR_ERR_UNSUPPORTED;

    std::lock_guard<std::mutex> lock(g_mu);
    // gradient spans inside the bucket must not overlap
    int64_t ns = 0;
    for (int p = 0; p < P; ++p)
        if (numel[p] > 0) g_spans[ns++] = {offset[p], offset[p] + numel[p]};
    std::sort(g_spans, g_spans + ns);
    for (int64_t i = 1; i < ns; ++i)
        if (g_spans[i].first < g_spans[i - 1].second) return DPR_ERR_ALIAS;
    // destination buckets must not overlap each other or any source
    const uint64_t dbytes = uint64_t(bucket_numel) * 2;
    for (int r = 0; r < K; ++r) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(dst[r]);
        for (int q = r + 1; q < K; ++q) {
            const uintptr_t b = reinterpret_cast<uintptr_t>(dst[q]);
            if (span_overlap(a, a + dbytes, b, b + dbytes)) return DPR_ERR_ALIAS;
        }
    }
    int64_t n_seg = 0, tiles = 0;
    for (int r = 0; r < K; ++r) {
        for (int p = 0; p < P; ++p) {
            if (numel[p] == 0) continue;
            const void* s = src[size_t(r) * P + p];
            if (!s) return DPR_ERR_INVALID_ARG;
            if (!is_aligned(s, 2)) return DPR_ERR_ALIGNMENT;
            const uintptr_t s0 = reinterpret_cast<uintptr_t>(s);
            const uintptr_t s1 = s0 + uintptr_t(numel[p]) * 2;
            for (int q = 0; q < K; ++q) {
                const uintptr_t d0 = reinterpret_cast<uintptr_t>(dst[q]);
                if (span_overlap(s0, s1, d0, d0 + dbytes)) return DPR_ERR_ALIAS;
            }
            FlatSeg& g = g_host_segs[n_seg++];
            g.src = static_cast<const uint16_t*>(s);
            g.dst_off = offset[p];
            g.numel = numel[p];
            g.tile0 = tiles;
            g.rank = r;
            g.pad = 0;
            tiles += (numel[p] + kFlatTile - 1) / kFlatTile;
        }
    }
    if (n_seg == 0) return DPR_OK;

    int dev = 0;
    e = cudaGetDevice(&dev);
    FlatSeg* table = nullptr;
    if (e == cudaSuccess) e = table_address(dev, &table);
    // Pageable-memory copy: returns once the host table has been staged, so the
    // host staging array can be reused by the next call; the device copy is
    // ordered on `stream` before the gather kernel.
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(table, g_host_segs, size_t(n_seg) * sizeof(FlatSeg),
                            cudaMemcpyHostToDevice, static_cast<cudaStream_t>(stream));
    if (e == cudaSuccess) {
        FlatParams prm;
        std::memset(&prm, 0, sizeof(prm));
        prm.segs = table;
        prm.n_seg = n_seg;
        prm.n_tiles = tiles;
        for (int r = 0; r < K; ++r) prm.dst[r] = static_cast<uint16_t*>(dst[r]);
        prm.order = kAfterPrevious;
        // plain launch: the kernel reads the table before any wait, so it must
        // not start before the copy above has landed
        e = launch_flatten(prm, static_cast<cudaStream_t>(stream), false);
    }
    return record_cuda_status(e);
}
