// Kernel parameter blocks and host-side launchers of libdpr (internal).
//
// Every parameter block is passed to its kernel by value as a
// __grid_constant__ argument, so a launch needs no device-side table of
// pointers and allocates nothing.
#pragma once

#include <cstdint>
#include <vector>

#include <cuda_runtime.h>

#include "../../include/dpr.h"

namespace dpr {

constexpr int kThreads = 256;      // threads per block of every kernel

// How a kernel orders itself after the grid before it on its stream when it
// is launched as a programmatic dependent launch (see launch_kernel):
//  kAfterPrevious   wait for the previous grid before the first access to any
//                   caller buffer (every single call);
//  kBesidePrevious  the previous grid is a member of the same batch call and
//                   the host has checked that it touches none of this grid's
//                   outputs, nor writes any of its inputs: start at once; one
//                   block waits for it before exiting, so this grid still
//                   completes after its predecessor and stream order of
//                   completion stays transitive for whatever comes next.
constexpr int kAfterPrevious = 0;
constexpr int kBesidePrevious = 1;

struct RsParams {
    const uint16_t* in[DPR_MAX_MICRO * DPR_MAX_RANKS];  // in[m*K + r]
    float* out[DPR_MAX_RANKS];                          // partition shard j
    int64_t S;          // elements per chunk
    uint32_t su;        // 2*width-element units per chunk (vector kernels), edge unit included
    int K;
    int M;
    float scale;
    int accumulate;
    int order;          // kAfterPrevious / kBesidePrevious
    int edge;           // see edge_unit(): width 8 with one 8-element unit per chunk
};

struct ArParams {
    const uint16_t* in[DPR_MAX_RANKS];
    uint16_t* out[DPR_MAX_RANKS];
    int64_t S;
    uint32_t su;
    int K;
    float scale;
    int order;
    int edge;
};

struct AgParams {
    const uint16_t* shard[DPR_MAX_RANKS];
    uint16_t* out[DPR_MAX_RANKS];
    int64_t S;
    uint64_t tiles_per_chunk;   // ceil(S / kAgTile) (vector kernel)
    uint64_t in_place;          // bit j: shard[j] == out[j] + j*S
    int K;
    int order;
};

// One gradient of one rank inside a flatten plan, or (src == nullptr) one
// range of a rank's bucket that no gradient covers, to be zeroed.
struct FlatSeg {
    const uint16_t* src;
    int64_t dst_off;    // element offset inside the rank's flat bucket
    int64_t numel;
    int64_t tile0;      // index of this segment's first tile in the plan
    int32_t rank;
    int32_t pad;
};

struct FlatParams {
    const FlatSeg* segs;
    int64_t n_seg;
    int64_t n_tiles;
    uint16_t* dst[DPR_MAX_RANKS];
    int order;
};

constexpr int64_t kFlatTile = 4096;     // elements per flatten tile (8 KB), one block each
constexpr int kAgTile = 8192;           // elements per all-gather tile (16 KB), one block each

// Access width of the vector kernels, in 32-bit words per rank and access:
// 8 (32-byte accesses) when every buffer is 32-byte aligned and S % 16 == 0,
// 4 (16-byte) when every buffer is 16-byte aligned and S % 8 == 0, else 0
// (element-wise kernels).
inline int access_width(int64_t S, bool aligned32, bool aligned16) {
    if (aligned32 && S % 16 == 0) return 8;
    if (aligned16 && S % 8 == 0) return 4;
    return 0;
}

// The reduce-scatter and all-reduce also take 32-byte accesses when every
// buffer is 32-byte aligned, S % 16 == 8, the chunk is long (S >=
// kEdgeMinChunk) and the layout is built for K (below, all even); the
// all-reduce only out of place.  Chunk j then starts 8 elements past a
// 32-byte boundary when j is odd.  Its 32-byte units start at the first
// boundary, and one more unit, a 32-byte window reaching 8 elements into the
// neighbouring chunk, covers the 8 elements left over: the head of an odd
// chunk, the tail of an even one (K even: every even chunk has a chunk after
// it).  The unit count per chunk is (S - 8) / 16 + 1.
// Measured on GB300 at K = 8 (isolated launches): 5-8% faster than 16-byte
// accesses from S = 4.2M elements up, equal at 3.7M, 3-5% slower at 3.1M and
// 2.1M (shorter launches gain from the 16-byte kernel's finer blocks), so
// shorter chunks keep 16-byte accesses.
// The layout is built for the reduce-scatter at K = 2, 4, 8, 16, 32 and the
// all-reduce at K = 2, 4, 8: there it fits 64 registers, spilling at most 4
// bytes (the fp32 reduce-scatter at K = 16 and 32).
constexpr int64_t kEdgeMinChunk = int64_t(1) << 22;
inline bool edge_unit(int64_t S, int K, bool aligned32, bool allreduce) {
    const bool built = allreduce ? (K == 2 || K == 4 || K == 8)
                                 : (K == 2 || K == 4 || K == 8 || K == 16 || K == 32);
    return built && aligned32 && S % 16 == 8 && S >= kEdgeMinChunk;
}

// Units per chunk of the vector kernels for `width` (and the edge layout).
inline uint32_t chunk_units(int64_t S, int width, bool edge) {
    if (width <= 0) return 0;
    return edge ? uint32_t((S - 8) / 16 + 1) : uint32_t(S / (2 * width));
}

// Launches `kernel` (kThreads threads per block) on `s` with the parameter
// block(s) in `args`.  When programmatic launches are enabled (the default,
// dpr_set_programmatic_launch) and `s` is not the legacy default stream, the
// launch carries CUDA's programmatic stream serialization attribute, so the
// grid may be scheduled while the previous grid on `s` drains; the kernel's
// `order` field says what it waits for.  `programmatic` = false forces a
// plain launch (work after cross-stream event waits, or after host-to-device
// copies of data the kernel reads before its wait).
cudaError_t launch_kernel(const void* kernel, dim3 grid, void** args, cudaStream_t s,
                          bool programmatic = true);

// Launchers: return cudaSuccess or the launch error.  `width` as above;
// RsParams::su / ArParams::su hold S / (2 * width) when width > 0.
// max_blocks > 0 caps the grid at about that many blocks (grid-stride).
cudaError_t launch_reduce_scatter(const RsParams& p, int mode, int width, cudaStream_t s,
                                  int max_blocks = 0, bool programmatic = true);

// The checks of dpr_reduce_scatter, filling `p` and the access width on
// success; nothing is launched.
dpr_status prepare_reduce_scatter(const void* const* in, int K, int M, int64_t N,
                                  float* const* out, int mode, float scale, int accumulate,
                                  RsParams* p, int* width);

// The checks of dpr_allgather and dpr_allreduce, filling the parameter block
// and the access width on success (nothing is launched).
dpr_status prepare_allgather(const void* const* shard, int K, int64_t N, void* const* out,
                             AgParams* p, int* width);
dpr_status prepare_allreduce(const void* const* in, int K, int64_t N, void* const* out,
                             int mode, float scale, ArParams* p, int* width);

// dpr_reduce_scatter with a block budget (0 = the whole GPU); `programmatic`
// as for launch_kernel.
dpr_status reduce_scatter_capped(const void* const* in, int K, int M, int64_t N, float* const* out,
                                 int mode, float scale, int accumulate, cudaStream_t stream,
                                 int max_blocks, bool programmatic = true);
cudaError_t launch_allreduce(const ArParams& p, int mode, int width, cudaStream_t s);
// bf16 partition shards (RsParams::out points at bf16 buffers).
cudaError_t launch_reduce_scatter_bf16(const RsParams& p, int mode, int width, cudaStream_t s);
cudaError_t launch_cast(const uint16_t* in, float* out, uint64_t n, bool vec, cudaStream_t s);
cudaError_t launch_allgather(const AgParams& p, int width, cudaStream_t s);
cudaError_t launch_flatten(const FlatParams& p, cudaStream_t s, bool programmatic = true);

// Maps a CUDA result to a status, remembering a failure for
// dpr_last_cuda_error() (per calling thread).
dpr_status record_cuda_status(cudaError_t e);

// Grid helper: blocks per chunk so that K chunks together fill the GPU with
// `blocks_per_sm` resident blocks per SM, and no more blocks than there is work.
cudaError_t blocks_per_chunk(const void* kernel, int K, uint64_t work_per_chunk, int* gx);

}  // namespace dpr

// A flatten plan (see dpr_flatten_plan_create): the host and device copies of
// its segment table.  The table lists the gradients' segments (tiles
// [0, n_tiles)) followed by one zero-fill segment per rank and uncovered
// range of the bucket (tiles [n_tiles, n_tiles_zero)); dpr_flatten_bucket
// runs the first part only, the bucket pipeline both, so that a reused IPG
// buffer holds no stale data where no gradient lands.
struct dpr_flatten_plan {
    int K = 0;
    int P = 0;
    int device = 0;
    int64_t bucket_numel = 0;
    int64_t n_tiles = 0;
    int64_t n_tiles_zero = 0;           // tiles including the zero-fill segments
    int64_t n_data_segs = 0;            // segments holding gradients
    std::vector<dpr::FlatSeg> segs;     // host copy
    dpr::FlatSeg* d_segs = nullptr;     // device copy
};

// Is programmatic dependent launch enabled (process-wide)?
bool programmatic_launch_enabled();
