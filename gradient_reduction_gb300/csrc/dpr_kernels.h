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

struct RsParams {
    const uint16_t* in[DPR_MAX_MICRO * DPR_MAX_RANKS];  // in[m*K + r]
    float* out[DPR_MAX_RANKS];                          // partition shard j
    int64_t S;          // elements per chunk
    uint32_t su;        // 2*width-element units per chunk (vector kernels)
    int K;
    int M;
    float scale;
    int accumulate;
};

struct ArParams {
    const uint16_t* in[DPR_MAX_RANKS];
    uint16_t* out[DPR_MAX_RANKS];
    int64_t S;
    uint32_t su;
    int K;
    float scale;
};

struct AgParams {
    const uint16_t* shard[DPR_MAX_RANKS];
    uint16_t* out[DPR_MAX_RANKS];
    int64_t S;
    uint64_t tiles_per_chunk;   // ceil(S / kAgTile) (vector kernel)
    uint64_t in_place;          // bit j: shard[j] == out[j] + j*S
    int K;
};

// One gradient of one rank inside a flatten plan.
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

// Launchers: return cudaSuccess or the launch error.  `width` as above;
// RsParams::su / ArParams::su hold S / (2 * width) when width > 0.
// max_blocks > 0 caps the grid at about that many blocks (grid-stride).
cudaError_t launch_reduce_scatter(const RsParams& p, int mode, int width, cudaStream_t s,
                                  int max_blocks = 0);

// dpr_reduce_scatter with a block budget (0 = the whole GPU).
dpr_status reduce_scatter_capped(const void* const* in, int K, int M, int64_t N, float* const* out,
                                 int mode, float scale, int accumulate, cudaStream_t stream,
                                 int max_blocks);
cudaError_t launch_allreduce(const ArParams& p, int mode, int width, cudaStream_t s);
// bf16 partition shards (RsParams::out points at bf16 buffers).
cudaError_t launch_reduce_scatter_bf16(const RsParams& p, int mode, int width, cudaStream_t s);
cudaError_t launch_cast(const uint16_t* in, float* out, uint64_t n, bool vec, cudaStream_t s);
cudaError_t launch_allgather(const AgParams& p, int width, cudaStream_t s);
cudaError_t launch_flatten(const FlatParams& p, cudaStream_t s);

// Maps a CUDA result to a status, remembering a failure for
// dpr_last_cuda_error() (per calling thread).
dpr_status record_cuda_status(cudaError_t e);

// Grid helper: blocks per chunk so that K chunks together fill the GPU with
// `blocks_per_sm` resident blocks per SM, and no more blocks than there is work.
cudaError_t blocks_per_chunk(const void* kernel, int K, uint64_t work_per_chunk, int* gx);

}  // namespace dpr

// A flatten plan (see dpr_flatten_plan_create): the host and device copies of
// its segment table.
struct dpr_flatten_plan {
    int K = 0;
    int P = 0;
    int device = 0;
    int64_t bucket_numel = 0;
    int64_t n_tiles = 0;
    std::vector<dpr::FlatSeg> segs;     // host copy
    dpr::FlatSeg* d_segs = nullptr;     // device copy
};
