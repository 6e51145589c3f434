// Stream-overlapped bucket pipeline: gradient buckets are gathered into a
// small ring of physical IPG buffers on the caller's (compute) stream and
// reduce-scattered on the pipeline's own reduction stream, so backward
// compute that produces bucket N+1 can run while bucket N is being reduced.
//
// Issue "ZeRO-1/2 average_tensor serializes backward compute behind the
// preceding reduction" (DeepSpeed issue 8364) describes the ordering rules:
//   - the reduction of a bucket must wait for every stream that produced its
//     gradients (the multi-producer dependency of issues 8061/8080);
//   - a physical IPG buffer must not be overwritten while the reduction of its
//     previous bucket still reads it (the ping-pong reuse race of 5606);
//   - making the compute stream wait for ALL queued reductions whenever a
//     bucket is enqueued (the "reverse wait") is what serialises compute
//     behind the previous bucket's collective; the proposed fix records a
//     completion event per physical buffer and waits on it only before that
//     buffer is written again.
// Both policies are available: DPR_WAIT_PER_BUFFER (the fix) and
// DPR_WAIT_REDUCTION_STREAM (the behaviour the issue measures), so the two
// can be compared on the same work.
#include <algorithm>
#include <cstring>
#include <new>
#include <utility>
#include <vector>

#include "dpr_kernels.h"

using namespace dpr;

struct dpr_bucket_pipeline {
    int K = 0;
    int n_buffers = 0;
    int policy = 0;
    int max_blocks = 0;                 // block budget of the reductions (0 = whole GPU)
    int device = 0;
    int64_t capacity = 0;               // elements per rank slice of one IPG buffer
    uint16_t* ipg = nullptr;            // n_buffers * K * capacity bf16
    cudaStream_t reduction = nullptr;
    std::vector<cudaEvent_t> done;      // per physical buffer: its last reduction finished
    std::vector<bool> used;
    int next = 0;
    uint64_t submitted = 0;
};

namespace {

void destroy_pipeline(dpr_bucket_pipeline* pl) {
    if (!pl) return;
    for (cudaEvent_t e : pl->done)
        if (e) cudaEventDestroy(e);
    if (pl->reduction) cudaStreamDestroy(pl->reduction);
    if (pl->ipg) cudaFree(pl->ipg);
    delete pl;
}

uint16_t* slice(const dpr_bucket_pipeline* pl, int b, int r) {
    return pl->ipg + (int64_t(b) * pl->K + r) * pl->capacity;
}

// Ranges of [0, bucket_numel) that no gradient of the plan covers (the padding
// that rounds a bucket up to equal chunks, or gaps between gradients).
std::vector<std::pair<int64_t, int64_t>> uncovered(const dpr_flatten_plan* plan) {
    std::vector<std::pair<int64_t, int64_t>> spans;
    for (const FlatSeg& g : plan->segs)
        if (g.rank == 0) spans.push_back({g.dst_off, g.dst_off + g.numel});
    std::sort(spans.begin(), spans.end());
    std::vector<std::pair<int64_t, int64_t>> gaps;
    int64_t at = 0;
    for (const auto& sp : spans) {
        if (sp.first > at) gaps.push_back({at, sp.first});
        at = std::max(at, sp.second);
    }
    if (at < plan->bucket_numel) gaps.push_back({at, plan->bucket_numel});
    return gaps;
}

}  // namespace

extern "C" {

dpr_status dpr_bucket_pipeline_create(dpr_bucket_pipeline** out, int K, int64_t bucket_capacity,
                                      int n_buffers, int wait_policy, int max_blocks) {
    if (!out) return DPR_ERR_INVALID_ARG;
    *out = nullptr;
    if (K < 2 || K > DPR_MAX_RANKS || n_buffers < 1 || n_buffers > 16 || bucket_capacity <= 0)
        return DPR_ERR_INVALID_ARG;
    if (wait_policy != DPR_WAIT_PER_BUFFER && wait_policy != DPR_WAIT_REDUCTION_STREAM)
        return DPR_ERR_INVALID_ARG;
    if (bucket_capacity > DPR_MAX_ELEMS) return DPR_ERR_UNSUPPORTED;
    if (max_blocks < 0) return DPR_ERR_INVALID_ARG;
    dpr_bucket_pipeline* pl = new (std::nothrow) dpr_bucket_pipeline();
    if (!pl) return DPR_ERR_CUDA;
    pl->K = K;
    pl->n_buffers = n_buffers;
    pl->policy = wait_policy;
    pl->max_blocks = max_blocks;
    pl->capacity = (bucket_capacity + 15) / 16 * 16;   // 32-byte aligned rank slices
    cudaError_t e = cudaGetDevice(&pl->device);
    if (e == cudaSuccess)
        e = cudaMalloc(reinterpret_cast<void**>(&pl->ipg),
                       size_t(n_buffers) * K * size_t(pl->capacity) * 2);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&pl->reduction, cudaStreamNonBlocking);
    for (int b = 0; b < n_buffers && e == cudaSuccess; ++b) {
        cudaEvent_t ev = nullptr;
        e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        pl->done.push_back(ev);
    }
    pl->used.assign(n_buffers, false);
    if (e != cudaSuccess) {
        destroy_pipeline(pl);
        return record_cuda_status(e);
    }
    *out = pl;
    return DPR_OK;
}

dpr_status dpr_bucket_pipeline_submit(dpr_bucket_pipeline* pl, const dpr_flatten_plan* plan,
                                      float* const* out, int mode, float scale, int accumulate,
                                      void* const* producers, int n_producers,
                                      void* current_stream) {
    if (!pl || !plan || !out || n_producers < 0 || (n_producers > 0 && !producers))
        return DPR_ERR_INVALID_ARG;
    if (plan->K != pl->K || plan->bucket_numel > pl->capacity) return DPR_ERR_INVALID_ARG;
    if (plan->bucket_numel % pl->K != 0) return DPR_ERR_INVALID_ARG;
    if (mode != DPR_SUM_RING_FP32 && mode != DPR_SUM_HOP_BF16) return DPR_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_status(e);
    if (dev != pl->device || dev != plan->device) return DPR_ERR_INVALID_ARG;
    if (plan->bucket_numel == 0) return DPR_OK;
    cudaStream_t cur = static_cast<cudaStream_t>(current_stream);
    const int b = pl->next;
    const int K = pl->K;

    // 1. every stream that produced this bucket's gradients finishes first
    for (int i = 0; i < n_producers && e == cudaSuccess; ++i) {
        cudaStream_t ps = static_cast<cudaStream_t>(producers[i]);
        if (ps == cur) continue;
        cudaEvent_t ev = nullptr;
        e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventRecord(ev, ps);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cur, ev, 0);
        if (ev) cudaEventDestroy(ev);   // released once the recorded work completes
    }
    // 2. buffer reuse: wait for this buffer's previous reduction (per buffer),
    //    or for everything queued on the reduction stream (reverse wait)
    if (e == cudaSuccess) {
        if (pl->policy == DPR_WAIT_PER_BUFFER) {
            if (pl->used[b]) e = cudaStreamWaitEvent(cur, pl->done[b], 0);
        } else if (pl->submitted > 0) {
            cudaEvent_t ev = nullptr;
            e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
            if (e == cudaSuccess) e = cudaEventRecord(ev, pl->reduction);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(cur, ev, 0);
            if (ev) cudaEventDestroy(ev);
        }
    }
    if (e != cudaSuccess) return record_cuda_status(e);
    // 3. gather the bucket into the physical buffer on the compute stream;
    //    positions no gradient covers are zeroed (stale data of earlier buckets)
    void* dst[DPR_MAX_RANKS];
    for (int r = 0; r < K; ++r) dst[r] = slice(pl, b, r);
    for (const auto& gap : uncovered(plan))
        for (int r = 0; r < K && e == cudaSuccess; ++r)
            e = cudaMemsetAsync(slice(pl, b, r) + gap.first, 0, size_t(gap.second - gap.first) * 2, cur);
    if (e != cudaSuccess) return record_cuda_status(e);
    dpr_status st = dpr_flatten_bucket(plan, dst, cur);
    if (st != DPR_OK) return st;
    // 4. the reduction stream waits for the gather, reduce-scatters, and marks
    //    the buffer's completion
    cudaEvent_t ready = nullptr;
    e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(ready, cur);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pl->reduction, ready, 0);
    if (ready) cudaEventDestroy(ready);
    if (e != cudaSuccess) return record_cuda_status(e);
    const void* in[DPR_MAX_RANKS];
    for (int r = 0; r < K; ++r) in[r] = slice(pl, b, r);
    st = reduce_scatter_capped(in, K, 1, plan->bucket_numel, out, mode, scale, accumulate,
                               pl->reduction, pl->max_blocks);
    if (st != DPR_OK) return st;
    e = cudaEventRecord(pl->done[b], pl->reduction);
    if (e != cudaSuccess) return record_cuda_status(e);
    pl->used[b] = true;
    pl->next = (b + 1) % pl->n_buffers;
    ++pl->submitted;
    return DPR_OK;
}

dpr_status dpr_bucket_pipeline_flush(dpr_bucket_pipeline* pl, void* current_stream) {
    if (!pl) return DPR_ERR_INVALID_ARG;
    cudaStream_t cur = static_cast<cudaStream_t>(current_stream);
    cudaError_t e = cudaSuccess;
    for (int b = 0; b < pl->n_buffers && e == cudaSuccess; ++b)
        if (pl->used[b]) e = cudaStreamWaitEvent(cur, pl->done[b], 0);
    return record_cuda_status(e);
}

dpr_status dpr_bucket_pipeline_stream(const dpr_bucket_pipeline* pl, void** stream) {
    if (!pl || !stream) return DPR_ERR_INVALID_ARG;
    *stream = pl->reduction;
    return DPR_OK;
}

dpr_status dpr_bucket_pipeline_destroy(dpr_bucket_pipeline* pl) {
    if (!pl) return DPR_OK;
    cudaError_t e = pl->reduction ? cudaStreamSynchronize(pl->reduction) : cudaSuccess;
    destroy_pipeline(pl);
    return record_cuda_status(e);
}

}  // extern "C"
