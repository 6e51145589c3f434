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
#include "host_checks.h"

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
    // every event is created once, here, and re-recorded on each use (a wait
    // enqueued earlier keeps referring to the record it saw)
    std::vector<cudaEvent_t> done;      // per physical buffer: its last reduction finished
    std::vector<cudaEvent_t> ready;     // per physical buffer: its gather finished
    std::vector<cudaEvent_t> produced;  // per producer slot: the producer's work so far
    cudaEvent_t tail = nullptr;         // everything queued on the reduction stream
    std::vector<bool> used;
    int next = 0;
    uint64_t submitted = 0;
};

namespace {

void destroy_pipeline(dpr_bucket_pipeline* pl) {
    if (!pl) return;
    for (auto* v : {&pl->done, &pl->ready, &pl->produced})
        for (cudaEvent_t e : *v)
            if (e) cudaEventDestroy(e);
    if (pl->tail) cudaEventDestroy(pl->tail);
    if (pl->reduction) cudaStreamDestroy(pl->reduction);
    if (pl->ipg) cudaFree(pl->ipg);
    delete pl;
}

uint16_t* slice(const dpr_bucket_pipeline* pl, int b, int r) {
    return pl->ipg + (int64_t(b) * pl->K + r) * pl->capacity;
}

cudaError_t make_events(std::vector<cudaEvent_t>* v, int n) {
    for (int i = 0; i < n; ++i) {
        cudaEvent_t ev = nullptr;
        const cudaError_t e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming);
        if (e != cudaSuccess) return e;
        v->push_back(ev);
    }
    return cudaSuccess;
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
    if (e == cudaSuccess) e = make_events(&pl->done, n_buffers);
    if (e == cudaSuccess) e = make_events(&pl->ready, n_buffers);
    if (e == cudaSuccess) e = make_events(&pl->produced, DPR_PIPELINE_MAX_PRODUCERS);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&pl->tail, cudaEventDisableTiming);
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
    // every check first: a rejected call enqueues nothing
    if (!pl || !plan || !out || n_producers < 0 || (n_producers > 0 && !producers))
        return DPR_ERR_INVALID_ARG;
    if (n_producers > DPR_PIPELINE_MAX_PRODUCERS) return DPR_ERR_UNSUPPORTED;
    if (plan->K != pl->K || plan->bucket_numel > pl->capacity) return DPR_ERR_INVALID_ARG;
    if (plan->bucket_numel % pl->K != 0) return DPR_ERR_INVALID_ARG;
    if (mode != DPR_SUM_RING_FP32 && mode != DPR_SUM_HOP_BF16) return DPR_ERR_INVALID_ARG;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_status(e);
    if (dev != pl->device || dev != plan->device) return DPR_ERR_INVALID_ARG;
    if (plan->bucket_numel == 0) return DPR_OK;
    const int K = pl->K;
    const int64_t S = plan->bucket_numel / K;
    std::vector<Span> outs;
    for (int j = 0; j < K; ++j) {
        if (!out[j]) return DPR_ERR_INVALID_ARG;
        if (!aligned(out[j], 4)) return DPR_ERR_ALIGNMENT;
        outs.push_back(span_of(out[j], uint64_t(S) * 4));
    }
    const Span ipg = span_of(pl->ipg, uint64_t(pl->n_buffers) * K * uint64_t(pl->capacity) * 2);
    if (!pairwise_disjoint(outs) || any_overlap(outs, {ipg})) return DPR_ERR_ALIAS;
    cudaStream_t cur = static_cast<cudaStream_t>(current_stream);
    const int b = pl->next;

    // 1. every stream that produced this bucket's gradients finishes first
    for (int i = 0; i < n_producers && e == cudaSuccess; ++i) {
        cudaStream_t ps = static_cast<cudaStream_t>(producers[i]);
        if (ps == cur) continue;
        e = cudaEventRecord(pl->produced[size_t(i)], ps);
        if (e == cudaSuccess) e = cudaStreamWaitEvent(cur, pl->produced[size_t(i)], 0);
    }
    // 2. buffer reuse: wait for this buffer's previous reduction (per buffer),
    //    or for everything queued on the reduction stream (reverse wait)
    if (e == cudaSuccess) {
        if (pl->policy == DPR_WAIT_PER_BUFFER) {
            if (pl->used[b]) e = cudaStreamWaitEvent(cur, pl->done[b], 0);
        } else if (pl->submitted > 0) {
            e = cudaEventRecord(pl->tail, pl->reduction);
            if (e == cudaSuccess) e = cudaStreamWaitEvent(cur, pl->tail, 0);
        }
    }
    if (e != cudaSuccess) return record_cuda_status(e);
    // 3. one kernel on the compute stream gathers the bucket into the physical
    //    buffer and zeroes the positions no gradient covers (stale data of
    //    earlier buckets); plain launches, since every kernel here follows a
    //    cross-stream wait
    FlatParams fp;
    std::memset(&fp, 0, sizeof(fp));
    fp.segs = plan->d_segs;
    fp.n_seg = int64_t(plan->segs.size());
    fp.n_tiles = plan->n_tiles_zero;
    for (int r = 0; r < K; ++r) fp.dst[r] = slice(pl, b, r);
    fp.order = kAfterPrevious;
    if (fp.n_tiles > 0) e = launch_flatten(fp, cur, false);
    // 4. the reduction stream waits for the gather, reduce-scatters, and marks
    //    the buffer's completion
    if (e == cudaSuccess) e = cudaEventRecord(pl->ready[b], cur);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(pl->reduction, pl->ready[b], 0);
    if (e != cudaSuccess) return record_cuda_status(e);
    const void* in[DPR_MAX_RANKS];
    for (int r = 0; r < K; ++r) in[r] = slice(pl, b, r);
    dpr_status st = reduce_scatter_capped(in, K, 1, plan->bucket_numel, out, mode, scale,
                                          accumulate, pl->reduction, pl->max_blocks, false);
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
