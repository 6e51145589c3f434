// Persistent collectives: a call's arguments are checked and its kernel
// parameter block is built once, at initialisation; each start launches the
// prepared kernel on a stream.  This follows the persistent collective
// operations of MPI-4 (MPI_Allreduce_init / MPI_Start): a training loop
// reduces the same buckets into the same partitions at every step, and for
// buckets of a few MiB the host's per-call checks cost as much as the GPU's
// work.
#include <cstring>
#include <new>

#include "dpr_kernels.h"
#include "host_checks.h"

using namespace dpr;

struct dpr_request {
    int kind = 0;          // 0 reduce-scatter, 1 all-gather, 2 all-reduce
    int mode = 0;
    int width = 0;
    int device = 0;
    bool empty = false;    // N == 0: start launches nothing
    RsParams rs;
    AgParams ag;
    ArParams ar;
};

namespace {

enum { kReduceScatter = 0, kAllGather = 1, kAllReduce = 2 };

dpr_status finish_init(dpr_request* rq, dpr_request** out) {
    const cudaError_t e = cudaGetDevice(&rq->device);
    if (e != cudaSuccess) {
        delete rq;
        return record_cuda_status(e);
    }
    *out = rq;
    return DPR_OK;
}

}  // namespace

extern "C" {

dpr_status dpr_reduce_scatter_init(dpr_request** req, const void* const* in, int K, int M,
                                   int64_t N, float* const* out, int mode, float scale,
                                   int accumulate) {
    if (!req) return DPR_ERR_INVALID_ARG;
    *req = nullptr;
    dpr_request* rq = new (std::nothrow) dpr_request();
    if (!rq) return DPR_ERR_CUDA;
    const dpr_status st = prepare_reduce_scatter(in, K, M, N, out, mode, scale, accumulate,
                                                 &rq->rs, &rq->width);
    if (st != DPR_OK) {
        delete rq;
        return st;
    }
    rq->kind = kReduceScatter;
    rq->mode = mode;
    rq->empty = N == 0;
    return finish_init(rq, req);
}

dpr_status dpr_allgather_init(dpr_request** req, const void* const* shard, int K, int64_t N,
                              void* const* out) {
    if (!req) return DPR_ERR_INVALID_ARG;
    *req = nullptr;
    dpr_request* rq = new (std::nothrow) dpr_request();
    if (!rq) return DPR_ERR_CUDA;
    const dpr_status st = prepare_allgather(shard, K, N, out, &rq->ag, &rq->width);
    if (st != DPR_OK) {
        delete rq;
        return st;
    }
    rq->kind = kAllGather;
    rq->empty = N == 0;
    return finish_init(rq, req);
}

dpr_status dpr_allreduce_init(dpr_request** req, const void* const* in, int K, int64_t N,
                              void* const* out, int mode, float scale) {
    if (!req) return DPR_ERR_INVALID_ARG;
    *req = nullptr;
    dpr_request* rq = new (std::nothrow) dpr_request();
    if (!rq) return DPR_ERR_CUDA;
    const dpr_status st = prepare_allreduce(in, K, N, out, mode, scale, &rq->ar, &rq->width);
    if (st != DPR_OK) {
        delete rq;
        return st;
    }
    rq->kind = kAllReduce;
    rq->mode = mode;
    rq->empty = N == 0;
    return finish_init(rq, req);
}

dpr_status dpr_start(const dpr_request* req, void* stream) {
    if (!req) return DPR_ERR_INVALID_ARG;
    if (req->empty) return DPR_OK;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return record_cuda_status(e);
    if (dev != req->device) return DPR_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    switch (req->kind) {
        case kReduceScatter: e = launch_reduce_scatter(req->rs, req->mode, req->width, s); break;
        case kAllGather: e = launch_allgather(req->ag, req->width, s); break;
        default: e = launch_allreduce(req->ar, req->mode, req->width, s); break;
    }
    return record_cuda_status(e);
}

dpr_status dpr_request_free(dpr_request* req) {
    delete req;
    return DPR_OK;
}

}  // extern "C"
