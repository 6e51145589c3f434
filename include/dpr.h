/*
 * dpr.h -- C ABI of libdpr: the data-parallel gradient-bucket reduction of
 * ZeRO, with the K data-parallel ranks simulated as K buffers in the memory
 * of one GPU (sm_103a).
 *
 * Conventions shared by every call (after the NCCL call shape described in
 * CMU 11-868 Lecture 14 notes, section 2.3: send/receive buffers, an element
 * count, the reduction, and a CUDA stream):
 *   - every buffer pointer is a DEVICE pointer owned by the caller; pointer
 *     ARRAYS (in, out, shard, src, dst) are HOST arrays of such pointers and
 *     are read during the call only;
 *   - bf16 buffers are 16-bit IEEE bfloat16 bit patterns, 2-byte aligned;
 *     fp32 buffers are 4-byte aligned.  Buffers that are all 16-byte aligned
 *     with 8-element-aligned chunks take the vectorised kernels; any other
 *     layout takes an element-wise kernel with the same results;
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream); work is
 *     enqueued asynchronously, nothing synchronises, and completion (and any
 *     asynchronous execution error) is observed by synchronising the stream;
 *   - the reduce-scatter, all-gather and all-reduce calls allocate nothing
 *     and launch exactly one kernel; N == 0 is a no-op that launches nothing;
 *   - on a stream other than the legacy default stream, kernels are launched
 *     as programmatic dependent launches (see dpr_set_programmatic_launch):
 *     a kernel may be scheduled while the previous kernel on the stream
 *     drains, but it touches no caller buffer before that kernel has
 *     completed, so stream order of data is kept;
 *   - arguments are validated on the host before anything is launched; a
 *     rejected call returns its status and has no effect.  DPR_ERR_CUDA
 *     means a CUDA call failed; dpr_last_cuda_error() then returns its
 *     cudaError_t (per calling thread).
 *
 * Chunks: a rank buffer of N elements is cut into K equal chunks of S = N/K,
 * chunk j = elements [j*S, (j+1)*S).  N must be a multiple of K.
 */
#ifndef DPR_H
#define DPR_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum dpr_status {
    DPR_OK = 0,
    DPR_ERR_INVALID_ARG = 1, /* null pointer, K/M/N out of range, N % K != 0, bad mode */
    DPR_ERR_ALIGNMENT = 2,   /* a bf16 pointer not 2-byte / fp32 pointer not 4-byte aligned */
    DPR_ERR_UNSUPPORTED = 3, /* a size beyond the documented limits */
    DPR_ERR_CUDA = 4,        /* a CUDA call failed; see dpr_last_cuda_error() */
    DPR_ERR_ALIAS = 5        /* outputs overlap inputs or each other (beyond allowed in-place forms) */
} dpr_status;

typedef enum dpr_sum_mode {
    /* fp32 partial sums: each hop is one fp32 add, round to nearest even */
    DPR_SUM_RING_FP32 = 0,
    /* bf16 partial sums on the wire: each hop's fp32 sum is rounded back to bf16 */
    DPR_SUM_HOP_BF16 = 1
} dpr_sum_mode;

#define DPR_MAX_RANKS 64                 /* 2 <= K <= 64 */
#define DPR_MAX_MICRO 2                  /* 1 <= M <= 2 */
#define DPR_MAX_ELEMS (((int64_t)1) << 34) /* N per rank buffer */
#define DPR_MAX_BATCH 4096               /* members of one batched call */

/*
 * Ring reduce-scatter with averaging and the fp32 partition-gradient cast.
 *
 * Defines: CMU 11-868 Lecture 14 notes, section 3.2 (ring reduce-scatter:
 * in round i rank r sends chunk (r - i) mod K, the receiver adds it; after
 * K-1 rounds rank r holds the complete chunk (r + 1) mod K) and "Ring
 * All-Reduce illustrated" (CSDN), Phase 1: chunk j starts at rank j and
 * collects ranks j+1, ..., j-1.  The result is therefore, per element t of
 * chunk j, the sum in ring order
 *     acc = ((x_j[t] + x_{j+1}[t]) + x_{j+2}[t]) + ... + x_{j-1}[t]
 * (indices mod K; in DPR_SUM_HOP_BF16 every partial sum is rounded to bf16).
 * With M = 2, each rank's input is first its local accumulation
 * x_r = bf16(g0_r + g1_r) (lecture section 4.2, accumulate before reduce).
 * The landed sum is averaged and cast to fp32 into partition slot j
 * (DeepSpeed ZeRO-3 source walkthrough, sections 1, 5.2, 5.3 and 8):
 *     accumulate == 0:  out[j][t] = fp32(acc) * scale          (copy_)
 *     accumulate != 0:  out[j][t] = out[j][t] + fp32(acc)*scale (add_)
 * with the multiply and the add each rounded (no fused multiply-add).
 *
 *   in    host array [M*K]; in[m*K + r] = rank r's micro-batch m gradient,
 *         bf16, N elements.  Input buffers may overlap each other.
 *   K     ranks, 2..64;   M  micro-batches, 1..2;   N  elements per rank.
 *   out   host array [K]; out[j] = partition shard j, fp32, N/K elements.
 *         Shards must not overlap each other or any input.
 *   mode  dpr_sum_mode;   scale  fp32 multiplier (1.0f/K averages).
 */
dpr_status dpr_reduce_scatter(const void* const* in, int K, int M, int64_t N,
                              float* const* out, int mode, float scale, int accumulate,
                              void* stream);

/*
 * n reduce-scatters in one call: the buckets of a backward pass that are
 * ready together (DeepSpeed ZeRO-3 source walkthrough, section 5.1: each
 * full bucket is reduced as soon as it is flushed, one after another on the
 * reduction stream).  The result is that of n dpr_reduce_scatter calls in
 * order; member i uses in[i*M*K .. (i+1)*M*K), N[i] and out[i*K .. (i+1)*K)
 * (host arrays), with K, M, mode, scale and accumulate shared, and each
 * member is checked as dpr_reduce_scatter checks it.  In addition no output
 * shard of any member may overlap an output shard of another member or any
 * member's input (DPR_ERR_ALIAS), so the members are independent.  One
 * kernel is launched per member with N[i] > 0.  Because they are
 * independent, each member after the first is allowed to run beside the one
 * before it (a programmatic dependent launch that does not wait): the next
 * bucket's blocks fill the SMs while the previous bucket's last blocks
 * drain.  Each member still completes only after the one before it, so work
 * that follows on the stream sees all of them.  n: 0..DPR_MAX_BATCH.
 */
dpr_status dpr_reduce_scatter_batch(int n, const void* const* in, int K, int M, const int64_t* N,
                                    float* const* out, int mode, float scale, int accumulate,
                                    void* stream);

/*
 * Reduce-scatter into bf16 partition shards: the literal ZeRO-3 data flow
 * (DeepSpeed ZeRO-3 source walkthrough, sections 1, 5.3 and 8), where the
 * reduced shard lands in the rank's bf16 partition buffer -- copy_ on the
 * first micro step, add_ (in bf16) on later ones -- and the one bf16 -> fp32
 * conversion happens later, in step() (dpr_cast_bf16_to_fp32).
 *     accumulate == 0:  out[j][t] = bf16(fp32(acc) * scale)
 *     accumulate != 0:  out[j][t] = bf16(out[j][t] + bf16(fp32(acc) * scale))
 * acc, in, K, M, N, mode and scale exactly as dpr_reduce_scatter; out: host
 * array [K] of bf16 shards of N/K elements, not overlapping each other or any
 * input.
 */
dpr_status dpr_reduce_scatter_bf16(const void* const* in, int K, int M, int64_t N,
                                   void* const* out, int mode, float scale, int accumulate,
                                   void* stream);

/*
 * The step()-time cast of a bf16 partition to fp32 (exact widening):
 * out[t] = fp32(in[t]), n elements; in and out must not overlap.
 */
dpr_status dpr_cast_bf16_to_fp32(const void* in, float* out, int64_t n, void* stream);

/*
 * Ring all-gather of K shards into K full replicas.
 *
 * Defines: lecture section 3.2 and CSDN Phase 2 (complete chunks travel the
 * ring and overwrite, so every rank ends with all K chunks); the ZeRO-3
 * parameter all-gather that rebuilds full parameters from 1/K shards
 * (DeepSpeed ZeRO-3 source walkthrough, sections 1 and 2.1):
 *     out[r][j*S + t] = shard[j][t]   for every r, j, t   (a bit copy)
 *
 *   shard  host array [K]; shard[j] = bf16, S = N/K elements.
 *   out    host array [K]; out[r] = bf16, N elements.  Outputs must not
 *          overlap each other or any shard, except the in-place form
 *          shard[j] == out[j] + j*S (rank j's shard lives inside its own
 *          full buffer).
 */
dpr_status dpr_allgather(const void* const* shard, int K, int64_t N, void* const* out,
                         void* stream);

/*
 * n all-gathers in one call: the parameter all-gathers of ZeRO-3 that a
 * forward pass issues one layer after another (DeepSpeed ZeRO-3 source
 * walkthrough, sections 1 and 2.1).  The result is that of n dpr_allgather
 * calls in order; member i uses shard[i*K .. (i+1)*K), N[i] and
 * out[i*K .. (i+1)*K) (host arrays), and is checked as dpr_allgather checks
 * it (its own in-place form included).  In addition no output of any member
 * may overlap another member's outputs or shards (DPR_ERR_ALIAS), so the
 * members are independent and run beside one another as described for
 * dpr_reduce_scatter_batch.  One kernel per member with N[i] > 0.
 * n: 0..DPR_MAX_BATCH.
 */
dpr_status dpr_allgather_batch(int n, const void* const* shard, int K, const int64_t* N,
                               void* const* out, void* stream);

/*
 * Ring all-reduce = reduce-scatter + all-gather (lecture section 2.2), fused
 * into one pass: each element's ring-order sum (as in dpr_reduce_scatter,
 * M = 1) is multiplied by scale, rounded once to bf16, and written to every
 * replica, so all K outputs are bitwise identical (CSDN, end of Phase 2):
 *     out[r][t] = bf16(fp32(acc) * scale)   for every r
 * This is the contiguous-gradient path of ZeRO-3 (DeepSpeed ZeRO-3 source
 * walkthrough, section 5.2: all-reduce the flat bucket, then slice).
 *
 *   in   host array [K], bf16, N elements each.
 *   out  host array [K], bf16, N elements each; out[r] == in[r] (in place)
 *        is allowed, any other overlap is rejected.
 */
dpr_status dpr_allreduce(const void* const* in, int K, int64_t N, void* const* out, int mode,
                         float scale, void* stream);

/*
 * Persistent collectives (after MPI-4's persistent collective operations,
 * MPI_Allreduce_init / MPI_Start).  A ZeRO training loop reduces the same
 * buckets into the same partitions at every step; these calls check the
 * arguments and build the kernel's parameters once, so that each start costs
 * one launch.
 *
 * dpr_reduce_scatter_init, dpr_allgather_init and dpr_allreduce_init take the
 * arguments of dpr_reduce_scatter, dpr_allgather and dpr_allreduce (without
 * the stream), check them exactly as those calls do, record the current
 * device and return a request in *req (NULL on failure).  They allocate host
 * memory only and make no other CUDA call.  The pointer arrays are read
 * during the call; the buffers they point to must stay valid for as long as
 * the request is started.
 *
 * dpr_start enqueues the prepared collective on `stream` (the device current
 * at initialisation must be current; DPR_ERR_INVALID_ARG otherwise) with the
 * same results and stream semantics as the one-shot call; a request built
 * for N == 0 launches nothing.  dpr_request_free releases a request (NULL is
 * a no-op); work already enqueued is unaffected.
 */
typedef struct dpr_request dpr_request;

dpr_status dpr_reduce_scatter_init(dpr_request** req, const void* const* in, int K, int M,
                                   int64_t N, float* const* out, int mode, float scale,
                                   int accumulate);
dpr_status dpr_allgather_init(dpr_request** req, const void* const* shard, int K, int64_t N,
                              void* const* out);
dpr_status dpr_allreduce_init(dpr_request** req, const void* const* in, int K, int64_t N,
                              void* const* out, int mode, float scale);
dpr_status dpr_start(const dpr_request* req, void* stream);
dpr_status dpr_request_free(dpr_request* req);

/*
 * Flat-bucket gather plan (the IPG bucket of ZeRO: DeepSpeed ZeRO-3 source
 * walkthrough, sections 3.2 and 5.1).  Gradient p of rank r occupies
 * elements [offset[p], offset[p] + numel[p]) of rank r's flat bucket.  In the
 * pages' system the gradient is written there directly; here the per-rank
 * gradients already exist as separate buffers, so flattening is a copy.
 *
 * dpr_flatten_plan_create records the table once (offsets are fixed after
 * initialisation): it allocates a device copy of it (plan and pipeline
 * constructors are the only calls that allocate), uploads it on `stream` and
 * waits for the upload, so the plan can then be used on any stream.
 *   src          host array [K*P]; src[r*P + p] = rank r's gradient p, bf16.
 *   numel, offset host arrays [P], elements; spans must lie inside
 *                [0, bucket_numel) and not overlap.  numel[p] == 0 is allowed.
 *   *plan        receives the plan (NULL on failure).
 */
typedef struct dpr_flatten_plan dpr_flatten_plan;

dpr_status dpr_flatten_plan_create(dpr_flatten_plan** plan, int K, int P, const void* const* src,
                                   const int64_t* numel, const int64_t* offset,
                                   int64_t bucket_numel, void* stream);

/*
 * Executes a plan: one kernel copies every gradient of every rank into the
 * flat buckets, dst[r][offset[p] + t] = src[r*P + p][t] (a bit copy).
 * Positions no gradient covers (padding) are not written.
 *   dst  host array [K]; dst[r] = rank r's flat bucket, bf16, bucket_numel
 *        elements; must not overlap each other or any source gradient.
 * The plan must stay alive until the copy has completed on the stream.
 */
dpr_status dpr_flatten_bucket(const dpr_flatten_plan* plan, void* const* dst, void* stream);

/* Frees a plan (its device table); synchronises the device.  NULL is a no-op. */
dpr_status dpr_flatten_plan_destroy(dpr_flatten_plan* plan);

/*
 * Flat-bucket gather that allocates nothing.  The pages have no counterpart
 * of this call; it exists for callers that cannot call cudaMalloc: a process
 * whose device memory a caching allocator has already reserved (a separate
 * cudaMalloc fails or fragments its pool), a plug-in whose host forbids
 * allocation after start-up, or a loop that cannot afford cudaMalloc and
 * cudaFree, which may synchronise the whole device.
 *
 * Same copy as dpr_flatten_plan_create + dpr_flatten_bucket, with the same
 * argument meanings and checks, in one call: the segment table is built on
 * the host and copied (cudaMemcpyAsync on `stream`) into a fixed array
 * compiled into the library, then one kernel does the gather.  Limits and
 * sharing:
 *   - at most DPR_NOALLOC_MAX_SEGMENTS (rank, non-empty gradient) pairs per
 *     call, i.e. K * P_nonempty <= 4096; larger calls return
 *     DPR_ERR_UNSUPPORTED and do nothing.  The array (160 KiB) is held by
 *     every GPU that loads the library until the process exits;
 *   - every call shares that array and overwrites the entries it uses (no
 *     entry needs to start at zero).  Calls ordered on one stream are safe;
 *     calls that overlap on the GPU (different streams, or other host threads'
 *     streams, without ordering between them) race on the table and must be
 *     avoided;
 *   - the first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress) with that device current;
 *   - the host table is copied from pageable memory, so the call returns
 *     only after the copy has been staged;
 *   - the call cannot be captured into a CUDA graph: a captured copy would
 *     re-read the shared host table at replay, when a later call may have
 *     overwritten it.  On a stream that is capturing it returns
 *     DPR_ERR_UNSUPPORTED, enqueues nothing and leaves the capture intact;
 *   - the gather kernel is a plain launch (it reads the table the copy just
 *     wrote), so it starts only after all earlier work on the stream.
 */
#define DPR_NOALLOC_MAX_SEGMENTS 4096

dpr_status dpr_flatten_bucket_noalloc(int K, int P, const void* const* src, const int64_t* numel,
                                      const int64_t* offset, int64_t bucket_numel,
                                      void* const* dst, void* stream);

/*
 * Reduce-scatter of a flat bucket straight from its fragments: the result of
 * dpr_flatten_bucket followed by dpr_reduce_scatter (M = 1), without the flat
 * bucket.  In ZeRO the gradients are written into the IPG bucket in the first
 * place (DeepSpeed ZeRO-3 source walkthrough, sections 3.2 and 5.1); when
 * they already exist as separate buffers, gathering them costs a write and a
 * re-read of the whole bucket, which this call skips.
 *
 * dpr_fragments_plan_create takes the arguments of dpr_flatten_plan_create
 * (same meanings and checks) and additionally needs K >= 2 and
 * bucket_numel % K == 0.  It records, for every tile of every chunk, which
 * gradient (or gap) covers which run of its elements, allocates and uploads
 * those tables and the pointer table (cudaMalloc), and waits for the upload.
 *
 * dpr_reduce_scatter_fragments: with B_r = rank r's bucket as
 * dpr_flatten_bucket would lay it out and positions no gradient covers equal
 * to zero,
 *     out[j][t] = scale * (ring-order sum over ranks, starting at rank j, of
 *                 B_r[j*S + t])                                   (copy_)
 *     out[j][t] = out[j][t] + that                                 (add_)
 * S = bucket_numel / K; mode, scale and accumulate as in dpr_reduce_scatter.
 * out: host array [K] of fp32 shards of S elements, not overlapping each other
 * or any source gradient.  One kernel launch on `stream`.
 */
typedef struct dpr_fragments_plan dpr_fragments_plan;

dpr_status dpr_fragments_plan_create(dpr_fragments_plan** plan, int K, int P, const void* const* src,
                                     const int64_t* numel, const int64_t* offset,
                                     int64_t bucket_numel, void* stream);
dpr_status dpr_reduce_scatter_fragments(const dpr_fragments_plan* plan, float* const* out, int mode,
                                        float scale, int accumulate, void* stream);
dpr_status dpr_fragments_plan_destroy(dpr_fragments_plan* plan);

/*
 * n buckets reduce-scattered straight from their fragments in one call, as
 * dpr_reduce_scatter_batch does for flat buckets: the result of n
 * dpr_reduce_scatter_fragments calls in order, member i with plans[i] and
 * out[i*K_i ..] (out is a host array of the members' K_i shard pointers,
 * concatenated), mode, scale and accumulate shared.  No output shard may
 * overlap another member's output shards or any member's source gradients
 * (DPR_ERR_ALIAS); the members then run beside one another as described for
 * dpr_reduce_scatter_batch.  n: 0..DPR_MAX_BATCH.
 */
dpr_status dpr_reduce_scatter_fragments_batch(int n, const dpr_fragments_plan* const* plans,
                                              float* const* out, int mode, float scale,
                                              int accumulate, void* stream);

/*
 * Per-parameter partitioning (ZeRO-3): the discrete reduction path and the
 * parameter all-gather.  DeepSpeed ZeRO-3 source walkthrough, section 1:
 * every parameter lives as a 1/N shard per rank; section 5.2: with
 * fragmented gradients the list of per-parameter gradients is
 * reduce-scattered directly, without a flat bucket.
 *
 * Layout: parameter p of numel[p] elements is treated as zero-padded to
 * K * s_p, s_p = ceil(numel[p] / K); rank j owns elements [j*s_p, (j+1)*s_p).
 * Rank j's partition buffer holds its shards of all parameters in parameter
 * order: the shard of p starts at offset_p = s_0 + ... + s_{p-1}, and the
 * partition holds dpr_coalesced_partition_numel() elements.
 *
 * dpr_coalesced_plan_create binds the K*P per-rank tensors (gradients for the
 * reduce-scatter, parameters for the all-gather; tensors[r*P + p] = rank r's
 * tensor of parameter p, bf16, numel[p] elements, non-overlapping) and
 * uploads a segment table, a per-tile map and the pointer table once
 * (cudaMalloc, about 8 bytes per 4096 gradient elements of one rank; waits for
 * the upload).  numel[p] == 0 is allowed.
 *
 * dpr_reduce_scatter_coalesced: out[j][offset_p + t] = scale * (ring-order
 * sum over ranks, starting at rank j, of tensors[r*P + p][j*s_p + t]), padding
 * summing to zero; mode, scale and accumulate as in dpr_reduce_scatter
 * (one micro-batch).  out: host array [K] of fp32 partition buffers, not
 * overlapping each other or the bound tensors.
 *
 * dpr_allgather_coalesced: tensors[r*P + p][j*s_p + t] = shards[j][offset_p + t]
 * for every r, j and every t with j*s_p + t < numel[p] (padding dropped).
 * shards: host array [K] of bf16 partition buffers, not overlapping the bound
 * tensors.
 *
 * Each call launches one kernel on `stream`; plan destruction frees the
 * tables and synchronises the device.
 */
typedef struct dpr_coalesced_plan dpr_coalesced_plan;

dpr_status dpr_coalesced_plan_create(dpr_coalesced_plan** plan, int K, int P, void* const* tensors,
                                     const int64_t* numel, void* stream);
dpr_status dpr_coalesced_partition_numel(const dpr_coalesced_plan* plan, int64_t* numel);
dpr_status dpr_reduce_scatter_coalesced(const dpr_coalesced_plan* plan, float* const* out, int mode,
                                        float scale, int accumulate, void* stream);
dpr_status dpr_allgather_coalesced(const dpr_coalesced_plan* plan, const void* const* shards,
                                   void* stream);
dpr_status dpr_coalesced_plan_destroy(dpr_coalesced_plan* plan);

/*
 * Stream-overlapped bucket pipeline.  The issue "ZeRO-1/2 average_tensor
 * serializes backward compute behind the preceding reduction" (DeepSpeed
 * issue 8364) states the ordering a ZeRO bucket reduction needs when
 * gradients are gathered into a ring of physical IPG buffers on the compute
 * stream and reduced on a separate reduction stream:
 *   - the reduction of a bucket waits for every stream that produced its
 *     gradients (multi-producer dependency);
 *   - a physical buffer is not overwritten while the reduction of its
 *     previous bucket still reads it (ping-pong reuse);
 * and shows that making the compute stream wait for ALL queued reductions at
 * every enqueue serialises compute behind the previous bucket's collective.
 * Its proposed fix waits, per physical buffer, only for that buffer's last
 * reduction.  Both behaviours are available for comparison:
 *   DPR_WAIT_PER_BUFFER        the per-buffer completion events (the fix);
 *   DPR_WAIT_REDUCTION_STREAM  the reverse wait on the whole reduction stream.
 *
 * dpr_bucket_pipeline_create allocates n_buffers (1..16) IPG buffers of K
 * rank slices of bucket_capacity bf16 elements each (cudaMalloc), a
 * non-blocking reduction stream and every event the pipeline records: a
 * completion and a gather event per buffer, one event per producer slot
 * (DPR_PIPELINE_MAX_PRODUCERS) and one for the reverse wait.  Submitting
 * creates no event and allocates nothing.
 * max_blocks > 0 caps each reduction at about that many thread blocks, so the
 * reduction leaves SMs to compute running beside it (as NCCL runs its
 * collectives on a small grid); 0 lets a reduction use the whole GPU.
 *
 * dpr_bucket_pipeline_submit, for one bucket described by a flatten plan:
 *   1. makes current_stream wait for each of the n_producers streams;
 *   2. makes current_stream wait for the chosen buffer's previous reduction
 *      (DPR_WAIT_PER_BUFFER) or for all queued reductions;
 *   3. on current_stream, one kernel gathers the bucket (as
 *      dpr_flatten_bucket) into the next physical buffer and zeroes the
 *      positions no gradient covers;
 *   4. on the reduction stream, after step 3, reduce-scatters the buffer into
 *      out (as dpr_reduce_scatter with M = 1, mode, scale, accumulate) and
 *      records the buffer's completion event.
 * Requires plan K == the pipeline's K, bucket_numel <= bucket_capacity and
 * n_producers <= DPR_PIPELINE_MAX_PRODUCERS (else DPR_ERR_UNSUPPORTED); out
 * (fp32 shards, 4-byte aligned) must not overlap each other or the
 * pipeline's buffers.  Every check runs before anything is enqueued.  out
 * must stay valid until the reduction completes.  The pipeline's kernels
 * are plain launches (they follow cross-stream waits).
 *
 * dpr_bucket_pipeline_flush makes current_stream wait for every submitted
 * reduction (the epilogue of a backward pass).  dpr_bucket_pipeline_stream
 * returns the reduction stream (a cudaStream_t owned by the pipeline) so that
 * callers can order other work against it.  dpr_bucket_pipeline_destroy
 * waits for the reduction stream and frees everything.
 */
#define DPR_WAIT_PER_BUFFER 0
#define DPR_WAIT_REDUCTION_STREAM 1
#define DPR_PIPELINE_MAX_PRODUCERS 8

typedef struct dpr_bucket_pipeline dpr_bucket_pipeline;

dpr_status dpr_bucket_pipeline_create(dpr_bucket_pipeline** pipeline, int K, int64_t bucket_capacity,
                                      int n_buffers, int wait_policy, int max_blocks);
dpr_status dpr_bucket_pipeline_submit(dpr_bucket_pipeline* pipeline, const dpr_flatten_plan* plan,
                                      float* const* out, int mode, float scale, int accumulate,
                                      void* const* producers, int n_producers,
                                      void* current_stream);
dpr_status dpr_bucket_pipeline_flush(dpr_bucket_pipeline* pipeline, void* current_stream);
dpr_status dpr_bucket_pipeline_stream(const dpr_bucket_pipeline* pipeline, void** stream);
dpr_status dpr_bucket_pipeline_destroy(dpr_bucket_pipeline* pipeline);

/*
 * Bucket formation, host only (DeepSpeed ZeRO-3 source walkthrough, sections
 * 3.1, 5.1, 5.4): gradients in arrival order are appended at the running
 * offset; the bucket is flushed first when adding the next gradient would
 * take it past `cap` elements; a gradient larger than `cap` forms its own
 * bucket; the last, partly filled bucket is flushed at the end.  Each
 * bucket's size is rounded up to a multiple of `pad_to` (K, for equal
 * chunks); the padding is never written by dpr_flatten_bucket.
 *   numel        [P] gradient sizes in arrival order (each >= 1)
 *   bucket_of    [P] out: bucket index of each gradient
 *   offset       [P] out: element offset of each gradient in its bucket
 *   bucket_numel [P] out: padded size of each bucket (first *n_buckets used)
 */
dpr_status dpr_bucket_assign(const int64_t* numel, int P, int64_t cap, int64_t pad_to,
                             int32_t* bucket_of, int64_t* offset, int64_t* bucket_numel,
                             int* n_buckets);

/*
 * Alpha-beta cost model (host only; CMU 11-868 Lecture 14 notes, sections 3.1,
 * 3.4 and 4.4).  A message of n bytes costs alpha + n / beta seconds; K
 * devices, `bytes` per device:
 *   DPR_ALGO_RING   2(K-1) (alpha + bytes / (K beta))
 *   DPR_ALGO_TREE   2 ceil(log2 K) (alpha + bytes / beta)
 *   DPR_ALGO_NAIVE  2 (alpha + (K-1) bytes / beta)
 * dpr_cost_ring_broadcast: a ring broadcast cut into S segments,
 *   (K - 2 + S) (alpha + bytes / (S beta)); S = 1 is the unsegmented case.
 * dpr_cost_best_segments: the best S among 1, 2, 4, ... <= max_segments.
 * dpr_cost_crossover: the message size at which two all-reduce algorithms
 *   cost the same (DPR_ERR_UNSUPPORTED if they never cross).
 * dpr_cost_dp_speedup: T1 / (T1 / K + ring all-reduce time), the speed-up of
 *   K-way data parallelism without overlap for a single-device step of T1.
 * Invalid arguments (beta <= 0, negative sizes, unknown algorithm) return
 * DPR_ERR_INVALID_ARG.
 */
#define DPR_ALGO_RING 0
#define DPR_ALGO_TREE 1
#define DPR_ALGO_NAIVE 2

dpr_status dpr_cost_allreduce(int algo, int K, double bytes, double alpha, double beta,
                              double* seconds);
dpr_status dpr_cost_ring_broadcast(int K, double bytes, double alpha, double beta, int64_t segments,
                                   double* seconds);
dpr_status dpr_cost_best_segments(int K, double bytes, double alpha, double beta,
                                  int64_t max_segments, int64_t* segments, double* seconds);
dpr_status dpr_cost_crossover(int algo_a, int algo_b, int K, double alpha, double beta,
                              double* bytes);
dpr_status dpr_cost_dp_speedup(double t1, int K, double bytes, double alpha, double beta,
                               double* speedup);

/*
 * Programmatic dependent launch, process-wide.  enable != 0 (the default):
 * on every stream but the legacy default stream, each kernel is launched
 * with CUDA's programmatic stream serialization, reads only its plan's fixed
 * tables and its own arguments before the previous kernel on the stream has
 * completed, and waits for that completion before touching any caller
 * buffer; it saves the gap between a grid's drain and the next grid's start.
 * Members after the first of a batched call do not wait (see
 * dpr_reduce_scatter_batch).  enable == 0 launches every kernel plainly
 * (for comparison); results are the same either way.  *previous (may be
 * NULL) receives the setting before the call.
 */
dpr_status dpr_set_programmatic_launch(int enable, int* previous);

/* Static description of a status code. */
const char* dpr_strerror(int status);

/* cudaError_t of the calling thread's last DPR_ERR_CUDA (0 if none). */
int dpr_last_cuda_error(void);

/* Library version string. */
const char* dpr_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DPR_H */
