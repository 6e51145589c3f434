"""ZeRO gradient-bucket reduction on one GB300 GPU (sm_103a).

K data-parallel ranks are simulated as K buffers in one GPU's memory.  The
library libdpr (C ABI in include/dpr.h, CUDA kernels in csrc/) provides the
flat-bucket gather of fragmented gradients, the ring-order reduce-scatter
with averaging and the fp32 partition cast, the all-gather and the fused
all-reduce.  This package is the thin Python binding of those calls.
"""
from ._binding import (  # noqa: F401
    WAIT_PER_BUFFER,
    WAIT_REDUCTION_STREAM,
    BucketPipeline,
    HOP_BF16,
    CoalescedPlan,
    LIB_PATH,
    RING_FP32,
    DprError,
    Request,
    FlattenPlan,
    FragmentsPlan,
    dpr_allgather,
    dpr_allgather_batch,
    dpr_allgather_init,
    dpr_allreduce,
    dpr_allreduce_init,
    dpr_allgather_coalesced,
    dpr_bucket_assign,
    dpr_cast_bf16_to_fp32,
    dpr_cost_allreduce,
    dpr_cost_best_segments,
    dpr_cost_crossover,
    dpr_cost_dp_speedup,
    dpr_cost_ring_broadcast,
    dpr_coalesced_plan_create,
    dpr_coalesced_plan_destroy,
    dpr_flatten_bucket,
    dpr_flatten_bucket_noalloc,
    dpr_flatten_plan_create,
    dpr_flatten_plan_destroy,
    dpr_fragments_plan_create,
    dpr_fragments_plan_destroy,
    dpr_reduce_scatter,
    dpr_reduce_scatter_batch,
    dpr_reduce_scatter_bf16,
    dpr_reduce_scatter_coalesced,
    dpr_reduce_scatter_fragments,
    dpr_reduce_scatter_fragments_batch,
    dpr_reduce_scatter_init,
    dpr_set_programmatic_launch,
    dpr_strerror,
    dpr_version,
    lib,
)
