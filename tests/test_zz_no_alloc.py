"""dpr_flatten_bucket_noalloc: the flat-bucket gather for callers that cannot
allocate device memory -- for example a process whose GPU memory a caching
allocator has reserved up front, a plug-in that may not allocate after
start-up, or a loop that cannot pay for cudaMalloc/cudaFree synchronising the
device.  It keeps its segment table in a fixed array inside the library.

These tests call it through the C ABI and compare its output, bit for bit,
with the plan-based gather (dpr_flatten_plan_create + dpr_flatten_bucket) and
with the oracle's gather on two calls in a row; check that a call beyond the
fixed table is refused, and that a call on a capturing stream is refused
without breaking the capture.  The file's name sorts it last, so a failure
here cannot stop a run that halts at the first failure before the other GPU
tests have run; it also passes on its own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import flatten as ofl
from tests import gpu_helpers as H
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu

UNSUPPORTED = 3


def _case(K, numel, seed, dev):
    offsets, o = [], 0
    for n in numel:
        offsets.append(o)
        o += n
    bucket = o + 11
    srcs = []
    for r in range(K):
        row = []
        for p, n in enumerate(numel):
            base = torch.empty(n + 8, dtype=torch.bfloat16, device=dev)
            t = base[(r + p) % 3:(r + p) % 3 + n]          # mixed alignments
            t.copy_(syn.gauss_bf16(0, n, syn.stream_key(seed, r, 0, p), 1e-3).to(dev))
            row.append(t)
        srcs.append(row)
    return srcs, offsets, bucket


def _call_noalloc(L, srcs, numel, offsets, bucket, dst, stream):
    return _call_noalloc_raw(L, srcs, numel, offsets, bucket, dst, stream.cuda_stream)


def _call_noalloc_raw(L, srcs, numel, offsets, bucket, dst, stream_handle):
    K, P = len(srcs), len(numel)
    src_ptrs = (ctypes.c_void_p * (K * P))(*[t.data_ptr() for row in srcs for t in row])
    dst_ptrs = (ctypes.c_void_p * K)(*[t.data_ptr() for t in dst])
    n_arr = (ctypes.c_int64 * P)(*numel)
    o_arr = (ctypes.c_int64 * P)(*offsets)
    return L.dpr_flatten_bucket_noalloc(K, P, src_ptrs, n_arr, o_arr, bucket, dst_ptrs,
                                        stream_handle)


def test_noalloc_matches_plan_based_gather_two_calls_in_a_row():
    dev = H.device()
    L = dpr.lib()
    stream = torch.cuda.Stream()
    cases = [(4, [1000, 7, 8192 * 3 + 5, 64, 0, 1]), (8, [16384, 3, 100_000, 8192])]
    built = [_case(K, numel, 50 + i, dev) for i, (K, numel) in enumerate(cases)]
    outs = []
    # two calls back to back on one stream, no synchronisation between them:
    # the second call's table upload is ordered after the first call's kernel
    for (K, numel), (srcs, offsets, bucket) in zip(cases, built):
        dst = [torch.zeros(bucket, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        assert _call_noalloc(L, srcs, numel, offsets, bucket, dst, stream) == 0
        outs.append(dst)
    stream.synchronize()
    for (K, numel), (srcs, offsets, bucket), got in zip(cases, built, outs):
        ref = [torch.zeros(bucket, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        with dpr.dpr_flatten_plan_create(srcs, numel, offsets, bucket) as plan:
            dpr.dpr_flatten_bucket(plan, ref)
            torch.cuda.synchronize()
        want = ofl.flatten_bucket([[H.bits(t) for t in row] for row in srcs], numel, offsets,
                                  bucket)
        for r in range(K):
            assert torch.equal(got[r].view(torch.int16), ref[r].view(torch.int16)), f"rank {r}"
            assert np.array_equal(H.bits(got[r]), want[r]), f"rank {r} differs from the oracle"


def test_noalloc_takes_no_device_memory_after_setup():
    dev = H.device()
    L = dpr.lib()
    stream = torch.cuda.Stream()
    srcs, offsets, bucket = _case(2, [5000, 300], 7, dev)
    dst = [torch.zeros(bucket, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    assert _call_noalloc(L, srcs, [5000, 300], offsets, bucket, dst, stream) == 0
    stream.synchronize()
    free0 = torch.cuda.mem_get_info()[0]
    for _ in range(3):
        assert _call_noalloc(L, srcs, [5000, 300], offsets, bucket, dst, stream) == 0
    stream.synchronize()
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_refuses_tables_beyond_the_fixed_array():
    dev = H.device()
    L = dpr.lib()
    K, P = 8, 513                  # 8 * 513 = 4104 segments > 4096
    srcs = [[torch.zeros(1, dtype=torch.bfloat16, device=dev) for _ in range(P)] for _ in range(K)]
    dst = [torch.zeros(P, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    assert _call_noalloc(L, srcs, [1] * P, list(range(P)), P, dst, torch.cuda.Stream()) == UNSUPPORTED
    with pytest.raises(dpr.DprError):
        dpr.dpr_flatten_bucket_noalloc(srcs, [1] * P, list(range(P)), P, dst)


def test_noalloc_is_refused_on_a_capturing_stream_and_the_capture_survives():
    """A captured call would replay a copy of the shared host table that later
    calls overwrite, so the call refuses a capturing stream; the capture goes
    on and the graph it makes replays."""
    dev = H.device()
    srcs, offsets, bucket = _case(2, [5000, 300], 9, dev)
    dst = [torch.zeros(bucket, dtype=torch.bfloat16, device=dev) for _ in range(2)]
    x = torch.ones(1024, device=dev)
    g = torch.cuda.CUDAGraph()
    refused = None
    with torch.cuda.graph(g):
        try:
            dpr.dpr_flatten_bucket_noalloc(srcs, [5000, 300], offsets, bucket, dst)
        except dpr.DprError as e:
            refused = e.status
        x.mul_(2.0)
    assert refused == UNSUPPORTED
    g.replay()
    torch.cuda.synchronize()
    assert float(x[0]) == 2.0
    assert all(int(t.view(torch.int16).abs().sum()) == 0 for t in dst)   # nothing was written
