"""ctypes binding of libdpr (include/dpr.h), with the same entry-point names.

Argument marshalling only: tensors are turned into device pointers and sizes,
the current CUDA stream is passed along, and a non-zero status becomes a
DprError.  The checks here (dtype, device, contiguity, element counts) exist
so that a wrongly sized tensor is rejected on the host instead of being read
out of bounds on the GPU.  Every step of the computation runs in libdpr's
kernels; there is no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
import os
from typing import Sequence

import torch

RING_FP32 = 0
HOP_BF16 = 1
_MODES = {"ring_fp32": RING_FP32, "hop_bf16": HOP_BF16, RING_FP32: RING_FP32, HOP_BF16: HOP_BF16}

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_lib", "libdpr.so")

_c_p = ctypes.c_void_p
_pp = ctypes.POINTER(ctypes.c_void_p)
_i64p = ctypes.POINTER(ctypes.c_int64)
_SIGS = {
    "dpr_reduce_scatter": [_pp, ctypes.c_int, ctypes.c_int, ctypes.c_int64, _pp, ctypes.c_int,
                           ctypes.c_float, ctypes.c_int, _c_p],
    "dpr_reduce_scatter_batch": [ctypes.c_int, _pp, ctypes.c_int, ctypes.c_int, _i64p, _pp,
                                 ctypes.c_int, ctypes.c_float, ctypes.c_int, _c_p],
    "dpr_allgather": [_pp, ctypes.c_int, ctypes.c_int64, _pp, _c_p],
    "dpr_allgather_batch": [ctypes.c_int, _pp, ctypes.c_int, _i64p, _pp, _c_p],
    "dpr_reduce_scatter_bf16": [_pp, ctypes.c_int, ctypes.c_int, ctypes.c_int64, _pp, ctypes.c_int,
                                ctypes.c_float, ctypes.c_int, _c_p],
    "dpr_cast_bf16_to_fp32": [_c_p, _c_p, ctypes.c_int64, _c_p],
    "dpr_allreduce": [_pp, ctypes.c_int, ctypes.c_int64, _pp, ctypes.c_int, ctypes.c_float, _c_p],
    "dpr_flatten_plan_create": [ctypes.POINTER(_c_p), ctypes.c_int, ctypes.c_int, _pp, _i64p,
                                _i64p, ctypes.c_int64, _c_p],
    "dpr_flatten_bucket": [_c_p, _pp, _c_p],
    "dpr_flatten_plan_destroy": [_c_p],
    "dpr_bucket_assign": [_i64p, ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                          ctypes.POINTER(ctypes.c_int32), _i64p, _i64p,
                          ctypes.POINTER(ctypes.c_int)],
    "dpr_flatten_bucket_noalloc": [ctypes.c_int, ctypes.c_int, _pp, _i64p, _i64p, ctypes.c_int64,
                                   _pp, _c_p],
    "dpr_fragments_plan_create": [ctypes.POINTER(_c_p), ctypes.c_int, ctypes.c_int, _pp, _i64p,
                                  _i64p, ctypes.c_int64, _c_p],
    "dpr_reduce_scatter_fragments": [_c_p, _pp, ctypes.c_int, ctypes.c_float, ctypes.c_int, _c_p],
    "dpr_reduce_scatter_fragments_batch": [ctypes.c_int, _pp, _pp, ctypes.c_int, ctypes.c_float,
                                           ctypes.c_int, _c_p],
    "dpr_fragments_plan_destroy": [_c_p],
    "dpr_coalesced_plan_create": [ctypes.POINTER(_c_p), ctypes.c_int, ctypes.c_int, _pp, _i64p,
                                  _c_p],
    "dpr_coalesced_partition_numel": [_c_p, _i64p],
    "dpr_reduce_scatter_coalesced": [_c_p, _pp, ctypes.c_int, ctypes.c_float, ctypes.c_int, _c_p],
    "dpr_allgather_coalesced": [_c_p, _pp, _c_p],
    "dpr_coalesced_plan_destroy": [_c_p],
    "dpr_bucket_pipeline_create": [ctypes.POINTER(_c_p), ctypes.c_int, ctypes.c_int64, ctypes.c_int,
                                   ctypes.c_int, ctypes.c_int],
    "dpr_bucket_pipeline_submit": [_c_p, _c_p, _pp, ctypes.c_int, ctypes.c_float, ctypes.c_int, _pp,
                                   ctypes.c_int, _c_p],
    "dpr_bucket_pipeline_flush": [_c_p, _c_p],
    "dpr_bucket_pipeline_stream": [_c_p, ctypes.POINTER(_c_p)],
    "dpr_bucket_pipeline_destroy": [_c_p],
    "dpr_cost_allreduce": [ctypes.c_int, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                           ctypes.c_double, ctypes.POINTER(ctypes.c_double)],
    "dpr_cost_ring_broadcast": [ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                                ctypes.c_int64, ctypes.POINTER(ctypes.c_double)],
    "dpr_cost_best_segments": [ctypes.c_int, ctypes.c_double, ctypes.c_double, ctypes.c_double,
                               ctypes.c_int64, ctypes.POINTER(ctypes.c_int64),
                               ctypes.POINTER(ctypes.c_double)],
    "dpr_cost_crossover": [ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_double,
                           ctypes.c_double, ctypes.POINTER(ctypes.c_double)],
    "dpr_cost_dp_speedup": [ctypes.c_double, ctypes.c_int, ctypes.c_double, ctypes.c_double,
                            ctypes.c_double, ctypes.POINTER(ctypes.c_double)],
    "dpr_set_programmatic_launch": [ctypes.c_int, ctypes.POINTER(ctypes.c_int)],
    "dpr_reduce_scatter_init": [ctypes.POINTER(_c_p), _pp, ctypes.c_int, ctypes.c_int,
                                ctypes.c_int64, _pp, ctypes.c_int, ctypes.c_float, ctypes.c_int],
    "dpr_allgather_init": [ctypes.POINTER(_c_p), _pp, ctypes.c_int, ctypes.c_int64, _pp],
    "dpr_allreduce_init": [ctypes.POINTER(_c_p), _pp, ctypes.c_int, ctypes.c_int64, _pp,
                           ctypes.c_int, ctypes.c_float],
    "dpr_start": [_c_p, _c_p],
    "dpr_request_free": [_c_p],
    "dpr_strerror": [ctypes.c_int],
    "dpr_last_cuda_error": [],
    "dpr_version": [],
}
_RESTYPES = {"dpr_strerror": ctypes.c_char_p, "dpr_version": ctypes.c_char_p}

_lib = None


class DprError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        msg = lib().dpr_strerror(status).decode()
        if status == 4:
            msg += f" (cudaError {lib().dpr_last_cuda_error()})"
        super().__init__(f"{fn}: {msg} [status {status}]")


def lib() -> ctypes.CDLL:
    """The loaded libdpr; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(
                f"libdpr is not built ({LIB_PATH} missing): run "
                "`python -m gradient_reduction_gb300.build` (needs nvcc)")
        L = ctypes.CDLL(LIB_PATH)
        for name, args in _SIGS.items():
            f = getattr(L, name)
            f.argtypes = args
            f.restype = _RESTYPES.get(name, ctypes.c_int)
        _lib = L
    return _lib


def _check(fn: str, status: int):
    if status != 0:
        raise DprError(fn, status)


def _ptrs(ts: Sequence[torch.Tensor]):
    return (ctypes.c_void_p * len(ts))(*[t.data_ptr() for t in ts])


# The current stream's handle without building a torch.cuda.Stream object
# (which costs a few microseconds per call); the public route serves when
# this accessor is absent or CUDA is not initialised yet.
_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream) -> int:
    if stream is None:
        if _raw_stream is not None and torch.cuda.is_initialized():
            return _raw_stream(torch.cuda.current_device())
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _rows_contiguous(x: torch.Tensor) -> bool:
    """Is every x[i] laid out contiguously (row-major over the dimensions after
    the first)?"""
    expect = 1
    for size, st in zip(reversed(x.shape[1:]), reversed(x.stride()[1:])):
        if size != 1 and st != expect:
            return False
        expect *= size
    return True


def _rows(x, count: int, dtype, n: int, what: str, check: bool = True):
    """Host array of `count` device pointers, one per rank buffer.  `x` is a
    sequence of tensors (one per buffer) or one CUDA tensor whose first
    dimension indexes the buffers, each of which is contiguous (for example a
    [K, N] tensor); the stacked form is checked once, whatever `count` is."""
    if not isinstance(x, torch.Tensor):
        if check:
            _need(x, count, dtype, n, what)
        return _ptrs(x)
    if check:
        if not x.is_cuda or x.dtype != dtype:
            raise ValueError(f"{what}: need a CUDA {dtype} tensor")
        dev = torch.cuda.current_device()
        if x.get_device() != dev:
            raise ValueError(f"{what}: tensor on cuda:{x.get_device()}, current device is cuda:{dev}")
        if x.dim() < 2 or x.shape[0] != count:
            raise ValueError(f"{what}: expected a tensor of {count} rows, got shape {tuple(x.shape)}")
        if not (x.is_contiguous() or _rows_contiguous(x)):
            raise ValueError(f"{what}: every row must be contiguous")
        if x.numel() // max(count, 1) < n:
            raise ValueError(f"{what}: rows of {x.numel() // max(count, 1)} elements, need {n}")
    base, step = x.data_ptr(), x.stride(0) * x.element_size()
    if step > 0:
        return (ctypes.c_void_p * count)(*range(base, base + count * step, step))
    return (ctypes.c_void_p * count)(*([base] * count))


def _need(ts: Sequence[torch.Tensor], count: int, dtype, n: int, what: str):
    if len(ts) != count:
        raise ValueError(f"{what}: expected {count} tensors, got {len(ts)}")
    dev = None
    for t in ts:
        if not t.is_cuda or t.dtype != dtype or not t.is_contiguous():
            raise ValueError(f"{what}: need contiguous CUDA {dtype} tensors")
        if dev is None:
            dev = torch.cuda.current_device()
        if t.get_device() != dev:
            # the kernels run on the current device and would fault on another's memory
            raise ValueError(f"{what}: tensor on cuda:{t.get_device()}, current device is cuda:{dev}")
        if t.numel() < n:
            raise ValueError(f"{what}: tensor of {t.numel()} elements, need {n}")


def dpr_reduce_scatter(inputs, K: int, M: int, N: int, outputs, mode=RING_FP32,
                       scale: float | None = None, accumulate: bool = False,
                       stream=None) -> None:
    """inputs[m*K + r]: bf16 (N,), rank r micro-batch m; outputs[j]: fp32 (N/K,).
    Either argument may also be one tensor of M*K (K) contiguous rows."""
    chk = N > 0
    ins = _rows(inputs, M * K, torch.bfloat16, N, "inputs", chk)
    outs = _rows(outputs, K, torch.float32, N // K if K else 0, "outputs", chk)
    st = lib().dpr_reduce_scatter(ins, K, M, N, outs, _MODES[mode],
                                  1.0 / K if scale is None else scale, int(bool(accumulate)),
                                  _stream(stream))
    _check("dpr_reduce_scatter", st)


def _member_rows(x, n: int, count: int, dtype, sizes: Sequence[int], what: str):
    """Pointers of n members' `count` buffers, member after member.  `x` is a
    sequence with one entry per member (each a sequence of tensors or one
    tensor of `count` rows), or one tensor [n, count, ...] whose rows are
    contiguous, checked once (its members may lie at any stride)."""
    if isinstance(x, torch.Tensor):
        if x.dim() < 3 or x.shape[0] != n or x.shape[1] != count:
            raise ValueError(f"{what}: expected a tensor of {n} members of {count} rows, "
                             f"got shape {tuple(x.shape)}")
        if n == 0 or x.stride(0) == count * x.stride(1):
            # merging the first two dimensions is a view, never a copy, given the strides
            return _rows(x.flatten(0, 1), n * count, dtype, max(sizes, default=0), what)
        # every member shares the first member's row layout: check that once
        _rows(x[0], count, dtype, max(sizes, default=0), what)
        es = x.element_size()
        base, s0, s1 = x.data_ptr(), x.stride(0) * es, x.stride(1) * es
        return (ctypes.c_void_p * (n * count))(
            *[base + i * s0 + j * s1 for i in range(n) for j in range(count)])
    if len(x) != n:
        raise ValueError(f"{what}: need one entry per member")
    arrs = [_rows(x[i], count, dtype, sizes[i], f"{what}[{i}]", sizes[i] > 0) for i in range(n)]
    for i, a in enumerate(arrs):
        if len(a) != count:
            raise ValueError(f"{what}[{i}]: expected {count} buffers, got {len(a)}")
    return (ctypes.c_void_p * (n * count))(*[p for a in arrs for p in a])


def dpr_reduce_scatter_batch(inputs, K: int, M: int, N: Sequence[int], outputs,
                             mode=RING_FP32, scale: float | None = None, accumulate: bool = False,
                             stream=None) -> None:
    """Member i: inputs[i][m*K + r] bf16 (N[i],), outputs[i][j] fp32 (N[i]/K,);
    inputs may also be one tensor [n, M*K, >= max N], outputs one tensor
    [n, K, >= max N/K].  The members must be independent (no output
    overlapping another member's outputs or any input)."""
    n = len(N)
    ins = _member_rows(inputs, n, M * K, torch.bfloat16, list(N), "inputs")
    outs = _member_rows(outputs, n, K, torch.float32, [x // K if K else 0 for x in N], "outputs")
    n_arr = (ctypes.c_int64 * max(n, 1))(*N)
    st = lib().dpr_reduce_scatter_batch(n, ins, K, M, n_arr, outs,
                                        _MODES[mode], 1.0 / K if scale is None else scale,
                                        int(bool(accumulate)), _stream(stream))
    _check("dpr_reduce_scatter_batch", st)


class Request:
    """A persistent collective (dpr_*_init): the arguments were checked once;
    start() enqueues the prepared kernel.  Keeps the bound tensors alive."""

    def __init__(self, handle: int, keep: tuple):
        self.handle = handle
        self._keep = keep
        self._start = lib().dpr_start

    def start(self, stream=None) -> None:
        st = self._start(self.handle, _stream(stream))
        if st != 0:
            raise DprError("dpr_start", st)

    def close(self):
        if self.handle:
            h, self.handle = self.handle, None
            _check("dpr_request_free", lib().dpr_request_free(h))

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dpr_reduce_scatter_init(inputs, K: int, M: int, N: int, outputs, mode=RING_FP32,
                            scale: float | None = None, accumulate: bool = False) -> Request:
    """A persistent dpr_reduce_scatter (same arguments, without the stream)."""
    chk = N > 0
    ins = _rows(inputs, M * K, torch.bfloat16, N, "inputs", chk)
    outs = _rows(outputs, K, torch.float32, N // K if K else 0, "outputs", chk)
    h = ctypes.c_void_p()
    st = lib().dpr_reduce_scatter_init(ctypes.byref(h), ins, K, M, N, outs, _MODES[mode],
                                       1.0 / K if scale is None else scale, int(bool(accumulate)))
    _check("dpr_reduce_scatter_init", st)
    return Request(h.value, (inputs, outputs))


def dpr_allgather_init(shards, K: int, N: int, outputs) -> Request:
    """A persistent dpr_allgather (same arguments, without the stream)."""
    chk = N > 0
    sh = _rows(shards, K, torch.bfloat16, N // K if K else 0, "shards", chk)
    outs = _rows(outputs, K, torch.bfloat16, N, "outputs", chk)
    h = ctypes.c_void_p()
    _check("dpr_allgather_init", lib().dpr_allgather_init(ctypes.byref(h), sh, K, N, outs))
    return Request(h.value, (shards, outputs))


def dpr_allreduce_init(inputs, K: int, N: int, outputs, mode=RING_FP32,
                       scale: float | None = None) -> Request:
    """A persistent dpr_allreduce (same arguments, without the stream)."""
    chk = N > 0
    ins = _rows(inputs, K, torch.bfloat16, N, "inputs", chk)
    outs = _rows(outputs, K, torch.bfloat16, N, "outputs", chk)
    h = ctypes.c_void_p()
    st = lib().dpr_allreduce_init(ctypes.byref(h), ins, K, N, outs, _MODES[mode],
                                  1.0 / K if scale is None else scale)
    _check("dpr_allreduce_init", st)
    return Request(h.value, (inputs, outputs))


def dpr_set_programmatic_launch(enable: bool) -> bool:
    """Turns programmatic dependent launch on or off (process-wide); returns
    the previous setting."""
    prev = ctypes.c_int()
    _check("dpr_set_programmatic_launch",
           lib().dpr_set_programmatic_launch(int(bool(enable)), ctypes.byref(prev)))
    return bool(prev.value)


def dpr_reduce_scatter_bf16(inputs: Sequence[torch.Tensor], K: int, M: int, N: int,
                            outputs: Sequence[torch.Tensor], mode=RING_FP32,
                            scale: float | None = None, accumulate: bool = False,
                            stream=None) -> None:
    """inputs[m*K + r]: bf16 (N,); outputs[j]: bf16 partition shard (N/K,).
    Either argument may also be one tensor of contiguous rows."""
    chk = N > 0
    ins = _rows(inputs, M * K, torch.bfloat16, N, "inputs", chk)
    outs = _rows(outputs, K, torch.bfloat16, N // K if K else 0, "outputs", chk)
    st = lib().dpr_reduce_scatter_bf16(ins, K, M, N, outs, _MODES[mode],
                                       1.0 / K if scale is None else scale, int(bool(accumulate)),
                                       _stream(stream))
    _check("dpr_reduce_scatter_bf16", st)


def dpr_cast_bf16_to_fp32(inp: torch.Tensor, out: torch.Tensor, stream=None) -> None:
    """out[:n] = fp32(inp[:n]), n = inp.numel()."""
    n = inp.numel()
    _need([inp], 1, torch.bfloat16, n, "in")
    _need([out], 1, torch.float32, n, "out")
    _check("dpr_cast_bf16_to_fp32", lib().dpr_cast_bf16_to_fp32(inp.data_ptr(), out.data_ptr(), n,
                                                                _stream(stream)))


def dpr_allgather(shards: Sequence[torch.Tensor], K: int, N: int,
                  outputs: Sequence[torch.Tensor], stream=None) -> None:
    """shards[j]: bf16 (N/K,); outputs[r]: bf16 (N,).  Either argument may also
    be one tensor of K contiguous rows."""
    chk = N > 0
    sh = _rows(shards, K, torch.bfloat16, N // K if K else 0, "shards", chk)
    outs = _rows(outputs, K, torch.bfloat16, N, "outputs", chk)
    _check("dpr_allgather", lib().dpr_allgather(sh, K, N, outs, _stream(stream)))


def dpr_allgather_batch(shards, K: int, N: Sequence[int], outputs, stream=None) -> None:
    """Member i: shards[i][j] bf16 (N[i]/K,), outputs[i][r] bf16 (N[i],);
    shards may also be one tensor [n, K, >= max N/K], outputs one tensor
    [n, K, >= max N].  The members must be independent (no output overlapping
    another member's outputs or shards)."""
    n = len(N)
    sh = _member_rows(shards, n, K, torch.bfloat16, [x // K if K else 0 for x in N], "shards")
    outs = _member_rows(outputs, n, K, torch.bfloat16, list(N), "outputs")
    n_arr = (ctypes.c_int64 * max(n, 1))(*N)
    _check("dpr_allgather_batch", lib().dpr_allgather_batch(n, sh, K, n_arr, outs, _stream(stream)))


def dpr_allreduce(inputs: Sequence[torch.Tensor], K: int, N: int,
                  outputs: Sequence[torch.Tensor], mode=RING_FP32, scale: float | None = None,
                  stream=None) -> None:
    """inputs[r], outputs[r]: bf16 (N,); outputs may be the inputs (in place).
    Either argument may also be one tensor of K contiguous rows."""
    chk = N > 0
    ins = _rows(inputs, K, torch.bfloat16, N, "inputs", chk)
    outs = _rows(outputs, K, torch.bfloat16, N, "outputs", chk)
    st = lib().dpr_allreduce(ins, K, N, outs, _MODES[mode],
                             1.0 / K if scale is None else scale, _stream(stream))
    _check("dpr_allreduce", st)


class FlattenPlan:
    """Owns a dpr_flatten_plan and keeps its source gradients alive."""

    def __init__(self, handle: int, K: int, bucket_numel: int, srcs: list):
        self.handle = handle
        self.K = K
        self.bucket_numel = bucket_numel
        self._srcs = srcs

    def close(self):
        if self.handle:
            h, self.handle = self.handle, None
            _check("dpr_flatten_plan_destroy", lib().dpr_flatten_plan_destroy(h))

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dpr_flatten_plan_create(srcs: Sequence[Sequence[torch.Tensor]], numel: Sequence[int],
                            offset: Sequence[int], bucket_numel: int, stream=None) -> FlattenPlan:
    """srcs[r][p]: rank r's gradient p (bf16, numel[p] elements, any shape)."""
    K = len(srcs)
    P = len(numel)
    flat = []
    for r in range(K):
        if len(srcs[r]) != P:
            raise ValueError("every rank needs P gradients")
        for p in range(P):
            t = srcs[r][p]
            _need([t], 1, torch.bfloat16, 0, "gradients")
            if t.numel() != numel[p]:
                raise ValueError(f"gradient {p} of rank {r}: {t.numel()} elements, numel says {numel[p]}")
            flat.append(t)
    h = ctypes.c_void_p()
    n_arr = (ctypes.c_int64 * P)(*numel)
    o_arr = (ctypes.c_int64 * P)(*offset)
    st = lib().dpr_flatten_plan_create(ctypes.byref(h), K, P, _ptrs(flat), n_arr, o_arr,
                                       bucket_numel, _stream(stream))
    _check("dpr_flatten_plan_create", st)
    return FlattenPlan(h.value, K, bucket_numel, flat)


def dpr_flatten_bucket(plan: FlattenPlan, dst: Sequence[torch.Tensor], stream=None) -> None:
    """dst[r]: rank r's flat bucket, bf16 (bucket_numel,)."""
    d = _rows(dst, plan.K, torch.bfloat16, plan.bucket_numel, "dst")
    _check("dpr_flatten_bucket", lib().dpr_flatten_bucket(plan.handle, d, _stream(stream)))


def dpr_flatten_plan_destroy(plan: FlattenPlan) -> None:
    plan.close()


class FragmentsPlan(FlattenPlan):
    """Owns a dpr_fragments_plan and keeps its source gradients alive."""

    def close(self):
        if self.handle:
            h, self.handle = self.handle, None
            _check("dpr_fragments_plan_destroy", lib().dpr_fragments_plan_destroy(h))


def _grad_table(srcs: Sequence[Sequence[torch.Tensor]], numel: Sequence[int]) -> list:
    K, P = len(srcs), len(numel)
    flat = []
    for r in range(K):
        if len(srcs[r]) != P:
            raise ValueError("every rank needs P gradients")
        for p in range(P):
            t = srcs[r][p]
            _need([t], 1, torch.bfloat16, 0, "gradients")
            if t.numel() != numel[p]:
                raise ValueError(f"gradient {p} of rank {r}: {t.numel()} elements, numel says {numel[p]}")
            flat.append(t)
    return flat


def dpr_fragments_plan_create(srcs: Sequence[Sequence[torch.Tensor]], numel: Sequence[int],
                              offset: Sequence[int], bucket_numel: int,
                              stream=None) -> FragmentsPlan:
    """srcs[r][p]: rank r's gradient p (bf16, numel[p] elements); the bucket
    layout as for dpr_flatten_plan_create."""
    K, P = len(srcs), len(numel)
    flat = _grad_table(srcs, numel)
    h = ctypes.c_void_p()
    n_arr = (ctypes.c_int64 * max(P, 1))(*numel)
    o_arr = (ctypes.c_int64 * max(P, 1))(*offset)
    st = lib().dpr_fragments_plan_create(ctypes.byref(h), K, P, _ptrs(flat), n_arr, o_arr,
                                         bucket_numel, _stream(stream))
    _check("dpr_fragments_plan_create", st)
    return FragmentsPlan(h.value, K, bucket_numel, flat)


def dpr_reduce_scatter_fragments(plan: FragmentsPlan, outputs: Sequence[torch.Tensor],
                                 mode=RING_FP32, scale: float | None = None,
                                 accumulate: bool = False, stream=None) -> None:
    """outputs[j]: fp32 shard j of the bucket (bucket_numel / K,)."""
    outs = _rows(outputs, plan.K, torch.float32, plan.bucket_numel // plan.K, "outputs")
    st = lib().dpr_reduce_scatter_fragments(plan.handle, outs, _MODES[mode],
                                            1.0 / plan.K if scale is None else scale,
                                            int(bool(accumulate)), _stream(stream))
    _check("dpr_reduce_scatter_fragments", st)


def dpr_reduce_scatter_fragments_batch(plans: Sequence[FragmentsPlan],
                                       outputs: Sequence[Sequence[torch.Tensor]], mode=RING_FP32,
                                       scale: float | None = None, accumulate: bool = False,
                                       stream=None) -> None:
    """Member i: plans[i] with outputs[i][j] fp32 (bucket_numel / K,).  The
    members must be independent (no output overlapping another member's
    outputs or any source gradient)."""
    n = len(plans)
    if len(outputs) != n:
        raise ValueError("plans and outputs need one entry per member")
    flat_out = []
    for i, (pl, outs) in enumerate(zip(plans, outputs)):
        _need(outs, pl.K, torch.float32, pl.bucket_numel // pl.K, f"outputs[{i}]")
        flat_out += list(outs)
    K = plans[0].K if plans else 1
    h = (ctypes.c_void_p * max(n, 1))(*[pl.handle for pl in plans])
    st = lib().dpr_reduce_scatter_fragments_batch(n, h, _ptrs(flat_out), _MODES[mode],
                                                  1.0 / K if scale is None else scale,
                                                  int(bool(accumulate)), _stream(stream))
    _check("dpr_reduce_scatter_fragments_batch", st)


def dpr_fragments_plan_destroy(plan: FragmentsPlan) -> None:
    plan.close()


class CoalescedPlan:
    """Owns a dpr_coalesced_plan and keeps its bound tensors alive."""

    def __init__(self, handle: int, K: int, numel: list, partition_numel: int, tensors: list):
        self.handle = handle
        self.K = K
        self.numel = list(numel)
        self.partition_numel = partition_numel
        self._tensors = tensors

    def close(self):
        if self.handle:
            h, self.handle = self.handle, None
            _check("dpr_coalesced_plan_destroy", lib().dpr_coalesced_plan_destroy(h))

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dpr_coalesced_plan_create(tensors: Sequence[Sequence[torch.Tensor]], numel: Sequence[int],
                              stream=None) -> CoalescedPlan:
    """tensors[r][p]: rank r's tensor of parameter p (bf16, numel[p] elements)."""
    K, P = len(tensors), len(numel)
    flat = []
    for r in range(K):
        if len(tensors[r]) != P:
            raise ValueError("every rank needs P tensors")
        for p in range(P):
            t = tensors[r][p]
            _need([t], 1, torch.bfloat16, 0, "tensors")
            if t.numel() != numel[p]:
                raise ValueError(f"tensor {p} of rank {r}: {t.numel()} elements, numel says {numel[p]}")
            flat.append(t)
    h = ctypes.c_void_p()
    n_arr = (ctypes.c_int64 * max(P, 1))(*numel)
    st = lib().dpr_coalesced_plan_create(ctypes.byref(h), K, P, _ptrs(flat), n_arr, _stream(stream))
    _check("dpr_coalesced_plan_create", st)
    pn = ctypes.c_int64()
    _check("dpr_coalesced_partition_numel", lib().dpr_coalesced_partition_numel(h, ctypes.byref(pn)))
    return CoalescedPlan(h.value, K, numel, pn.value, flat)


def dpr_reduce_scatter_coalesced(plan: CoalescedPlan, outputs: Sequence[torch.Tensor],
                                 mode=RING_FP32, scale: float | None = None,
                                 accumulate: bool = False, stream=None) -> None:
    """outputs[j]: rank j's fp32 partition (plan.partition_numel,)."""
    outs = _rows(outputs, plan.K, torch.float32, plan.partition_numel, "outputs")
    st = lib().dpr_reduce_scatter_coalesced(plan.handle, outs, _MODES[mode],
                                            1.0 / plan.K if scale is None else scale,
                                            int(bool(accumulate)), _stream(stream))
    _check("dpr_reduce_scatter_coalesced", st)


def dpr_allgather_coalesced(plan: CoalescedPlan, shards: Sequence[torch.Tensor],
                            stream=None) -> None:
    """shards[j]: rank j's bf16 partition (plan.partition_numel,); writes the
    plan's bound parameter tensors."""
    sh = _rows(shards, plan.K, torch.bfloat16, plan.partition_numel, "shards")
    _check("dpr_allgather_coalesced", lib().dpr_allgather_coalesced(plan.handle, sh,
                                                                    _stream(stream)))


def dpr_coalesced_plan_destroy(plan: CoalescedPlan) -> None:
    plan.close()


WAIT_PER_BUFFER = 0
WAIT_REDUCTION_STREAM = 1


class BucketPipeline:
    """Owns a dpr_bucket_pipeline.  Each submitted bucket's plan and outputs
    are kept alive in the slot of the physical buffer it used, until a later
    submit reuses that buffer (after which the submitting stream is ordered
    behind the old reduction) or the pipeline is flushed or closed."""

    def __init__(self, K: int, bucket_capacity: int, n_buffers: int = 2,
                 wait_policy: int = WAIT_PER_BUFFER, max_blocks: int = 0):
        h = ctypes.c_void_p()
        _check("dpr_bucket_pipeline_create",
               lib().dpr_bucket_pipeline_create(ctypes.byref(h), K, bucket_capacity, n_buffers,
                                                wait_policy, max_blocks))
        self.handle, self.K = h.value, K
        self._slots = [None] * n_buffers
        self._next = 0

    def submit(self, plan: FlattenPlan, outputs: Sequence[torch.Tensor], mode=RING_FP32,
               scale: float | None = None, accumulate: bool = False, producers=(), stream=None):
        _need(outputs, self.K, torch.float32, plan.bucket_numel // self.K, "outputs")
        prod = [_stream(p) for p in producers]
        parr = (ctypes.c_void_p * max(len(prod), 1))(*prod)
        st = lib().dpr_bucket_pipeline_submit(self.handle, plan.handle, _ptrs(outputs), _MODES[mode],
                                              1.0 / self.K if scale is None else scale,
                                              int(bool(accumulate)), parr, len(prod),
                                              _stream(stream))
        _check("dpr_bucket_pipeline_submit", st)
        if plan.bucket_numel > 0:       # an empty bucket uses no buffer
            self._slots[self._next] = (plan, list(outputs))
            self._next = (self._next + 1) % len(self._slots)

    def reduction_stream(self) -> torch.cuda.ExternalStream:
        """The pipeline's reduction stream, for ordering or timing other work."""
        h = ctypes.c_void_p()
        _check("dpr_bucket_pipeline_stream", lib().dpr_bucket_pipeline_stream(self.handle, ctypes.byref(h)))
        return torch.cuda.ExternalStream(h.value)

    def flush(self, stream=None):
        _check("dpr_bucket_pipeline_flush", lib().dpr_bucket_pipeline_flush(self.handle, _stream(stream)))
        self._slots = [None] * len(self._slots)

    def close(self):
        if self.handle:
            h, self.handle = self.handle, None
            _check("dpr_bucket_pipeline_destroy", lib().dpr_bucket_pipeline_destroy(h))
            self._slots = [None] * len(self._slots)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def dpr_flatten_bucket_noalloc(srcs: Sequence[Sequence[torch.Tensor]], numel: Sequence[int],
                               offset: Sequence[int], bucket_numel: int,
                               dst: Sequence[torch.Tensor], stream=None) -> None:
    """The flat-bucket gather without any device allocation, for callers that
    cannot call cudaMalloc (see include/dpr.h).  Same arguments as
    dpr_flatten_plan_create plus the destinations of dpr_flatten_bucket."""
    K, P = len(srcs), len(numel)
    flat = []
    for r in range(K):
        if len(srcs[r]) != P:
            raise ValueError("every rank needs P gradients")
        for p in range(P):
            t = srcs[r][p]
            _need([t], 1, torch.bfloat16, 0, "gradients")
            if t.numel() != numel[p]:
                raise ValueError(f"gradient {p} of rank {r}: {t.numel()} elements, numel says {numel[p]}")
            flat.append(t)
    _need(dst, K, torch.bfloat16, bucket_numel, "dst")
    n_arr = (ctypes.c_int64 * max(P, 1))(*numel)
    o_arr = (ctypes.c_int64 * max(P, 1))(*offset)
    st = lib().dpr_flatten_bucket_noalloc(K, P, _ptrs(flat), n_arr, o_arr, bucket_numel,
                                          _ptrs(dst), _stream(stream))
    _check("dpr_flatten_bucket_noalloc", st)


def dpr_bucket_assign(numel: Sequence[int], cap: int, pad_to: int = 1):
    """Returns (bucket_of[P], offset[P], bucket_numel[n_buckets])."""
    P = len(numel)
    n_arr = (ctypes.c_int64 * max(P, 1))(*numel)
    b_of = (ctypes.c_int32 * max(P, 1))()
    off = (ctypes.c_int64 * max(P, 1))()
    bn = (ctypes.c_int64 * max(P, 1))()
    nb = ctypes.c_int()
    st = lib().dpr_bucket_assign(n_arr, P, cap, pad_to, b_of, off, bn, ctypes.byref(nb))
    _check("dpr_bucket_assign", st)
    return list(b_of[:P]), list(off[:P]), list(bn[:nb.value])


def dpr_strerror(status: int) -> str:
    return lib().dpr_strerror(status).decode()


def dpr_version() -> str:
    return lib().dpr_version().decode()


ALGO_RING, ALGO_TREE, ALGO_NAIVE = 0, 1, 2
_ALGOS = {"ring": ALGO_RING, "tree": ALGO_TREE, "naive": ALGO_NAIVE,
          ALGO_RING: ALGO_RING, ALGO_TREE: ALGO_TREE, ALGO_NAIVE: ALGO_NAIVE}


def dpr_cost_allreduce(algo, K: int, nbytes: float, alpha: float, beta: float) -> float:
    out = ctypes.c_double()
    _check("dpr_cost_allreduce", lib().dpr_cost_allreduce(_ALGOS[algo], K, nbytes, alpha, beta,
                                                          ctypes.byref(out)))
    return out.value


def dpr_cost_ring_broadcast(K: int, nbytes: float, alpha: float, beta: float, segments: int = 1) -> float:
    out = ctypes.c_double()
    _check("dpr_cost_ring_broadcast", lib().dpr_cost_ring_broadcast(K, nbytes, alpha, beta, segments,
                                                                    ctypes.byref(out)))
    return out.value


def dpr_cost_best_segments(K: int, nbytes: float, alpha: float, beta: float,
                           max_segments: int = 1 << 20):
    s, t = ctypes.c_int64(), ctypes.c_double()
    _check("dpr_cost_best_segments", lib().dpr_cost_best_segments(K, nbytes, alpha, beta, max_segments,
                                                                  ctypes.byref(s), ctypes.byref(t)))
    return s.value, t.value


def dpr_cost_crossover(algo_a, algo_b, K: int, alpha: float, beta: float) -> float:
    out = ctypes.c_double()
    _check("dpr_cost_crossover", lib().dpr_cost_crossover(_ALGOS[algo_a], _ALGOS[algo_b], K, alpha,
                                                          beta, ctypes.byref(out)))
    return out.value


def dpr_cost_dp_speedup(t1: float, K: int, nbytes: float, alpha: float, beta: float) -> float:
    out = ctypes.c_double()
    _check("dpr_cost_dp_speedup", lib().dpr_cost_dp_speedup(t1, K, nbytes, alpha, beta,
                                                            ctypes.byref(out)))
    return out.value
