"""Loader of the C ring simulation, oracle/ring_sim.c (oracle; test
infrastructure).

The C simulation restates the same rounds as `oracle.ring` (see the C file's
header for the pages it follows) in plain C, so that the host's cores run it
faster than numpy: the bench's CPU baseline times it, and the tests check it
against its own pins and against the numpy simulation.  Results use the same
representation as `oracle.ring`: uint16 arrays of bf16 bits, float32 arrays
for fp32 partitions.

build() compiles it with the host C compiler into oracle/_build/ (with OpenMP
when the compiler has it): -O2, no contraction of a*b+c into fused
multiply-adds, no fast-math, so every float operation is one IEEE binary32
operation rounded to nearest even.
"""
from __future__ import annotations

import ctypes
import os
import shutil
import subprocess

import numpy as np

RING_FP32 = 0
HOP_BF16 = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(_HERE, "ring_sim.c")
LIB = os.path.join(_HERE, "_build", "libring_sim.so")
FLAGS = ["-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-Wall", "-Wextra",
         "-fPIC", "-shared"]

_lib = None


def build(force: bool = False) -> str:
    """Compiles ring_sim.c (if the library is missing or older than its source)
    and returns the library's path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        raise RuntimeError("no host C compiler (gcc/cc) to build the C oracle")
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    tmp = LIB + f".{os.getpid()}.tmp"
    r = subprocess.run([cc] + FLAGS + ["-fopenmp", "-o", tmp, SRC], capture_output=True, text=True)
    if r.returncode != 0:          # a compiler without OpenMP: one thread
        r = subprocess.run([cc] + FLAGS + ["-o", tmp, SRC], capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"building the C oracle failed:\n{r.stderr}")
    os.replace(tmp, LIB)
    return LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        pp = ctypes.POINTER(ctypes.c_void_p)
        i64p = ctypes.POINTER(ctypes.c_int64)
        L.oracle_reduce_scatter.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int64, pp,
                                            ctypes.c_int, ctypes.c_float, ctypes.c_int, pp, i64p]
        L.oracle_allgather.argtypes = [ctypes.c_int, ctypes.c_int64, pp, pp, i64p]
        L.oracle_allreduce.argtypes = [ctypes.c_int, ctypes.c_int64, pp, ctypes.c_int,
                                       ctypes.c_float, pp, i64p]
        L.oracle_flatten.argtypes = [ctypes.c_int, ctypes.c_int, pp, i64p, i64p, ctypes.c_int64, pp]
        L.oracle_threads.argtypes = []
        for f in (L.oracle_reduce_scatter, L.oracle_allgather, L.oracle_allreduce,
                  L.oracle_flatten, L.oracle_threads):
            f.restype = ctypes.c_int
        _lib = L
    return _lib


def threads() -> int:
    """Threads the simulation's element loops use."""
    return lib().oracle_threads()


def _arr(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=dtype))


def _ptrs(arrs):
    return (ctypes.c_void_p * max(len(arrs), 1))(*[a.ctypes.data for a in arrs])


def _run(name: str, status: int):
    if status == 1:
        raise ValueError(f"{name}: invalid argument")
    if status != 0:
        raise MemoryError(f"{name}: out of host memory")


class Counters:
    """Rounds run and elements each rank sent, as the simulation counted them."""

    def __init__(self, raw: np.ndarray):
        self.rounds = int(raw[0])
        self.sent = [int(v) for v in raw[1:]]


def reduce_scatter(x: list, K: int, M: int = 1, mode: int = RING_FP32, scale: float = 1.0,
                   out_init: list | None = None):
    """Same arguments and result as oracle.ring.reduce_scatter: x[m*K + r] bf16
    bits of N; returns (K float32 shards of N/K, Counters)."""
    xs = [_arr(a, np.uint16) for a in x]
    if len(xs) != M * K:
        raise ValueError("expected M*K input buffers, x[m*K + r]")
    N = len(xs[0])
    if any(len(a) != N for a in xs):
        raise ValueError("input buffers of different lengths")
    S = N // K if K else 0
    outs = [np.zeros(S, dtype=np.float32) if out_init is None else _arr(out_init[j], np.float32).copy()
            for j in range(K)]
    raw = np.zeros(1 + K, dtype=np.int64)
    _run("reduce_scatter", lib().oracle_reduce_scatter(
        K, M, N, _ptrs(xs), mode, float(np.float32(scale)), int(out_init is not None), _ptrs(outs),
        raw.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))))
    return outs, Counters(raw)


def allgather(shards: list, K: int):
    """Same as oracle.ring.allgather: K bf16 shards of S -> K buffers of K*S."""
    sh = [_arr(a, np.uint16) for a in shards]
    if len(sh) != K or any(len(a) != len(sh[0]) for a in sh):
        raise ValueError("need K shards of equal length")
    S = len(sh[0])
    outs = [np.empty(K * S, dtype=np.uint16) for _ in range(K)]
    raw = np.zeros(1 + K, dtype=np.int64)
    _run("allgather", lib().oracle_allgather(K, S, _ptrs(sh), _ptrs(outs),
                                             raw.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))))
    return outs, Counters(raw)


def allreduce(x: list, K: int, mode: int = RING_FP32, scale: float = 1.0):
    """Same as oracle.ring.allreduce: K bf16 buffers of N -> K bf16 buffers."""
    xs = [_arr(a, np.uint16) for a in x]
    if len(xs) != K:
        raise ValueError("need K input buffers")
    N = len(xs[0])
    if any(len(a) != N for a in xs):
        raise ValueError("input buffers of different lengths")
    outs = [np.empty(N, dtype=np.uint16) for _ in range(K)]
    raw = np.zeros(1 + K, dtype=np.int64)
    _run("allreduce", lib().oracle_allreduce(K, N, _ptrs(xs), mode, float(np.float32(scale)),
                                             _ptrs(outs),
                                             raw.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))))
    return outs, Counters(raw)


def flatten_bucket(src: list, numel: list, offset: list, bucket_numel: int,
                   dst_init: list | None = None) -> list:
    """Same as oracle.flatten.flatten_bucket (without its overlap checks):
    src[r][p] bf16 bits of numel[p] -> K flat buckets."""
    K, P = len(src), len(numel)
    flat = [_arr(src[r][p], np.uint16).reshape(-1) for r in range(K) for p in range(P)]
    for i, a in enumerate(flat):
        if len(a) != numel[i % P]:
            raise ValueError("numel does not match the gradient")
    dst = [np.zeros(bucket_numel, dtype=np.uint16) if dst_init is None
           else _arr(dst_init[r], np.uint16).copy() for r in range(K)]
    n_arr = (ctypes.c_int64 * max(P, 1))(*numel)
    o_arr = (ctypes.c_int64 * max(P, 1))(*offset)
    _run("flatten", lib().oracle_flatten(K, P, _ptrs(flat), n_arr, o_arr, bucket_numel, _ptrs(dst)))
    return dst
