"""C-ABI checks that need no GPU: the library builds and loads, exports every
function include/dpr.h declares, rejects bad arguments on the host before
anything reaches CUDA, and its host-only bucket formation matches the oracle.

Rejection tests pass fake device addresses: a rejected call returns before
any CUDA call, so those addresses are never dereferenced."""
import ctypes
import os
import random
import re

import pytest

from oracle import flatten as ofl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dpr.h")

OK, INVALID, ALIGN, UNSUP, CUDA, ALIAS = range(6)


@pytest.fixture(scope="module")
def L():
    from gradient_reduction_gb300 import build
    build.build()
    import gradient_reduction_gb300 as g
    return g.lib()


def _declared():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dpr_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_function(L):
    names = _declared()
    assert len(names) == 40
    for n in names:
        assert hasattr(L, n), n


def test_header_is_plain_c():
    """The header compiles as C (no torch or CUDA types in the signatures)."""
    import subprocess
    import tempfile
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "t.c")
        with open(c, "w") as f:
            f.write('#include "dpr.h"\nint main(void){return dpr_version()==0;}\n')
        r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-fsyntax-only",
                            "-I", os.path.join(ROOT, "include"), c], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr


def _arr(vals):
    return (ctypes.c_void_p * len(vals))(*vals)


BASE = 0x7F0000000000   # fake, 256-byte aligned device addresses; never dereferenced


def _bufs(n, size, start=BASE):
    return [start + i * size for i in range(n)]


def test_reduce_scatter_rejections(L):
    K, N = 4, 64
    ins, outs = _bufs(K, 1 << 20), _bufs(K, 1 << 20, BASE + (1 << 30))
    rs = L.dpr_reduce_scatter
    assert rs(_arr(ins), 1, 1, N, _arr(outs), 0, 1.0, 0, None) == INVALID      # K < 2
    assert rs(_arr(ins), 65, 1, N, _arr(outs), 0, 1.0, 0, None) == INVALID     # K > 64
    assert rs(_arr(ins), K, 3, N, _arr(outs), 0, 1.0, 0, None) == INVALID      # M > 2
    assert rs(_arr(ins), K, 1, N + 1, _arr(outs), 0, 1.0, 0, None) == INVALID  # N % K
    assert rs(_arr(ins), K, 1, -4, _arr(outs), 0, 1.0, 0, None) == INVALID
    assert rs(_arr(ins), K, 1, 1 << 36, _arr(outs), 0, 1.0, 0, None) == UNSUP
    assert rs(_arr(ins), K, 1, N, _arr(outs), 7, 1.0, 0, None) == INVALID      # mode
    assert rs(None, K, 1, N, _arr(outs), 0, 1.0, 0, None) == INVALID
    assert rs(_arr(ins[:3] + [0]), K, 1, N, _arr(outs), 0, 1.0, 0, None) == INVALID
    assert rs(_arr(ins[:3] + [ins[3] + 1]), K, 1, N, _arr(outs), 0, 1.0, 0, None) == ALIGN
    assert rs(_arr(ins), K, 1, N, _arr(outs[:3] + [outs[3] + 2]), 0, 1.0, 0, None) == ALIGN
    # outputs overlapping each other / an input
    assert rs(_arr(ins), K, 1, N, _arr(outs[:3] + [outs[2] + 8]), 0, 1.0, 0, None) == ALIAS
    assert rs(_arr(ins), K, 1, N, _arr(outs[:3] + [ins[1] + 16]), 0, 1.0, 0, None) == ALIAS
    # N == 0 is a no-op that touches nothing
    assert rs(None, K, 1, 0, None, 0, 1.0, 0, None) == OK


def test_allgather_rejections(L):
    K, N = 4, 64
    S = N // K
    sh, outs = _bufs(K, 1 << 20), _bufs(K, 1 << 20, BASE + (1 << 30))
    ag = L.dpr_allgather
    assert ag(_arr(sh), K, N + 2, _arr(outs), None) == INVALID
    assert ag(_arr(sh), K, N, _arr(outs[:3] + [outs[3] + 1]), None) == ALIGN
    assert ag(_arr(sh), K, N, _arr(outs[:3] + [outs[2] + 2 * N - 2]), None) == ALIAS
    # a shard inside some other rank's output
    assert ag(_arr(sh[:1] + [outs[0] + 2] + sh[2:]), K, N, _arr(outs), None) == ALIAS
    # shard j inside out[j] but not at j*S is not the in-place form
    assert ag(_arr(sh[:2] + [outs[2]] + sh[3:]), K, N, _arr(outs), None) == ALIAS


def test_allreduce_rejections(L):
    K, N = 4, 64
    ins, outs = _bufs(K, 1 << 20), _bufs(K, 1 << 20, BASE + (1 << 30))
    ar = L.dpr_allreduce
    assert ar(_arr(ins), K, N, _arr(outs), 2, 1.0, None) == INVALID
    # in[1] == out[0]: in-place is only allowed rank by rank
    assert ar(_arr(ins), K, N, _arr([ins[1]] + outs[1:]), 0, 1.0, None) == ALIAS
    assert ar(_arr(ins), K, N, _arr(outs[:2] + [outs[1]] + outs[3:]), 0, 1.0, None) == ALIAS


def test_flatten_plan_rejections(L):
    h = ctypes.c_void_p()
    src = _arr(_bufs(2, 1 << 20))
    n = (ctypes.c_int64 * 2)(8, 8)
    o_bad = (ctypes.c_int64 * 2)(0, 4)        # spans overlap
    assert L.dpr_flatten_plan_create(ctypes.byref(h), 1, 2, src, n, o_bad, 16, None) == ALIAS
    o_oob = (ctypes.c_int64 * 2)(0, 12)       # second span leaves the bucket
    assert L.dpr_flatten_plan_create(ctypes.byref(h), 1, 2, src, n, o_oob, 16, None) == INVALID
    o = (ctypes.c_int64 * 2)(0, 8)
    odd = _arr([BASE, BASE + (1 << 20) + 1])
    assert L.dpr_flatten_plan_create(ctypes.byref(h), 1, 2, odd, n, o, 16, None) == ALIGN
    assert h.value is None
    assert L.dpr_flatten_plan_destroy(None) == OK
    assert L.dpr_flatten_bucket(None, None, None) == INVALID


def test_strerror_and_version(L):
    import gradient_reduction_gb300 as g
    assert g.dpr_strerror(ALIAS) == "buffers overlap"
    assert "sm_103a" in g.dpr_version()
    assert L.dpr_last_cuda_error() == 0


@pytest.mark.parametrize("seed", range(20))
def test_bucket_assign_matches_oracle(L, seed):
    import gradient_reduction_gb300 as g
    rng = random.Random(seed)
    numel = [rng.choice([1, 3, 8, 100, 4096, 70000]) for _ in range(rng.randint(1, 80))]
    cap = rng.choice([1, 64, 5000, 100000])
    pad = rng.choice([1, 2, 8, 64])
    b_of, off, bn = g.dpr_bucket_assign(numel, cap, pad)
    ref = ofl.assign_buckets(numel, cap, pad)
    assert bn == [b.numel for b in ref]
    for bi, b in enumerate(ref):
        for p, o in zip(b.params, b.offsets):
            assert b_of[p] == bi and off[p] == o


def test_bucket_assign_config3(L):
    import gradient_reduction_gb300 as g
    from workloads import configs as C
    numel = [n for *_, n in C.CFG3.arrival_order()]
    _, _, bn = g.dpr_bucket_assign(numel, C.CFG3.bucket_cap, 8)
    assert bn == [b.numel for b in ofl.assign_buckets(numel, C.CFG3.bucket_cap, 8)]
    assert len(bn) == 42


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    from gradient_reduction_gb300 import _binding
    monkeypatch.setattr(_binding, "_lib", None)
    monkeypatch.setattr(_binding, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _binding.lib()


def test_coalesced_rejections(L):
    h = ctypes.c_void_p()
    n = (ctypes.c_int64 * 2)(64, 64)
    t = _arr(_bufs(4, 1 << 20))
    assert L.dpr_coalesced_plan_create(ctypes.byref(h), 1, 2, t, n, None) == INVALID     # K < 2
    over = _arr([BASE, BASE + 64, BASE + (1 << 20), BASE + (2 << 20)])                   # tensors overlap
    assert L.dpr_coalesced_plan_create(ctypes.byref(h), 2, 2, over, n, None) == ALIAS
    odd = _arr([BASE + 1, BASE + (1 << 20), BASE + (2 << 20), BASE + (3 << 20)])
    assert L.dpr_coalesced_plan_create(ctypes.byref(h), 2, 2, odd, n, None) == ALIGN
    assert h.value is None
    assert L.dpr_reduce_scatter_coalesced(None, None, 0, 1.0, 0, None) == INVALID
    assert L.dpr_allgather_coalesced(None, None, None) == INVALID
    assert L.dpr_coalesced_plan_destroy(None) == OK


def test_pipeline_rejections(L):
    h = ctypes.c_void_p()
    assert L.dpr_bucket_pipeline_create(ctypes.byref(h), 1, 1024, 2, 0, 0) == INVALID   # K < 2
    assert L.dpr_bucket_pipeline_create(ctypes.byref(h), 4, 1024, 0, 0, 0) == INVALID   # no buffers
    assert L.dpr_bucket_pipeline_create(ctypes.byref(h), 4, 1024, 2, 9, 0) == INVALID   # policy
    assert L.dpr_bucket_pipeline_create(ctypes.byref(h), 4, 0, 2, 0, 0) == INVALID      # capacity
    assert L.dpr_bucket_pipeline_create(ctypes.byref(h), 4, 1024, 2, 0, -1) == INVALID  # budget
    assert h.value is None
    assert L.dpr_bucket_pipeline_submit(None, None, None, 0, 1.0, 0, None, 0, None) == INVALID
    assert L.dpr_bucket_pipeline_flush(None, None) == INVALID
    assert L.dpr_bucket_pipeline_destroy(None) == OK


def test_bf16_partition_rejections(L):
    K, N = 4, 64
    ins, outs = _bufs(K, 1 << 20), _bufs(K, 1 << 20, BASE + (1 << 30))
    rs = L.dpr_reduce_scatter_bf16
    assert rs(_arr(ins), K, 1, N + 1, _arr(outs), 0, 1.0, 0, None) == INVALID
    assert rs(_arr(ins), K, 1, N, _arr(outs[:3] + [outs[3] + 1]), 0, 1.0, 0, None) == ALIGN
    assert rs(_arr(ins), K, 1, N, _arr(outs[:3] + [ins[0]]), 0, 1.0, 0, None) == ALIAS
    c = L.dpr_cast_bf16_to_fp32
    assert c(ctypes.c_void_p(BASE), ctypes.c_void_p(BASE + 2), 16, None) == ALIGN
    assert c(ctypes.c_void_p(BASE), ctypes.c_void_p(BASE + 16), 16, None) == ALIAS
    assert c(None, None, 0, None) == OK
    assert c(ctypes.c_void_p(BASE), ctypes.c_void_p(BASE + 4096), -1, None) == INVALID


def test_coalesced_plan_refuses_more_tiles_than_a_grid_holds(L):
    """1000 parameters of 2^34 elements at K=64 need about 4.2e9 reduce-scatter
    tiles of 4096 elements, more than a 1-D grid holds: refused on the host
    (fake, non-overlapping addresses; nothing is dereferenced or allocated)."""
    K, P = 64, 1000
    n = 1 << 34
    numel = (ctypes.c_int64 * P)(*([n] * P))
    t = _arr([BASE + i * (1 << 35) for i in range(K * P)])
    h = ctypes.c_void_p()
    assert L.dpr_coalesced_plan_create(ctypes.byref(h), K, P, t, numel, None) == UNSUP
    assert h.value is None


def test_binding_refuses_host_tensors_before_touching_the_library():
    """The Python binding checks tensors first: host (CPU) tensors, wrong
    dtypes and short tensors are refused with ValueError, with no CUDA call."""
    import torch
    import gradient_reduction_gb300 as dpr
    x = [torch.zeros(64, dtype=torch.bfloat16) for _ in range(4)]
    out = [torch.zeros(16, dtype=torch.float32) for _ in range(4)]
    for call in (lambda: dpr.dpr_reduce_scatter(x, 4, 1, 64, out),
                 lambda: dpr.dpr_allgather([t[:16] for t in x], 4, 64, x),
                 lambda: dpr.dpr_allreduce(x, 4, 64, x),
                 lambda: dpr.dpr_cast_bf16_to_fp32(x[0], out[0]),
                 lambda: dpr.dpr_flatten_plan_create([[t] for t in x], [64], [0], 64),
                 lambda: dpr.dpr_coalesced_plan_create([[t] for t in x], [64])):
        with pytest.raises(ValueError):
            call()


def test_fragments_plan_rejections(L):
    """Host-side checks of the fused gather + reduce-scatter plan; the fake
    addresses are never dereferenced (every case is refused before any CUDA
    call)."""
    h = ctypes.c_void_p()
    c = L.dpr_fragments_plan_create
    K, P = 2, 2
    src = _arr([BASE, BASE + (1 << 20), BASE + (2 << 20), BASE + (3 << 20)])
    n = (ctypes.c_int64 * P)(16, 16)
    off = (ctypes.c_int64 * P)(0, 16)
    assert c(ctypes.byref(h), 1, P, src, n, off, 32, None) == INVALID          # K < 2
    assert c(ctypes.byref(h), K, P, src, n, off, 33, None) == INVALID          # bucket % K
    assert c(ctypes.byref(h), K, P, src, n, off, 24, None) == INVALID          # span past the bucket
    assert c(ctypes.byref(h), K, P, src, n, (ctypes.c_int64 * P)(0, 8), 32, None) == ALIAS
    odd = _arr([BASE + 1, BASE + (1 << 20), BASE + (2 << 20), BASE + (3 << 20)])
    assert c(ctypes.byref(h), K, P, odd, n, off, 32, None) == ALIGN
    assert c(ctypes.byref(h), K, P, src, n, off, 1 << 40, None) == UNSUP
    assert h.value is None
    assert L.dpr_reduce_scatter_fragments(None, None, 0, 1.0, 0, None) == INVALID
    assert L.dpr_fragments_plan_destroy(None) == OK


def test_reduce_scatter_batch_rejections(L):
    """The batched reduce-scatter checks every member as the single call does,
    and refuses members that are not independent, before any CUDA call."""
    K, M, N = 4, 1, 64
    rs = L.dpr_reduce_scatter_batch
    ins = _bufs(2 * K, 1 << 20)
    outs = _bufs(2 * K, 1 << 20, BASE + (1 << 30))
    n2 = (ctypes.c_int64 * 2)(N, N)
    assert rs(-1, _arr(ins), K, M, n2, _arr(outs), 0, 1.0, 0, None) == INVALID
    assert rs(4097, _arr(ins), K, M, n2, _arr(outs), 0, 1.0, 0, None) == UNSUP
    assert rs(0, None, K, M, None, None, 0, 1.0, 0, None) == OK
    assert rs(2, None, K, M, n2, _arr(outs), 0, 1.0, 0, None) == INVALID
    assert rs(2, _arr(ins), 1, M, n2, _arr(outs), 0, 1.0, 0, None) == INVALID       # K < 2
    assert rs(2, _arr(ins), K, M, (ctypes.c_int64 * 2)(N, N + 1), _arr(outs), 0, 1.0, 0,
              None) == INVALID                                                      # N % K
    bad = outs[:K + 1] + [outs[K + 1] + 2] + outs[K + 2:]
    assert rs(2, _arr(ins), K, M, n2, _arr(bad), 0, 1.0, 0, None) == ALIGN
    # member 1 writes into member 0's output
    clash = outs[:K] + [outs[0] + 16] + outs[K + 1:]
    assert rs(2, _arr(ins), K, M, n2, _arr(clash), 0, 1.0, 0, None) == ALIAS
    # member 1 writes into member 0's input
    into_in = outs[:K] + [ins[2] + 32] + outs[K + 1:]
    assert rs(2, _arr(ins), K, M, n2, _arr(into_in), 0, 1.0, 0, None) == ALIAS
    # member 0 writes into member 1's input
    into_in1 = [ins[K + 3] + 64] + outs[1:]
    assert rs(2, _arr(ins), K, M, n2, _arr(into_in1), 0, 1.0, 0, None) == ALIAS


def test_fragments_batch_and_launch_switch(L):
    b = L.dpr_reduce_scatter_fragments_batch
    assert b(0, None, None, 0, 1.0, 0, None) == OK
    assert b(-1, None, None, 0, 1.0, 0, None) == INVALID
    assert b(4097, None, None, 0, 1.0, 0, None) == UNSUP
    assert b(1, None, None, 0, 1.0, 0, None) == INVALID
    assert b(1, _arr([0]), _arr([BASE]), 0, 1.0, 0, None) == INVALID             # null plan
    prev = ctypes.c_int()
    assert L.dpr_set_programmatic_launch(0, ctypes.byref(prev)) == OK
    assert prev.value == 1
    assert L.dpr_set_programmatic_launch(1, None) == OK
    assert L.dpr_set_programmatic_launch(1, ctypes.byref(prev)) == OK
    assert prev.value == 1


def test_noalloc_records_a_failing_cuda_call():
    """dpr_flatten_bucket_noalloc reports a failing CUDA call as DPR_ERR_CUDA
    and keeps its code for dpr_last_cuda_error(), like every other entry
    point.  Its first CUDA call is the capture-status query of the stream,
    which fails on a machine without a GPU.  A source pointer is null, so on a
    machine with a GPU the call is refused right after that query instead;
    either way nothing is launched.  Run in a child process, so the recorded
    error does not outlive the test."""
    import subprocess
    import sys
    code = r"""
import ctypes, sys
sys.path.insert(0, %r)
import gradient_reduction_gb300 as g
L = g.lib()
src = (ctypes.c_void_p * 2)(0x7F0000000000, 0)
dst = (ctypes.c_void_p * 2)(0x7F0000100000, 0x7F0000200000)
n = (ctypes.c_int64 * 1)(16)
o = (ctypes.c_int64 * 1)(0)
st = L.dpr_flatten_bucket_noalloc(2, 1, src, n, o, 16, dst, None)
print(st, L.dpr_last_cuda_error())
""" % ROOT
    out = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    st, err = map(int, out.stdout.split())
    assert st in (CUDA, INVALID)
    if st == CUDA:
        assert err != 0
    else:
        assert err == 0


def test_allgather_batch_rejections(L):
    K, N = 4, 64
    S = N // K
    ag = L.dpr_allgather_batch
    sh = _bufs(2 * K, 1 << 20)
    outs = _bufs(2 * K, 1 << 20, BASE + (1 << 30))
    n2 = (ctypes.c_int64 * 2)(N, N)
    assert ag(0, None, K, None, None, None) == OK
    assert ag(-1, _arr(sh), K, n2, _arr(outs), None) == INVALID
    assert ag(4097, _arr(sh), K, n2, _arr(outs), None) == UNSUP
    assert ag(2, _arr(sh), 1, n2, _arr(outs), None) == INVALID                 # K < 2
    assert ag(2, _arr(sh), K, (ctypes.c_int64 * 2)(N, N + 1), _arr(outs), None) == INVALID
    # member 1 writes into member 0's output
    assert ag(2, _arr(sh), K, n2, _arr(outs[:K] + [outs[1] + 64] + outs[K + 1:]), None) == ALIAS
    # member 1 writes over member 0's shard
    assert ag(2, _arr(sh), K, n2, _arr(outs[:K] + [sh[0]] + outs[K + 1:]), None) == ALIAS
    # member 0 writes over member 1's shard
    assert ag(2, _arr(sh), K, n2, _arr([sh[K + 2] - 2 * S] + outs[1:]), None) == ALIAS


def test_request_init_rejections(L):
    """Persistent requests check their arguments as the one-shot calls do,
    before any CUDA call; a refused init returns no request."""
    K, N = 4, 64
    ins, outs = _bufs(K, 1 << 20), _bufs(K, 1 << 20, BASE + (1 << 30))
    h = ctypes.c_void_p(123)
    assert L.dpr_reduce_scatter_init(ctypes.byref(h), _arr(ins), 1, 1, N, _arr(outs), 0, 1.0,
                                     0) == INVALID
    assert h.value is None
    assert L.dpr_reduce_scatter_init(ctypes.byref(h), _arr(ins), K, 1, N,
                                     _arr(outs[:3] + [ins[1] + 16]), 0, 1.0, 0) == ALIAS
    assert L.dpr_reduce_scatter_init(None, _arr(ins), K, 1, N, _arr(outs), 0, 1.0, 0) == INVALID
    assert L.dpr_allgather_init(ctypes.byref(h), _arr(ins), K, N + 2, _arr(outs)) == INVALID
    assert L.dpr_allgather_init(ctypes.byref(h), _arr(ins), K, N,
                                _arr(outs[:3] + [outs[3] + 1])) == ALIGN
    assert L.dpr_allreduce_init(ctypes.byref(h), _arr(ins), K, N, _arr(outs), 5, 1.0) == INVALID
    assert h.value is None
    assert L.dpr_start(None, None) == INVALID
    assert L.dpr_request_free(None) == OK
