"""Guard bytes around every buffer of a call.

All buffers of one call live in one device allocation, each behind a gap of
guard bytes and at a chosen distance from 256-byte alignment, so that every
layout runs: 32-byte vectors, 16-byte vectors and the element-wise kernels,
with chunk lengths that leave ragged tails (the 32-byte kernels with an
8-element edge unit per chunk need chunks of 2^22 elements and more; they
have a test of their own below).  After the call, every byte outside
the regions the call may write is compared with its value before the call:
- the guard gaps (no write before or after a buffer);
- the inputs (never written);
- the positions of a flat bucket that no gradient covers.
The written regions are compared with the oracle, bit for bit.
"""
import numpy as np
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import bf16 as obf
from oracle import flatten as ofl
from oracle import ring
from tests import gpu_helpers as H
from tests.gpu_helpers import PAT, Arena
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


def _bf16_data(n, seed):
    return syn.bf16_bits(syn.gauss_bf16(0, n, syn.stream_key(seed, 1), 1e-2, 0.01, 100.0))


def _put_bf16(view, bits):
    view.copy_(syn.bits_to_bf16(bits).to(view.device))


# (chunk length S, shift of the bf16 buffers in bytes, shift of fp32 buffers in bytes)
LAYOUTS = {
    "v32": (528, 0, 0),          # 32-byte vectors
    "v16_len": (536, 0, 0),      # S % 16 == 8: 16-byte vectors
    "v16_addr": (528, 16, 16),   # 16-byte but not 32-byte aligned
    "scalar_len": (531, 0, 0),   # odd S: element-wise
    "scalar_addr": (528, 2, 4),  # 2-byte aligned bf16: element-wise
}


@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("K", [8, 5])
@pytest.mark.parametrize("mode", H.MODES)
def test_reduce_scatter_guards(layout, K, mode):
    dev = H.device()
    S, sb, sf = LAYOUTS[layout]
    N, M = K * S, 2
    a = Arena()
    ins = [a.add(N, torch.bfloat16, sb) for _ in range(M * K)]
    outs = [a.add(S, torch.float32, sf) for _ in range(K)]
    v = a.build(dev)
    x = [_bf16_data(N, 100 * K + i) for i in range(M * K)]
    init = [obf.to_f32(_bf16_data(S, 900 + j)) for j in range(K)]
    for i in range(M * K):
        _put_bf16(v[ins[i]], x[i])
    for j in range(K):
        v[outs[j]].copy_(torch.from_numpy(init[j]))
    a.snapshot()
    dpr.dpr_reduce_scatter([v[i] for i in ins], K, M, N, [v[o] for o in outs], mode=mode,
                           scale=1.0 / K, accumulate=True)
    a.check_untouched([(o, 0, S) for o in outs])
    want, _ = ring.reduce_scatter(x, K, M, mode, 1.0 / K, out_init=init)
    for j in range(K):
        H.assert_f32_equal(v[outs[j]].cpu().numpy(), want[j], f"shard {j}")


@pytest.mark.parametrize("layout", list(LAYOUTS))
def test_reduce_scatter_bf16_partition_guards(layout):
    dev = H.device()
    K, M = 8, 1
    S, sb, _ = LAYOUTS[layout]
    N = K * S
    a = Arena()
    ins = [a.add(N, torch.bfloat16, sb) for _ in range(K)]
    outs = [a.add(S, torch.bfloat16, sb) for _ in range(K)]
    v = a.build(dev)
    x = [_bf16_data(N, 300 + i) for i in range(K)]
    init = [_bf16_data(S, 400 + j) for j in range(K)]
    for i in range(K):
        _put_bf16(v[ins[i]], x[i])
    for j in range(K):
        _put_bf16(v[outs[j]], init[j])
    a.snapshot()
    dpr.dpr_reduce_scatter_bf16([v[i] for i in ins], K, M, N, [v[o] for o in outs],
                                mode=ring.HOP_BF16, scale=1.0 / K, accumulate=True)
    a.check_untouched([(o, 0, S) for o in outs])
    want, _ = ring.reduce_scatter_bf16(x, K, M, ring.HOP_BF16, 1.0 / K, out_init=init)
    for j in range(K):
        H.assert_bf16_equal(H.bits(v[outs[j]]), want[j], f"shard {j}")


@pytest.mark.parametrize("n,sb,sf", [(1600, 0, 0), (1607, 0, 0), (1600, 2, 4), (1600, 16, 16)])
def test_cast_guards(n, sb, sf):
    dev = H.device()
    a = Arena()
    i = a.add(n, torch.bfloat16, sb)
    o = a.add(n, torch.float32, sf)
    v = a.build(dev)
    x = _bf16_data(n, 77)
    _put_bf16(v[i], x)
    a.snapshot()
    dpr.dpr_cast_bf16_to_fp32(v[i], v[o])
    a.check_untouched([(o, 0, n)])
    H.assert_f32_equal(v[o].cpu().numpy(), ring.cast_partition(x), "cast")


@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("in_place", [False, True])
def test_allgather_guards(layout, in_place):
    dev = H.device()
    K = 8
    S, sb, _ = LAYOUTS[layout]
    N = K * S
    a = Arena()
    outs = [a.add(N, torch.bfloat16, sb) for _ in range(K)]
    shards_idx = [] if in_place else [a.add(S, torch.bfloat16, sb) for _ in range(K)]
    v = a.build(dev)
    sh = [_bf16_data(S, 500 + j) for j in range(K)]
    if in_place:
        shards = [v[outs[j]][j * S:(j + 1) * S] for j in range(K)]
    else:
        shards = [v[s] for s in shards_idx]
    for j in range(K):
        _put_bf16(shards[j], sh[j])
    a.snapshot()
    dpr.dpr_allgather(shards, K, N, [v[o] for o in outs])
    a.check_untouched([(o, 0, N) for o in outs])
    want, _ = ring.allgather(sh, K)
    for r in range(K):
        H.assert_bf16_equal(H.bits(v[outs[r]]), want[r], f"replica {r}")


@pytest.mark.parametrize("layout", list(LAYOUTS))
@pytest.mark.parametrize("in_place", [False, True])
def test_allreduce_guards(layout, in_place):
    dev = H.device()
    K = 8
    S, sb, _ = LAYOUTS[layout]
    N = K * S
    a = Arena()
    ins = [a.add(N, torch.bfloat16, sb) for _ in range(K)]
    outs = ins if in_place else [a.add(N, torch.bfloat16, sb) for _ in range(K)]
    v = a.build(dev)
    x = [_bf16_data(N, 600 + r) for r in range(K)]
    for r in range(K):
        _put_bf16(v[ins[r]], x[r])
    a.snapshot()
    dpr.dpr_allreduce([v[i] for i in ins], K, N, [v[o] for o in outs], mode=ring.RING_FP32,
                      scale=1.0 / K)
    a.check_untouched([(o, 0, N) for o in outs])
    want, _ = ring.allreduce(x, K, ring.RING_FP32, 1.0 / K)
    for r in range(K):
        H.assert_bf16_equal(H.bits(v[outs[r]]), want[r], f"replica {r}")


# gradients of odd and tile-crossing sizes, placed in the bucket with gaps
FLAT_NUMEL = [1, 4095, 4096, 4097, 9000, 17, 8192]
FLAT_GAPS = [3, 0, 5, 16, 1, 0, 2, 7]


def _flat_layout():
    offset, at = [], 0
    for n, g in zip(FLAT_NUMEL, FLAT_GAPS):
        at += g
        offset.append(at)
        at += n
    return offset, at + FLAT_GAPS[-1]


@pytest.mark.parametrize("shift", [0, 2, 16])
@pytest.mark.parametrize("noalloc", [False, True])
def test_flatten_guards(shift, noalloc):
    dev = H.device()
    K = 3
    P = len(FLAT_NUMEL)
    offset, bucket = _flat_layout()
    a = Arena()
    src = [[a.add(FLAT_NUMEL[p], torch.bfloat16, shift if p % 2 else 0) for p in range(P)]
           for _ in range(K)]
    dst = [a.add(bucket, torch.bfloat16, shift) for _ in range(K)]
    v = a.build(dev)
    g = [[_bf16_data(FLAT_NUMEL[p], 700 + 10 * r + p) for p in range(P)] for r in range(K)]
    for r in range(K):
        for p in range(P):
            _put_bf16(v[src[r][p]], g[r][p])
    a.snapshot()
    srcs = [[v[src[r][p]] for p in range(P)] for r in range(K)]
    dsts = [v[d] for d in dst]
    if noalloc:
        dpr.dpr_flatten_bucket_noalloc(srcs, FLAT_NUMEL, offset, bucket, dsts)
    else:
        with dpr.dpr_flatten_plan_create(srcs, FLAT_NUMEL, offset, bucket) as plan:
            dpr.dpr_flatten_bucket(plan, dsts)
    a.check_untouched([(dst[r], offset[p], FLAT_NUMEL[p]) for r in range(K) for p in range(P)])
    pat = np.full(bucket, (PAT << 8) | PAT, np.uint16)
    want = ofl.flatten_bucket(g, FLAT_NUMEL, offset, bucket, dst_init=[pat] * K)
    for r in range(K):
        H.assert_bf16_equal(H.bits(v[dst[r]]), want[r], f"bucket {r}")
