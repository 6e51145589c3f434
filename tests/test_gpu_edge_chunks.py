"""Long chunks whose length is 8 more than a multiple of 16, with 32-byte
aligned buffers: the reduce-scatter (K = 2, 4, 8, 16, 32) and the out-of-place
all-reduce (K = 2, 4, 8) then take 32-byte accesses, and the 8 elements of
each chunk left outside its 32-byte units (the head of an odd chunk, the tail
of an even one) are summed through a 32-byte window that reaches into the
neighbouring chunk.  That layout starts at 2^22 elements per chunk; shorter
chunks keep 16-byte accesses and are covered by the other parity tests, as is
the in-place all-reduce here, which keeps them at any length.

Every element is compared with the oracle's C ring simulation (bit-exact, NaN
as NaN), for every K, micro-batch count and summation mode the edge kernels
are built for, copy and accumulate; a guard test checks that no byte outside the written regions
changes, so the window's reads of the neighbouring chunk leave no trace."""
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import bf16 as obf
from oracle import ring_c
from tests import gpu_helpers as H
from tests.gpu_helpers import Arena
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu

S_EDGE = (1 << 22) + 8          # S % 16 == 8, at the edge layout's threshold
S_EDGE_LONG = (1 << 22) + 4104  # S % 16 == 8, not a power of two plus 8
assert S_EDGE % 16 == 8 and S_EDGE_LONG % 16 == 8


def _x_dev(K, M, N, seed, dev):
    """M*K seeded bf16 buffers generated on the device, and their host bits."""
    xd = [syn.gauss_bf16(0, N, syn.stream_key(seed, i % K, i // K), 1e-3, 0.01, 100.0,
                         device=dev) for i in range(M * K)]
    return xd, [H.bits(t) for t in xd]


# every (K, M) the reduce-scatter's edge kernels are built for, both modes below
RS_EDGE = [(2, S_EDGE, 1), (2, S_EDGE_LONG, 2), (4, S_EDGE_LONG, 1), (4, S_EDGE, 2),
           (8, S_EDGE, 1), (8, S_EDGE_LONG, 2), (16, S_EDGE, 1), (16, S_EDGE, 2),
           (32, S_EDGE, 1), (32, S_EDGE, 2)]


@pytest.mark.parametrize("K,S,M", RS_EDGE)
@pytest.mark.parametrize("mode", H.MODES)
def test_reduce_scatter_edge_layout(K, S, M, mode):
    dev = H.device()
    N = K * S
    xin, x = _x_dev(K, M, N, 7000 + K + 10 * M + mode, dev)
    init = [obf.to_f32(_x_dev(1, 1, S, 7100 + j, dev)[1][0]).copy() for j in range(K)]
    for acc in (False, True):
        out = [torch.from_numpy(i.copy()).to(dev) for i in init]
        dpr.dpr_reduce_scatter(xin, K, M, N, out, mode=mode, scale=1.0 / K, accumulate=acc)
        want, _ = ring_c.reduce_scatter(x, K, M, mode, 1.0 / K, out_init=init if acc else None)
        torch.cuda.synchronize()
        for j in range(K):
            H.assert_f32_equal(out[j].cpu().numpy(), want[j], f"acc={acc} shard {j}")


@pytest.mark.parametrize("K,S", [(2, S_EDGE), (4, S_EDGE_LONG), (8, S_EDGE)])
@pytest.mark.parametrize("mode", H.MODES)
@pytest.mark.parametrize("in_place", [False, True])
def test_allreduce_edge_layout(K, S, mode, in_place):
    dev = H.device()
    N = K * S
    xin, x = _x_dev(K, 1, N, 7200 + K + mode, dev)
    out = xin if in_place else [torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    dpr.dpr_allreduce(xin, K, N, out, mode=mode, scale=1.0 / K)
    want, _ = ring_c.allreduce(x, K, mode, 1.0 / K)
    torch.cuda.synchronize()
    for r in range(K):
        H.assert_bf16_equal(H.bits(out[r]), want[r], f"replica {r}")


@pytest.mark.parametrize("K", [2, 4])
def test_edge_layout_guards(K):
    """Every buffer in one allocation behind guard gaps: after a reduce-scatter
    (two micro-batches, accumulate) and an all-reduce, only the outputs have
    changed, and they hold the oracle's values."""
    dev = H.device()
    S, M = S_EDGE if K == 2 else S_EDGE_LONG, 2
    N = K * S
    a = Arena()
    ins = [a.add(N, torch.bfloat16) for _ in range(M * K)]
    outs = [a.add(S, torch.float32) for _ in range(K)]
    ar = [a.add(N, torch.bfloat16) for _ in range(K)]
    v = a.build(dev)
    xd, x = _x_dev(K, M, N, 7300 + K, dev)
    init = [obf.to_f32(_x_dev(1, 1, S, 7400 + j, dev)[1][0]) for j in range(K)]
    for i in range(M * K):
        v[ins[i]].copy_(xd[i])
    del xd
    for j in range(K):
        v[outs[j]].copy_(torch.from_numpy(init[j]))
    a.snapshot()
    dpr.dpr_reduce_scatter([v[i] for i in ins], K, M, N, [v[o] for o in outs],
                           mode=H.MODES[1], scale=1.0 / K, accumulate=True)
    dpr.dpr_allreduce([v[i] for i in ins[:K]], K, N, [v[o] for o in ar], mode=H.MODES[0],
                      scale=1.0 / K)
    a.check_untouched([(o, 0, S) for o in outs] + [(o, 0, N) for o in ar])
    want, _ = ring_c.reduce_scatter(x, K, M, H.MODES[1], 1.0 / K, out_init=init)
    for j in range(K):
        H.assert_f32_equal(v[outs[j]].cpu().numpy(), want[j], f"shard {j}")
    want_ar, _ = ring_c.allreduce(x[:K], K, H.MODES[0], 1.0 / K)
    for r in range(K):
        H.assert_bf16_equal(H.bits(v[ar[r]]), want_ar[r], f"replica {r}")
