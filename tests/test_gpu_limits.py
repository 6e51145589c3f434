"""Sizes past 32-bit element offsets: chunks of 2**32 elements, and a flat
gradient and a per-parameter shard longer than 2**31 elements.  Every index of
the kernels and the host checks must be 64-bit.

Results are compared with the oracle at sampled positions on both sides of the
2**31 and 2**32 boundaries.  Where the result is fixed by an invariant
(replicas identical, copies equal to their source), it is checked in full on
the device.
"""
import gc

import numpy as np
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import ring
from tests import gpu_helpers as H
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu

SIGMA = 1e-3


def _need_gib(g):
    gc.collect()
    torch.cuda.empty_cache()
    free, _ = torch.cuda.mem_get_info()
    if free / 2 ** 30 < g:
        pytest.skip(f"needs {g} GiB free on the device")


def _edges(S, seed):
    t = {0, 1, 15, 16, 17}
    for b in (1 << 31, 1 << 32):
        t |= {b - 17, b - 16, b - 1, b, b + 1, b + 16}
    t |= {S - 17, S - 16, S - 1}
    rng = np.random.default_rng(seed)
    t |= set(int(v) for v in rng.integers(0, S, 32))
    return np.array(sorted(v for v in t if 0 <= v < S), dtype=np.int64)


def test_flat_collectives_with_2_pow_32_element_chunks():
    """K=2, N=2**33 bf16 per rank: each chunk is 2**32 elements long."""
    dev = H.device()
    _need_gib(66)
    K, N = 2, 1 << 33
    S = N // K
    keys = [syn.stream_key(0xB16, r) for r in range(K)]
    x = [syn.gauss_bf16(0, N, keys[r], SIGMA, device=dev) for r in range(K)]
    T = _edges(S, 1)
    idx = H.chunk_positions(K, S, T)
    xh = [H.bits(syn.gauss_bf16_at(idx, keys[r], SIGMA)) for r in range(K)]
    idx_d = torch.as_tensor(idx, device=dev)
    T_d = torch.as_tensor(T, device=dev)
    for r in range(K):     # the device inputs are the generator's values
        H.assert_bf16_equal(H.bits(x[r][idx_d]), xh[r], f"input {r}")

    out = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
    for mode in H.MODES:
        dpr.dpr_reduce_scatter(x, K, 1, N, out, mode=mode, scale=0.5)
        want, _ = ring.reduce_scatter(xh, K, 1, mode, 0.5)
        for j in range(K):
            H.assert_f32_equal(out[j][T_d].cpu().numpy(), want[j], f"mode {mode} shard {j}")
    del out
    torch.cuda.empty_cache()

    y = [torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    dpr.dpr_allreduce(x, K, N, y, mode=ring.RING_FP32, scale=0.5)
    want, _ = ring.allreduce(xh, K, ring.RING_FP32, 0.5)
    for r in range(K):
        H.assert_bf16_equal(H.bits(y[r][idx_d]), want[r], f"allreduce replica {r}")
    assert torch.equal(y[0].view(torch.int16), y[1].view(torch.int16))

    shards = [x[j][:S] for j in range(K)]
    dpr.dpr_allgather(shards, K, N, y)
    torch.cuda.synchronize()
    for r in range(K):
        for j in range(K):
            assert torch.equal(y[r][j * S:(j + 1) * S].view(torch.int16),
                               shards[j].view(torch.int16)), (r, j)
    del x, y, shards
    torch.cuda.empty_cache()


def test_flatten_of_a_gradient_longer_than_2_pow_32():
    dev = H.device()
    _need_gib(36)
    K, n, off = 2, (1 << 32) + 24, 8
    bucket = off + n + 8
    src = [syn.gauss_bf16(0, n, syn.stream_key(0xF1A, r), SIGMA, device=dev) for r in range(K)]
    dst = [torch.full((bucket,), 0x3C3C, dtype=torch.int16, device=dev).view(torch.bfloat16)
           for _ in range(K)]
    with dpr.dpr_flatten_plan_create([[s] for s in src], [n], [off], bucket) as plan:
        dpr.dpr_flatten_bucket(plan, dst)
        torch.cuda.synchronize()
    for r in range(K):
        assert torch.equal(dst[r][off:off + n].view(torch.int16), src[r].view(torch.int16))
        head = dst[r][:off].view(torch.int16).cpu().numpy()
        tail = dst[r][off + n:].view(torch.int16).cpu().numpy()
        assert np.all(head == 0x3C3C) and np.all(tail == 0x3C3C)
    del src, dst
    torch.cuda.empty_cache()


def test_per_parameter_shards_longer_than_2_pow_31():
    """One parameter of 2**32 + 41 elements at K=2 (shard 2**31 + 21, not a
    multiple of 16, so every tile takes the element-wise path; the last shard
    ends in one element of zero padding) and a small one after it."""
    dev = H.device()
    _need_gib(40)
    K = 2
    numel = [(1 << 32) + 41, 1000]
    s0 = (numel[0] + K - 1) // K
    keys = [[syn.stream_key(0xC0A, r, 0, p) for p in range(2)] for r in range(K)]
    grads = [[syn.gauss_bf16(0, numel[p], keys[r][p], SIGMA, device=dev) for p in range(2)]
             for r in range(K)]
    T = _edges(s0, 2)
    T_d = torch.as_tensor(T, device=dev)

    def at(r, _m, idx):
        idx = np.asarray(idx, dtype=np.int64)
        out = torch.zeros(len(idx), dtype=torch.bfloat16)
        ok = np.flatnonzero(idx < numel[0])
        out[torch.from_numpy(ok)] = syn.gauss_bf16_at(idx[ok], keys[r][0], SIGMA)
        return out

    with dpr.dpr_coalesced_plan_create(grads, numel) as plan:
        L = plan.partition_numel
        assert L == s0 + numel[1] // K
        part = [torch.empty(L, dtype=torch.float32, device=dev) for _ in range(K)]
        dpr.dpr_reduce_scatter_coalesced(plan, part, mode=ring.RING_FP32, scale=0.5)
        want = H.oracle_rs_sampled(at, K, 1, s0, T, ring.RING_FP32, 0.5)
        for j in range(K):
            H.assert_f32_equal(part[j][T_d].cpu().numpy(), want[j], f"partition {j}")
        del part
        torch.cuda.empty_cache()

        shards = [syn.uniform_bf16(0, L, syn.stream_key(0xC0B, j), 0.02, device=dev)
                  for j in range(K)]
        for r in range(K):
            for p in range(2):
                grads[r][p].zero_()
        dpr.dpr_allgather_coalesced(plan, shards)
        torch.cuda.synchronize()
        s1 = numel[1] // K
        for r in range(K):
            for j in range(K):
                n0 = min(s0, numel[0] - j * s0)
                assert torch.equal(grads[r][0][j * s0:j * s0 + n0].view(torch.int16),
                                   shards[j][:n0].view(torch.int16)), (r, j)
                assert torch.equal(grads[r][1][j * s1:(j + 1) * s1].view(torch.int16),
                                   shards[j][s0:s0 + s1].view(torch.int16)), (r, j)
    del grads, shards
    torch.cuda.empty_cache()
