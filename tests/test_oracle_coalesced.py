"""Pins of the oracle's per-parameter (ZeRO-3 discrete path) reduce-scatter and
all-gather: partition sizes, exact brute force per element in ring order with
zero padding, the AllReduce = ReduceScatter + AllGather identity per parameter,
and replicas identical after the all-gather."""
import random

import numpy as np
import pytest

from oracle import bf16 as obf
from oracle import ring
from tests import exact_fp as X
from tests.test_oracle_ring import _random_bf16


def test_shard_layout():
    sizes, offs, total = ring.shard_layout([4097, 8, 1, 0, 16], 8)
    assert sizes == [513, 1, 1, 0, 2] and offs == [0, 513, 514, 515, 515] and total == 517


@pytest.mark.parametrize("mode", [ring.RING_FP32, ring.HOP_BF16])
@pytest.mark.parametrize("K", [2, 3, 5])
def test_bruteforce_per_element(K, mode):
    rng = random.Random(K * 7 + mode)
    numel = [1, K, 2 * K + 1, 7, 0, 3 * K]
    grads = [[_random_bf16(rng, n, spread=12) for n in numel] for _ in range(K)]
    init = [np.full(ring.shard_layout(numel, K)[2], 0.25, np.float32) for _ in range(K)]
    scale = np.float32(1.0 / K)
    parts = ring.reduce_scatter_coalesced(grads, numel, K, mode, float(scale), out_init=init)
    sizes, offs, _ = ring.shard_layout(numel, K)
    R = X.f32 if mode == ring.RING_FP32 else X.bf16
    for p, (n, s, o) in enumerate(zip(numel, sizes, offs)):
        for j in range(K):
            for t in range(s):
                e = j * s + t

                def x(r):
                    return X.of_bf16_bits(grads[r][p][e]) if e < n else X.Fraction(0)
                acc = x(j)
                for k in range(1, K):
                    acc = R(X.add(acc, x((j + k) % K)))
                want = X.f32(X.of_f32(0.25) + X.f32(acc * X.of_f32(scale)))
                assert X.same(X.of_f32(parts[j][o + t]), want), (p, j, t)


@pytest.mark.parametrize("K", [2, 4, 7])
def test_allgather_coalesced_replicas_and_identity(K):
    rng = random.Random(K)
    numel = [3, 2 * K, 1, 5 * K + 2]
    grads = [[_random_bf16(rng, n, spread=10) for n in numel] for _ in range(K)]
    parts = ring.reduce_scatter_coalesced(grads, numel, K, ring.RING_FP32, 1.0 / K)
    params = ring.allgather_coalesced([obf.from_f32(pj) for pj in parts], numel, K)
    for p, n in enumerate(numel):
        for r in range(1, K):
            assert np.array_equal(params[r][p], params[0][p])
        # per parameter: RS then AG equals the all-reduce of the zero-padded gradient
        s = -(-n // K)
        padded = [np.concatenate([grads[r][p], np.zeros(K * s - n, np.uint16)]) for r in range(K)]
        ar, _ = ring.allreduce(padded, K, ring.RING_FP32, 1.0 / K)
        assert np.array_equal(params[0][p], ar[0][:n])
        assert len(params[0][p]) == n
