"""Pins of the oracle's bf16 partition path: exact brute force (the shard
rounded once to bf16, add_ rounded once more), the identity with the fp32
reduce-scatter (copy_ == bf16 of the fp32 shard), and the exact cast."""
import random

import numpy as np
import pytest

from oracle import bf16 as obf
from oracle import ring
from tests import exact_fp as X
from tests.test_oracle_ring import _random_bf16


@pytest.mark.parametrize("mode", [ring.RING_FP32, ring.HOP_BF16])
@pytest.mark.parametrize("K", [2, 3, 4, 8])
def test_bruteforce(K, mode):
    rng = random.Random(40 + K + mode)
    S = 5
    N = K * S
    x = [_random_bf16(rng, N, spread=12) for _ in range(2 * K)]
    init = [_random_bf16(rng, S, spread=6) for _ in range(K)]
    scale = np.float32(1.0 / K)
    got, _ = ring.reduce_scatter_bf16(x, K, 2, mode, float(scale), out_init=init)
    R = X.f32 if mode == ring.RING_FP32 else X.bf16
    for j in range(K):
        for t in range(S):
            e = j * S + t

            def g(r):
                return X.bf16(X.of_bf16_bits(x[r][e]) + X.of_bf16_bits(x[K + r][e]))
            acc = g(j)
            for k in range(1, K):
                acc = R(acc + g((j + k) % K))
            shard = X.bf16(X.f32(acc * X.of_f32(scale)))
            want = X.bf16(X.of_bf16_bits(init[j][t]) + shard)
            assert X.same(X.of_bf16_bits(got[j][t]), want), (j, t)


def test_copy_equals_bf16_of_fp32_shard():
    rng = random.Random(3)
    K, S = 8, 9
    x = [_random_bf16(rng, K * S, spread=14) for _ in range(K)]
    for mode in (ring.RING_FP32, ring.HOP_BF16):
        b, _ = ring.reduce_scatter_bf16(x, K, 1, mode, 0.125)
        f, _ = ring.reduce_scatter(x, K, 1, mode, 0.125)
        for j in range(K):
            assert np.array_equal(b[j], obf.from_f32(f[j]))


def test_cast_is_exact_widening():
    bits = np.arange(0, 65536, 7, dtype=np.uint32).astype(np.uint16)
    f = ring.cast_partition(bits)
    finite = ~np.isnan(f)
    assert np.array_equal(obf.from_f32(f)[finite], bits[finite])
    assert np.array_equal(f.view(np.uint32) & 0xFFFF, np.zeros(len(f), np.uint32))
