"""Pins of the C ring simulation (oracle/ring_sim.c) against what the pages and
the mathematics fix -- the worked example's final values, closed forms,
traffic counts, invariants and exact-rational brute force -- and, beyond
those pins, agreement bit for bit with the numpy simulation of the same
rounds on random and special-value inputs."""
import random

import numpy as np
import pytest

from oracle import bf16 as obf
from oracle import flatten as ofl
from oracle import ring
from oracle import ring_c
from tests import exact_fp as X
from tests.test_oracle_ring import _random_bf16, _ring_expected
from workloads import synthetic as syn

MODES = (ring_c.RING_FP32, ring_c.HOP_BF16)


def _int_example(K):
    """x_r[c] = (c + 1) * 2**r, one element per chunk (N = K)."""
    return [syn.bf16_bits(t) for t in syn.integer_example(K, K)]


def _same_bits_f32(a, b):
    """Equal float32 arrays, NaN matching NaN."""
    a, b = np.asarray(a, np.float32), np.asarray(b, np.float32)
    na, nb = np.isnan(a), np.isnan(b)
    return np.array_equal(na, nb) and np.array_equal(a.view(np.uint32)[~na], b.view(np.uint32)[~nb])


def test_builds_and_reports_threads():
    assert ring_c.threads() >= 1


# --- the pages' worked examples ------------------------------------------------------

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("K", [3, 4])
def test_worked_example_final_values(K, mode):
    """Ring All-Reduce illustrated (4 GPUs) and Lecture 14 exercise 3 (K = 3):
    after the reduce-scatter slot j holds a_j + b_j + ... = (2^K - 1)(j + 1);
    after the all-reduce every GPU holds that sum for every chunk; x 1/4 is
    exact for K = 4."""
    x = _int_example(K)
    shards, ctr = ring_c.reduce_scatter(x, K, 1, mode, 1.0)
    for j in range(K):
        assert float(shards[j][0]) == (2 ** K - 1) * (j + 1)
    assert ctr.rounds == K - 1
    outs, ctr = ring_c.allreduce(x, K, mode, 1.0)
    for r in range(K):
        assert list(obf.to_f32(outs[r])) == [float((2 ** K - 1) * (c + 1)) for c in range(K)]
    assert ctr.rounds == 2 * (K - 1)
    if K == 4:
        shards, _ = ring_c.reduce_scatter(x, K, 1, mode, 0.25)
        assert [float(s[0]) for s in shards] == [15 * (j + 1) / 4 for j in range(4)]


# --- closed forms, counters, invariants -------------------------------------------------

@pytest.mark.parametrize("K", [2, 3, 4, 5, 8, 16])
def test_traffic_counters(K):
    """Each device sends 2(K-1) N/K elements in 2(K-1) rounds (lecture section
    3.2, exercise 4; CSDN summary)."""
    N = K * 6
    x = [np.zeros(N, np.uint16) for _ in range(K)]
    _, ctr = ring_c.allreduce(x, K)
    assert ctr.rounds == 2 * (K - 1) and ctr.sent == [2 * (K - 1) * N // K] * K
    _, ctr = ring_c.reduce_scatter(x, K)
    assert ctr.rounds == K - 1 and ctr.sent == [(K - 1) * N // K] * K
    _, ctr = ring_c.allgather([np.zeros(N // K, np.uint16)] * K, K)
    assert ctr.rounds == K - 1 and ctr.sent == [(K - 1) * N // K] * K


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("K", [2, 3, 4, 8, 16, 64])
def test_closed_form_integer_sum(K, mode):
    """Small integers sum exactly in any order: slot j = sum_r x_r over chunk j,
    times 1/K (exact for K a power of two)."""
    rng = np.random.default_rng(100 + K)
    S = 7
    N = K * S
    vals = rng.integers(-7, 8, size=(K, N))
    x = [obf.from_f32(v.astype(np.float32)) for v in vals]
    scale = 1.0 / K if K & (K - 1) == 0 else 1.0
    shards, _ = ring_c.reduce_scatter(x, K, 1, mode, scale)
    total = vals.sum(axis=0)
    for j in range(K):
        assert np.array_equal(shards[j], (total[j * S:(j + 1) * S] * scale).astype(np.float32))


@pytest.mark.parametrize("K", [2, 3, 5, 8])
def test_allgather_replicas_identical_and_concatenated(K):
    """Every replica equals the shards concatenated in order (lecture section
    2.2; Ring illustrated, the end of Phase 2)."""
    rng = np.random.default_rng(K)
    S = 11
    sh = [rng.integers(0, 1 << 16, size=S).astype(np.uint16) for _ in range(K)]
    outs, _ = ring_c.allgather(sh, K)
    want = np.concatenate(sh)
    for r in range(K):
        assert np.array_equal(outs[r], want)


def test_flatten_matches_an_element_loop():
    """dst_r[offset_p + t] = src_{r,p}[t]; uncovered positions keep their value."""
    rng = np.random.default_rng(3)
    K, numel, offset, n = 3, [5, 0, 9, 1], [0, 5, 7, 16], 20
    src = [[rng.integers(0, 1 << 16, size=k).astype(np.uint16) for k in numel] for _ in range(K)]
    init = [np.full(n, 0xABCD, np.uint16) for _ in range(K)]
    got = ring_c.flatten_bucket(src, numel, offset, n, init)
    for r in range(K):
        want = [0xABCD] * n
        for p in range(len(numel)):
            for t in range(numel[p]):
                want[offset[p] + t] = int(src[r][p][t])
        assert got[r].tolist() == want


# --- exact brute force --------------------------------------------------------------

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("K", [2, 3, 4, 5, 8])
def test_bruteforce_exact_rounding(K, mode):
    """Every rounding step against exact rationals rounded to nearest even, in
    ring order (chunk j starts at rank j)."""
    rng = random.Random(2000 + K + 10 * mode)
    S = 6
    N = K * S
    x = [_random_bf16(rng, N, spread=14, zero_frac=0.05) for _ in range(K)]
    scale = np.float32(1.0 / K)
    got, _ = ring_c.reduce_scatter(x, K, 1, mode, float(scale))
    want = _ring_expected(x, K, 1, mode, scale)
    for j in range(K):
        for t in range(S):
            assert X.same(X.of_f32(got[j][t]), want[j][t]), (j, t)


@pytest.mark.parametrize("mode", MODES)
def test_bruteforce_two_microbatches_and_accumulate(mode):
    rng = random.Random(77 + mode)
    K, S = 4, 5
    N = K * S
    x = [_random_bf16(rng, N, spread=10) for _ in range(2 * K)]
    init = [np.asarray([float(np.float32(rng.uniform(-1, 1))) for _ in range(S)], np.float32)
            for _ in range(K)]
    got, _ = ring_c.reduce_scatter(x, K, 2, mode, 0.25, out_init=init)
    want = _ring_expected(x, K, 2, mode, np.float32(0.25), acc_init=init)
    for j in range(K):
        for t in range(S):
            assert X.same(X.of_f32(got[j][t]), want[j][t]), (j, t)


# --- the same rounds as the numpy simulation ---------------------------------------------

CASES = [(K, S, M, mode, acc) for K in (2, 3, 4, 5, 8, 16, 64) for S in (1, 7, 33)
         for M in (1, 2) for mode in MODES for acc in (False, True)]


@pytest.mark.parametrize("K,S,M,mode,acc", CASES)
def test_reduce_scatter_equals_numpy_simulation(K, S, M, mode, acc):
    N = K * S
    key = 9000 + K * 100 + S
    x = [syn.bf16_bits(syn.gauss_bf16(0, N, syn.stream_key(key, r, m), 1e-3))
         for m in range(M) for r in range(K)]
    init = None
    if acc:
        init = [np.random.default_rng(key + j).standard_normal(S).astype(np.float32)
                for j in range(K)]
    a, ca = ring_c.reduce_scatter(x, K, M, mode, 1.0 / K, out_init=init)
    b, cb = ring.reduce_scatter(x, K, M, mode, 1.0 / K, out_init=init)
    for j in range(K):
        assert _same_bits_f32(a[j], b[j]), j
    assert ca.rounds == cb.rounds and ca.sent == cb.sent


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("K", [2, 4, 7, 8, 16])
def test_allreduce_equals_numpy_simulation(K, mode):
    N = K * 29
    x = [syn.bf16_bits(syn.gauss_bf16(0, N, syn.stream_key(31 + K, r, 0), 1e-2)) for r in range(K)]
    a, ca = ring_c.allreduce(x, K, mode, 1.0 / K)
    b, cb = ring.allreduce(x, K, mode, 1.0 / K)
    for r in range(K):
        assert np.array_equal(a[r], b[r]), r
    assert ca.rounds == cb.rounds and ca.sent == cb.sent


@pytest.mark.parametrize("mode", MODES)
def test_special_values_equal_numpy_simulation(mode):
    """NaN, +-Inf, signed zeros, subnormals, the largest finite values."""
    K, S = 4, 64
    N = K * S
    rng = np.random.default_rng(5)
    pool = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x0001, 0x8001, 0x007F, 0x7F7F,
                     0xFF7F, 0x3F80, 0xBF80, 0x0080, 0x4000], np.uint16)
    x = [pool[rng.integers(0, len(pool), size=N)] for _ in range(K)]
    a, _ = ring_c.reduce_scatter(x, K, 1, mode, 0.25)
    b, _ = ring.reduce_scatter(x, K, 1, mode, 0.25)
    for j in range(K):
        assert _same_bits_f32(a[j], b[j]), j
    ra, _ = ring_c.allreduce(x, K, mode, 0.25)
    rb, _ = ring.allreduce(x, K, mode, 0.25)
    for r in range(K):
        assert np.array_equal(ra[r], rb[r]), r


def test_flatten_equals_numpy_gather():
    numel = [1000, 7, 3 * 4096 + 5, 64, 1]
    offset, o = [], 0
    for n in numel:
        offset.append(o)
        o += n
    K = 4
    src = [[syn.bf16_bits(syn.gauss_bf16(0, n, syn.stream_key(7, r, p), 1e-3))
            for p, n in enumerate(numel)] for r in range(K)]
    a = ring_c.flatten_bucket(src, numel, offset, o + 3)
    b = ofl.flatten_bucket(src, numel, offset, o + 3)
    for r in range(K):
        assert np.array_equal(a[r], b[r])


def test_argument_checks():
    with pytest.raises(ValueError):
        ring_c.reduce_scatter([np.zeros(6, np.uint16)] * 4, 4)       # N % K != 0
    with pytest.raises(ValueError):
        ring_c.reduce_scatter([np.zeros(8, np.uint16)] * 4, 4, 1, mode=5)
    with pytest.raises(ValueError):
        ring_c.allreduce([np.zeros(8, np.uint16)], 1)                 # K < 2
