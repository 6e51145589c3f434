"""Pins of the CPU oracle's ring simulation against what the pages and the
mathematics fix: the printed worked examples (round by round), closed forms,
traffic counts, invariants, error bounds and exact-rational brute force."""
import random

import numpy as np
import pytest

from oracle import bf16 as obf
from oracle import ring
from tests import exact_fp as X
from tests import golden_io
from workloads import synthetic as syn

MODES = (ring.RING_FP32, ring.HOP_BF16)


# --- helpers ---------------------------------------------------------------------

def _int_example(K):
    """x_r[c] = (c + 1) * 2**r, one element per chunk (N = K)."""
    return [syn.bf16_bits(t) for t in syn.integer_example(K, K)]


def _decode(state_arr, c):
    """Contributor set of chunk c's copy (one element) in a traced state."""
    arr = np.asarray(state_arr)
    v = float(arr[c]) if arr.dtype == np.float32 else float(obf.to_f32(arr[c:c + 1])[0])
    mask = v / (c + 1)
    assert mask == int(mask), "integer example decodes to an integer mask"
    m = int(mask)
    return frozenset(r for r in range(16) if m >> r & 1)


def _check_against_golden(golden, trace, K):
    by_round = {(ph, i + 1): (sends, states) for ph, i, sends, states in trace.rounds}
    checked = 0
    for key, want in golden.items():
        sends, states = by_round[key]
        for s in want["sends"]:
            assert s in sends, f"{key}: the page's transfer {s} is not in the simulation"
        for r, row in enumerate(want["rows"]):
            for c, cell in enumerate(row):
                if cell is None:
                    continue
                got = _decode(states[r], c)
                assert got == cell, f"{key} rank {r} chunk {c}: {sorted(got)} != {sorted(cell)}"
                checked += 1
    return checked


def _random_bf16(rng, n, spread=20, zero_frac=0.0):
    """Random finite bf16 bit patterns with exponents spread over +-spread."""
    out = np.empty(n, dtype=np.uint16)
    for i in range(n):
        if rng.random() < zero_frac:
            out[i] = 0
            continue
        s = rng.getrandbits(1)
        e = 127 + rng.randint(-spread, spread)
        m = rng.getrandbits(7)
        out[i] = (s << 15) | (e << 7) | m
    return out


def _ring_expected(x, K, M, mode, scale, acc_init=None):
    """Brute force in exact rationals: chunk j starts at rank j and adds ranks
    j+1, ..., j-1, each add rounded to the mode's format; then x scale (f32)."""
    N = len(x[0])
    S = N // K
    R = X.f32 if mode == ring.RING_FP32 else X.bf16
    sc = X.of_f32(np.float32(scale))
    out = []
    for j in range(K):
        shard = []
        for t in range(S):
            e = j * S + t

            def g(r):
                v = X.of_bf16_bits(x[r][e])
                for m in range(1, M):
                    v = X.bf16(X.add(v, X.of_bf16_bits(x[m * K + r][e])))
                return v
            acc = g(j)
            for s in range(1, K):
                acc = R(X.add(acc, g((j + s) % K)))
            v = X.f32(X.mul(acc, sc))
            if acc_init is not None:
                v = X.f32(X.add(X.of_f32(acc_init[j][t]), v))
            shard.append(v)
        out.append(shard)
    return out


# --- the pages' worked examples ----------------------------------------------------

def test_worked_example_4gpu_round_by_round():
    """Ring All-Reduce illustrated (CSDN): every state table of both phases."""
    golden = golden_io.load("ring_allreduce_illustrated_4gpu.txt")
    tr = ring.Trace()
    outs, ctr = ring.allreduce(_int_example(4), 4, ring.RING_FP32, 1.0, trace=tr)
    n = _check_against_golden(golden, tr, 4)
    assert n == 4 * 4 * 3 + 8 + 12 + 16      # RS cells + stated AG cells
    # final: a_j + b_j + c_j + d_j = 15 (j + 1) on every GPU
    for r in range(4):
        assert list(obf.to_f32(outs[r])) == [15.0 * (j + 1) for j in range(4)]


def test_worked_example_4gpu_hop_bf16_same_trace():
    """The same tables hold with bf16 on the wire (integer values are exact)."""
    golden = golden_io.load("ring_allreduce_illustrated_4gpu.txt")
    tr = ring.Trace()
    ring.allreduce(_int_example(4), 4, ring.HOP_BF16, 1.0, trace=tr)
    _check_against_golden(golden, tr, 4)


def test_lecture_exercise3_k3():
    """CMU 11-868 Lecture 14 notes, exercise 3 answer (K = 3 ring)."""
    golden = golden_io.load("lecture14_exercise3_k3.txt")
    tr = ring.Trace()
    ring.allreduce(_int_example(3), 3, ring.RING_FP32, 1.0, trace=tr)
    _check_against_golden(golden, tr, 3)


def test_landing_rank_and_partition_slot():
    """After K-1 rounds rank r holds the complete chunk (r+1) mod K (lecture
    section 3.2); reduce_scatter puts that chunk in slot j = chunk index."""
    for K in (2, 3, 4, 5, 8):
        tr = ring.Trace()
        shards, _ = ring.reduce_scatter(_int_example(K), K, 1, ring.RING_FP32, 1.0, trace=tr)
        last = tr.rounds[-1][3]
        for r in range(K):
            c = (r + 1) % K
            assert _decode(last[r], c) == frozenset(range(K))
        for j in range(K):
            assert float(shards[j][0]) == (2 ** K - 1) * (j + 1)


# --- closed forms, counters, shape contracts ----------------------------------------

@pytest.mark.parametrize("K", [2, 3, 4, 5, 8, 16])
def test_traffic_counters(K):
    """Each device sends 2(K-1) N/K elements in 2(K-1) rounds (lecture section
    3.2, exercise 4; CSDN summary: 2 x (N-1) rounds)."""
    N = K * 6
    x = [np.zeros(N, np.uint16) for _ in range(K)]
    _, ctr = ring.allreduce(x, K)
    assert ctr.rounds == 2 * (K - 1)
    assert ctr.sent == [2 * (K - 1) * N // K] * K
    _, ctr = ring.reduce_scatter(x, K)
    assert ctr.rounds == K - 1 and ctr.sent == [(K - 1) * N // K] * K
    _, ctr = ring.allgather([np.zeros(N // K, np.uint16)] * K, K)
    assert ctr.rounds == K - 1 and ctr.sent == [(K - 1) * N // K] * K


def test_buffer_sizes_exercise2():
    """Lecture exercise 2: with 4 devices and N inputs the reduce-scatter output
    is N/4 per device; the all-gather output is K times its input."""
    K, N = 4, 32
    x = [np.zeros(N, np.uint16) for _ in range(K)]
    shards, _ = ring.reduce_scatter(x, K)
    assert [len(s) for s in shards] == [N // 4] * K
    outs, _ = ring.allgather([np.zeros(N // 4, np.uint16)] * K, K)
    assert [len(o) for o in outs] == [N] * K


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("K", [2, 3, 4, 8, 16])
def test_closed_form_integer_sum(K, mode):
    """Small integers sum exactly in any order: the result is sum_r x_r,
    scaled by 1/K exactly when K is a power of two."""
    rng = np.random.default_rng(K)
    S = 5
    N = K * S
    vals = rng.integers(-7, 8, size=(K, N))
    x = [obf.from_f32(v.astype(np.float32)) for v in vals]
    scale = 1.0 / K if K & (K - 1) == 0 else 1.0
    shards, _ = ring.reduce_scatter(x, K, 1, mode, scale)
    total = vals.sum(axis=0)
    for j in range(K):
        assert np.array_equal(shards[j], (total[j * S:(j + 1) * S] * scale).astype(np.float32))


# --- exact brute force ------------------------------------------------------------

@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("K", [2, 3, 4, 5, 8])
def test_bruteforce_exact_rounding(K, mode):
    rng = random.Random(1000 + K + 10 * mode)
    S = 6
    N = K * S
    x = [_random_bf16(rng, N, spread=14, zero_frac=0.05) for _ in range(K)]
    scale = np.float32(1.0 / K)
    got, _ = ring.reduce_scatter(x, K, 1, mode, float(scale))
    want = _ring_expected(x, K, 1, mode, scale)
    for j in range(K):
        for t in range(S):
            assert X.same(X.of_f32(got[j][t]), want[j][t]), (j, t)


@pytest.mark.parametrize("mode", MODES)
def test_bruteforce_two_microbatches_and_accumulate(mode):
    """A2 (g = bf16(g0 + g1) before the ring) and the accumulate epilogue
    (out = out + acc * scale, two roundings)."""
    rng = random.Random(77 + mode)
    K, S = 4, 5
    N = K * S
    x = [_random_bf16(rng, N, spread=10) for _ in range(2 * K)]
    init = [np.float32(rng.uniform(-3, 3)) * np.ones(S, np.float32) for _ in range(K)]
    for j in range(K):
        init[j][::2] = np.float32(2.0 ** rng.randint(-20, 5))
    got, _ = ring.reduce_scatter(x, K, 2, mode, 0.25, out_init=init)
    want = _ring_expected(x, K, 2, mode, np.float32(0.25), acc_init=init)
    for j in range(K):
        for t in range(S):
            assert X.same(X.of_f32(got[j][t]), want[j][t]), (j, t)


@pytest.mark.parametrize("mode", MODES)
def test_ring_order_is_what_the_pin_checks(mode):
    """The brute-force inputs are order-sensitive: summing every chunk in rank
    order 0..K-1 (a plausible bug: ignoring the chunk's start rank) changes
    some results, so the exact-order pin above does discriminate."""
    rng = random.Random(5 + mode)
    K, S = 5, 16
    N = K * S
    x = [_random_bf16(rng, N, spread=14) for _ in range(K)]
    ring_res = _ring_expected(x, K, 1, mode, np.float32(1.0))
    R = X.f32 if mode == ring.RING_FP32 else X.bf16
    differ = 0
    for j in range(1, K):
        for t in range(S):
            e = j * S + t
            acc = X.of_bf16_bits(x[0][e])
            for r in range(1, K):
                acc = R(acc + X.of_bf16_bits(x[r][e]))
            differ += X.f32(acc) != ring_res[j][t]
    assert differ > 0


# --- all-gather / all-reduce invariants -------------------------------------------

@pytest.mark.parametrize("K", [2, 3, 4, 8])
def test_allgather_replicas_identical_and_concatenated(K):
    """After the all-gather all K buffers are identical (CSDN Phase 2 end state)
    and equal to the shards concatenated in rank order."""
    rng = np.random.default_rng(K)
    S = 7
    shards = [rng.integers(0, 65536, S, dtype=np.uint16) for _ in range(K)]
    outs, _ = ring.allgather(shards, K)
    cat = np.concatenate(shards)
    for o in outs:
        assert np.array_equal(o, cat)


@pytest.mark.parametrize("mode", MODES)
@pytest.mark.parametrize("K", [2, 3, 4, 8])
def test_allreduce_equals_reduce_scatter_then_allgather(K, mode):
    """AllReduce = ReduceScatter + AllGather (lecture section 2.2): every
    replica equals bf16(reduce-scatter shards) concatenated."""
    rng = random.Random(K * 3 + mode)
    S = 9
    x = [_random_bf16(rng, K * S, spread=12) for _ in range(K)]
    scale = 1.0 / K
    outs, _ = ring.allreduce(x, K, mode, scale)
    shards, _ = ring.reduce_scatter(x, K, 1, mode, scale)
    want = np.concatenate([obf.from_f32(s) for s in shards])
    for o in outs:
        assert np.array_equal(o, want)


# --- error bound and "ring order != np.sum" --------------------------------------

@pytest.mark.parametrize("mode,u", [(ring.RING_FP32, 2.0 ** -24), (ring.HOP_BF16, 2.0 ** -8)])
def test_recursive_summation_error_bound(mode, u):
    """|ring sum - exact sum| <= gamma_{K-1} * sum |x|, gamma_n = n u / (1 - n u)
    (standard bound for recursive summation, Higham, Accuracy and Stability of
    Numerical Algorithms, section 4.2)."""
    K, S = 16, 64
    x = [syn.bf16_bits(syn.gauss_bf16(0, K * S, syn.stream_key(9, r), 1e-3)) for r in range(K)]
    shards, _ = ring.reduce_scatter(x, K, 1, mode, 1.0)
    xs = np.stack([obf.to_f32(a).astype(np.float64) for a in x])
    exact = xs.sum(axis=0)          # <= 16 terms of 8-bit significands: exact in fp64
    absum = np.abs(xs).sum(axis=0)
    got = np.concatenate(shards).astype(np.float64)
    n = K - 1
    gamma = n * u / (1 - n * u)
    assert np.all(np.abs(got - exact) <= gamma * absum)


@pytest.mark.parametrize("mode", MODES)
def test_ring_order_differs_from_other_orders_in_last_bits(mode):
    """Lecture section 3.3: the ring sums chunk by chunk in ring order, so the
    rounded result differs from another summation order in the last bits for
    some elements (K = 64); with bf16 on the wire, for many."""
    K, S = 64, 64
    x = [syn.bf16_bits(syn.gauss_bf16(0, K * S, syn.stream_key(11, r), 1e-3)) for r in range(K)]
    shards, _ = ring.reduce_scatter(x, K, 1, mode, 1.0)
    got = np.concatenate(shards).astype(np.float64)
    other = np.zeros(K * S, np.uint16) if mode == ring.HOP_BF16 else np.zeros(K * S, np.float32)
    for r in range(K):                      # rank order 0..K-1 for every chunk
        if mode == ring.HOP_BF16:
            other = obf.add(other, x[r])
        else:
            other = other + obf.to_f32(x[r])
    other = (obf.to_f32(other) if mode == ring.HOP_BF16 else other).astype(np.float64)
    differ = np.mean(got != other)
    assert differ > (0.2 if mode == ring.HOP_BF16 else 0.0)
    xs = np.stack([obf.to_f32(a).astype(np.float64) for a in x])
    u = 2.0 ** -8 if mode == ring.HOP_BF16 else 2.0 ** -24
    gamma = (K - 1) * u / (1 - (K - 1) * u)
    assert np.all(np.abs(got - other) <= 2 * gamma * np.abs(xs).sum(axis=0))


# --- special values and argument checks ----------------------------------------------

def test_nan_inf_propagate():
    K, N = 4, 8
    x = [np.full(N, obf.from_f32(np.float32([1.0]))[0], np.uint16) for _ in range(K)]
    x[2][1] = 0x7FC0           # NaN in chunk 0
    x[1][3] = 0x7F80           # +Inf in chunk 1
    # chunk 2 (ring order: ranks 2, 3, 0, 1): 1 + max_bf16 + 2**119 + 1.  The
    # sum max_bf16 + 2**119 is exactly halfway between max_bf16 and 2**128, so
    # it rounds (ties to even) to +Inf in bf16 but is a finite fp32 value.
    x[3][5] = 0x7F7F           # largest finite bf16, (2 - 2**-7) * 2**127
    x[0][5] = 0x7B00           # 2**119
    for mode in MODES:
        sh, _ = ring.reduce_scatter(x, K, 1, mode, 1.0)
        v = np.concatenate(sh)
        assert np.isnan(v[1]) and v[3] == np.inf
        assert (v[5] == np.inf) == (mode == ring.HOP_BF16)


def test_argument_checks():
    with pytest.raises(ValueError):
        ring.reduce_scatter([np.zeros(4, np.uint16)], 1)
    with pytest.raises(ValueError):
        ring.reduce_scatter([np.zeros(5, np.uint16)] * 2, 2)
    with pytest.raises(ValueError):
        ring.reduce_scatter([np.zeros(4, np.uint16)] * 3, 2, M=2)


def test_trace_sends_follow_the_index_formula():
    """Lecture section 3.2: reduce-scatter round i sends chunk (r - i) mod K,
    all-gather round i (after reduce-scatter) sends chunk (r + 1 - i) mod K."""
    for K in (3, 4, 7):
        tr = ring.Trace()
        ring.allreduce([np.zeros(K * 2, np.uint16)] * K, K, trace=tr)
        for phase, i, sends, _ in tr.rounds:
            for s, d, c in sends:
                assert d == (s + 1) % K
                assert c == ((s - i) % K if phase == "rs" else (s + 1 - i) % K)
