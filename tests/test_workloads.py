"""The seeded input generator: reproducible, slab-addressable, and shaped as
the configurations state.  (It holds none of the reduction's arithmetic.)"""
import numpy as np
import torch

from workloads import configs as C
from workloads import synthetic as syn


def _bits(t):
    return syn.bf16_bits(t)


def test_reproducible_and_slab_addressable():
    a = C.CFG2.slab(3, 0, 0, 100_000)
    b = C.CFG2.slab(3, 0, 0, 100_000)
    assert np.array_equal(_bits(a), _bits(b))
    c = C.CFG2.slab(3, 0, 70_001, 999)
    assert np.array_equal(_bits(a)[70_001:71_000], _bits(c))


def test_streams_differ():
    a = _bits(C.CFG2.slab(0, 0, 0, 4096))
    b = _bits(C.CFG2.slab(1, 0, 0, 4096))
    m = _bits(C.cfg5(8, 1 << 20).slab(0, 1, 0, 4096))
    assert np.mean(a == b) < 0.05 and np.mean(a == m) < 0.05


def test_gauss_moments_and_outliers():
    x = C.CFG2.slab(0, 0, 0, 1 << 20).float().numpy().astype(np.float64)
    # 99% N(0, 1e-3) + 1% x100: std = sqrt(0.99e-6 + 0.01e-2) ~ 1.0045e-2
    assert abs(x.std() - 1.0045e-2) < 3e-4
    assert abs(np.mean(np.abs(x) > 5e-3) - 0.0096) < 0.002
    y = C.CFG1.slab(0, 0, 0, 1 << 18).float().numpy()
    assert abs(y.std() - 1e-2) < 2e-4 and abs(y.mean()) < 1e-4


def test_uniform_range():
    u = C.cfg4_slab(0, 1 << 20).float().numpy()
    assert u.min() >= -0.0201 and u.max() <= 0.0201
    assert abs(u.std() - 0.02 / np.sqrt(3)) < 2e-4


def test_hash_split_multiply_matches_python_ints():
    vals = torch.tensor([0, 1, 0xFFFF, 0x10000, 0xDEADBEEF, 0xFFFFFFFF], dtype=torch.int64)
    got = syn._fmix32(vals).tolist()
    assert got == [syn.fmix32_int(int(v)) for v in vals.tolist()]


def test_integer_example_values():
    bufs = syn.integer_example(4, 8)
    assert [b.float().tolist() for b in bufs][2] == [4, 4, 8, 8, 12, 12, 16, 16]


def test_config_sizes():
    assert C.CFG4_N == 973_078_528 and C.CFG4_N % 64 == 0
    assert len(C.CFG3.arrival_order()) == 56 and len(C.CFG3_224.arrival_order()) == 224
    assert sum(n for *_, n in C.CFG3.arrival_order()) == 1_101_062_144
    pts = C.cfg5_points()
    assert len(pts) == 55 and (64, 1 << 30) in pts and (2, 1024) in pts
    assert C.BENCH.n_frag * C.BENCH.frag_numel == C.BENCH.N


def test_index_evaluation_matches_ranges():
    idx = np.array([0, 5, 4096, 99_999, 7, 7, 123_456], dtype=np.int64)
    for cfg in (C.CFG2, C.cfg5(8, 1 << 20)):
        full = _bits(cfg.slab(1, 0, 0, 123_457))
        assert np.array_equal(_bits(cfg.at(1, 0, idx)), full[idx])
    u = _bits(C.cfg4_slab(0, 123_457))
    assert np.array_equal(_bits(C.cfg4_at(idx)), u[idx])


def test_series_logarithm_matches_libm():
    """The generator's own ln(u1) (exact split, atanh series) is within 2 ulp
    of the C library's log over a spread of words, the ends included."""
    w = torch.arange(0, 1 << 18, dtype=torch.int64) * 16381 % (1 << 32)
    w = torch.cat([w, torch.tensor([0, 1, 2, 3, 4, (1 << 31) - 1, 1 << 31, 3037000499,
                                    (1 << 32) - 2, (1 << 32) - 1])])
    got = syn._ln_u1(w).numpy()
    want = np.log((w.numpy().astype(np.float64) + 1.0) * 2.0 ** -32)
    nz = want != 0
    assert got[~nz].tolist() == [0.0]                       # u1 = 1
    ulps = np.abs(got - want)[nz] / np.spacing(np.abs(want[nz]))
    assert ulps.max() <= 2.0


def test_series_cosine_matches_libm():
    """cos(2 pi u2) by exact octant reduction and Taylor polynomials agrees
    with the C library's cos to 1e-15 absolute, including every octant edge."""
    edges = [o << 29 for o in range(8)]
    edges += [e + d for e in edges for d in (-1, 1) if 0 <= e + d < (1 << 32)]
    w = torch.cat([torch.arange(0, 1 << 18, dtype=torch.int64) * 16411 % (1 << 32),
                   torch.tensor(edges + [(1 << 32) - 1], dtype=torch.int64)])
    got = syn._cos_2pi_u2(w).numpy()
    want = np.cos(2.0 * np.pi * (w.numpy().astype(np.float64) * 2.0 ** -32))
    assert np.abs(got - want).max() < 1e-15
    assert got[w.numpy() == 0][0] == 1.0


def test_gauss_is_a_normal_sample():
    """Box-Muller values: Kolmogorov-Smirnov against N(0, 1) (the bf16 grid is
    far finer than the test's resolution at this sample size), the first two
    moments, and the 6.66-sigma cut of the tails."""
    from scipy import stats
    x = syn.gauss_bf16(0, 1 << 18, syn.stream_key(5, 1), 1.0).double().numpy()
    assert stats.kstest(x, "norm").pvalue > 1e-3
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1.0) < 0.01
    assert np.abs(x).max() <= 6.67
    y = syn.gauss_bf16(0, 1 << 16, syn.stream_key(5, 2), 1e-3).double().numpy()
    assert abs(y.std() - 1e-3) < 2e-5
