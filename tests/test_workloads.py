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
