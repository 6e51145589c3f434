"""Pins of the oracle's bucket formation and flat-bucket gather against the
flush rule of the DeepSpeed ZeRO-3 source walkthrough (sections 3.1, 5.1, 5.4)
worked by hand, against invariants, and against an element-by-element loop."""
import random

import numpy as np
import pytest

from oracle import flatten as ofl
from workloads import configs as C


def test_flush_rule_small_hand_example():
    # numels in arrival order; cap 8.  3+4 = 7 fits; +10 would exceed -> flush;
    # 10 alone exceeds the cap and stands alone; 2+2 = 4 is flushed at the end.
    b = ofl.assign_buckets([3, 4, 10, 2, 2], cap=8)
    assert [x.params for x in b] == [[0, 1], [2], [3, 4]]
    assert [x.offsets for x in b] == [[0, 3], [0], [0, 2]]
    assert [x.used for x in b] == [7, 10, 4]


def test_exact_fill_does_not_flush_early():
    b = ofl.assign_buckets([4, 4, 1], cap=8)
    assert [x.params for x in b] == [[0, 1], [2]]


def test_padding_to_a_multiple_of_K():
    b = ofl.assign_buckets([5, 6, 20], cap=16, pad_to=8)
    assert [(x.used, x.numel) for x in b] == [(11, 16), (20, 24)]


def test_transformer_buckets_worked_by_hand():
    """Config 3 (hidden 4096, 7 layers) with a 25,000,000-element cap, in
    gradient-arrival order (last layer first, each layer's tensors reversed):
    fc2 and fc1 (45,088,768 each) exceed the cap and stand alone; norm2 + o
    fit (16,781,312); v and k cannot join (33.5 M) and stand alone; q and the
    next norm1 fit (16,781,312).  Six buckets per layer."""
    arr = C.CFG3.arrival_order()
    b = ofl.assign_buckets([n for _, _, n in arr], cap=C.CFG3.bucket_cap, pad_to=8)
    assert len(b) == 42
    per_layer = [["fc2"], ["fc1"], ["norm2", "o"], ["v"], ["k"], ["q", "norm1"]]
    for i, bk in enumerate(b):
        names = [arr[p][0].split(".")[1] for p in bk.params]
        assert names == per_layer[i % 6]
    sizes = sorted({x.numel for x in b})
    assert sizes == [16_777_216, 16_781_312, 45_088_768]
    assert all(x.used == x.numel for x in b)


@pytest.mark.parametrize("seed", range(5))
def test_bucket_invariants(seed):
    rng = random.Random(seed)
    numel = [rng.choice([1, 7, 64, 1000, 5000, 40000]) for _ in range(60)]
    cap = rng.choice([100, 4096, 20000])
    b = ofl.assign_buckets(numel, cap, pad_to=4)
    seen = []
    for x in b:
        assert x.offsets[0] == 0
        for k in range(1, len(x.params)):
            assert x.offsets[k] == x.offsets[k - 1] + numel[x.params[k - 1]]
        assert x.used == sum(numel[p] for p in x.params)
        assert x.used <= cap or len(x.params) == 1
        assert x.numel % 4 == 0 and x.used <= x.numel < x.used + 4
        seen += x.params
    assert seen == list(range(len(numel)))           # each once, arrival order
    # greedy: the next bucket's first gradient would not have fit
    for x, y in zip(b, b[1:]):
        assert x.used + numel[y.params[0]] > cap


def test_flatten_elementwise_loop():
    rng = np.random.default_rng(0)
    K = 3
    numel = [5, 1, 17, 8]
    offset = [0, 5, 6, 23]
    bucket = 32
    src = [[rng.integers(0, 65536, n, dtype=np.uint16) for n in numel] for _ in range(K)]
    init = [rng.integers(0, 65536, bucket, dtype=np.uint16) for _ in range(K)]
    got = ofl.flatten_bucket(src, numel, offset, bucket, dst_init=init)
    for r in range(K):
        want = init[r].copy()
        for p in range(len(numel)):
            for t in range(numel[p]):
                want[offset[p] + t] = src[r][p][t]
        assert np.array_equal(got[r], want)
        assert np.array_equal(got[r][31:], init[r][31:])     # uncovered tail kept


def test_flatten_rejects_overlap_and_out_of_bounds():
    s = [[np.zeros(4, np.uint16), np.zeros(4, np.uint16)]]
    with pytest.raises(ValueError):
        ofl.flatten_bucket(s, [4, 4], [0, 3], 8)
    with pytest.raises(ValueError):
        ofl.flatten_bucket(s, [4, 4], [0, 5], 8)
