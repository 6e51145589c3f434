"""One step of the bench workload at its full size (K = 8, 1 GiB per rank,
N = 2**29), with every element of both reduce-scatters and of the all-reduce
compared against the oracle, bit for bit (a NaN matches any NaN); and the
metric's own reduce-scatter (one micro-batch, both modes) at the same size
against the oracle's C ring simulation.

The inputs the oracle consumes are the generator's: the bucket's fragments,
the second micro-batch and the partitions the hop-mode reduce-scatter
accumulates into, copied to the host before the step runs (they are checked
against the generator evaluated on the host at sampled positions).  The
oracle's flat bucket is its own gather of those fragments.

Every element position of the K chunks is independent of the others, so the
oracle runs on slabs: the same positions [t0, t1) of every chunk form a
sub-problem of K * (t1 - t0) elements per rank whose shard j is the full
problem's shard j at [t0, t1).  The slabs run on a pool of host threads (numpy
releases the interpreter lock inside its array operations).
"""
import concurrent.futures as cf
import os

import numpy as np
import pytest
import torch

from oracle import flatten as ofl
from oracle import ring
from oracle import ring_c
from tests import gpu_helpers as H
from workloads import configs as C

pytestmark = pytest.mark.gpu

SLAB = 1 << 20          # positions per chunk in one oracle task


def _host(t: torch.Tensor) -> np.ndarray:
    return t.cpu().numpy()


def test_bench_step_every_element():
    dev = H.device()
    import bench
    torch.cuda.empty_cache()
    w = C.BENCH
    K, N, F, P = w.K, w.N, w.frag_numel, w.n_frag
    S = N // K
    stream = torch.cuda.Stream()
    wl = bench.Workload(dev, stream)
    # the generator's inputs, before the step consumes them
    frags = _host(wl.frag_all.view(torch.int16)).view(np.uint16).reshape(K, P, F)
    ipg0 = _host(wl.ipg0_all.view(torch.int16)).view(np.uint16)
    init_hop = _host(wl.part_hop_all)
    wl.step(bench.STEP_KERNELS)
    stream.synchronize()
    got_fp32 = _host(wl.part_f32_all)
    got_hop = _host(wl.part_hop_all)
    got_ar = _host(wl.ar_all.view(torch.int16)).view(np.uint16)
    wl.plan.close()
    del wl
    torch.cuda.empty_cache()

    # the copied inputs are the generator's values
    rng = np.random.default_rng(3)
    idx = rng.integers(0, N, 4096)
    for r in range(K):
        H.assert_bf16_equal(ipg0[r][idx], H.bits(w.dist.at(idx, w.micro0_key(r))), f"input {r}")
        p = int(rng.integers(0, P))
        fi = rng.integers(0, F, 512)
        H.assert_bf16_equal(frags[r, p][fi], H.bits(w.dist.at(fi, w.frag_key(r, p))),
                            f"fragment {p} of rank {r}")

    flat = ofl.flatten_bucket([list(frags[r]) for r in range(K)], [F] * P,
                              [p * F for p in range(P)], N)
    del frags

    def sub(bufs, t0, t1):
        return [np.concatenate([b[c * S + t0:c * S + t1] for c in range(K)]) for b in bufs]

    def check(t0):
        t1 = min(S, t0 + SLAB)
        x = sub(list(ipg0) + flat, t0, t1)              # x[m*K + r]
        want, _ = ring.reduce_scatter(x, K, 2, ring.RING_FP32, 1.0 / K)
        for j in range(K):
            H.assert_f32_equal(got_fp32[j][t0:t1], want[j], f"rs fp32 shard {j} at {t0}")
        want, _ = ring.reduce_scatter(x, K, 2, ring.HOP_BF16, 1.0 / K,
                                      out_init=[init_hop[j][t0:t1] for j in range(K)])
        for j in range(K):
            H.assert_f32_equal(got_hop[j][t0:t1], want[j], f"rs hop shard {j} at {t0}")
        outs, _ = ring.allreduce(x[K:], K, ring.RING_FP32, 1.0 / K)
        gar = sub(list(got_ar), t0, t1)
        for r in range(K):
            H.assert_bf16_equal(gar[r], outs[r], f"allreduce replica {r} at {t0}")
        return t1 - t0

    workers = max(1, min(32, os.cpu_count() or 1))
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        done = sum(ex.map(check, range(0, S, SLAB)))
    assert done == S


def test_metric_reduce_scatter_every_element():
    """The metric's own operation at its full size -- the reduce-scatter of one
    micro-batch, K = 8, 1 GiB per rank, in both summation modes, launched as
    the bench launches it -- at every element against the oracle's C ring
    simulation, slab by slab."""
    dev = H.device()
    import bench
    torch.cuda.empty_cache()
    w = C.BENCH
    K, N = w.K, w.N
    S = N // K
    stream = torch.cuda.Stream()
    wl = bench.Workload(dev, stream)
    ipg0 = _host(wl.ipg0_all.view(torch.int16)).view(np.uint16)
    got = {}
    for name in ("rs_fp32_m1", "rs_hop_m1"):
        wl.launch(name)
        stream.synchronize()
        got[name] = _host(wl.part_f32_all)
    wl.plan.close()
    del wl
    torch.cuda.empty_cache()

    def sub(bufs, t0, t1):
        return [np.concatenate([b[c * S + t0:c * S + t1] for c in range(K)]) for b in bufs]

    for t0 in range(0, S, SLAB):
        t1 = min(S, t0 + SLAB)
        x = sub(list(ipg0), t0, t1)
        for name, mode in (("rs_fp32_m1", ring_c.RING_FP32), ("rs_hop_m1", ring_c.HOP_BF16)):
            want, _ = ring_c.reduce_scatter(x, K, 1, mode, 1.0 / K)
            for j in range(K):
                H.assert_f32_equal(got[name][j][t0:t1], want[j], f"{name} shard {j} at {t0}")
