"""Seeded randomized parity of every collective entry point against the CPU
oracle, bit-exact: random K (including odd and non-power-of-two), ragged
chunk sizes (vector, 16-byte and element-wise layouts), micro-batches,
summation modes, accumulate, in-place forms and misaligned buffers."""
import random

import numpy as np
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import flatten as ofl
from oracle import ring
from tests import gpu_helpers as H
from tests.test_gpu_collectives import _spread_bf16
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu

KS = [2, 3, 4, 5, 7, 8, 12, 16, 31, 32, 64]
SS = [1, 7, 8, 15, 16, 17, 24, 64, 100, 1000, 4096, 4104]


def _dev_bf16(a, dev, off):
    b = torch.empty(len(a) + 24, dtype=torch.bfloat16, device=dev)
    t = b[off:off + len(a)]
    t.copy_(syn.bits_to_bf16(a).to(dev))
    return t


@pytest.mark.parametrize("case", range(40))
def test_fuzz_reduce_scatter(case):
    dev = H.device()
    rng = random.Random(9000 + case)
    nrng = np.random.default_rng(case)
    K, S, M = rng.choice(KS), rng.choice(SS), rng.choice([1, 2])
    mode, acc = rng.choice(H.MODES), rng.random() < 0.5
    N = K * S
    ioff, ooff = rng.choice([0, 0, 1, 8]), rng.choice([0, 0, 1, 4])
    x = [_spread_bf16(nrng, N, spread=rng.choice([4, 12, 20])) for _ in range(M * K)]
    xin = [_dev_bf16(a, dev, ioff) for a in x]
    init = [nrng.standard_normal(S).astype(np.float32) for _ in range(K)]
    outs = []
    for i in init:
        b = torch.empty(S + 8, dtype=torch.float32, device=dev)
        o = b[ooff:ooff + S]
        o.copy_(torch.from_numpy(i))
        outs.append(o)
    scale = rng.choice([1.0 / K, 1.0, 0.37])
    dpr.dpr_reduce_scatter(xin, K, M, N, outs, mode=mode, scale=scale, accumulate=acc)
    want, _ = ring.reduce_scatter(x, K, M, mode, scale, out_init=init if acc else None)
    torch.cuda.synchronize()
    for j in range(K):
        H.assert_f32_equal(outs[j].cpu().numpy(), want[j], f"K={K} S={S} M={M} shard {j}")


@pytest.mark.parametrize("case", range(30))
def test_fuzz_allreduce_allgather(case):
    dev = H.device()
    rng = random.Random(7000 + case)
    nrng = np.random.default_rng(100 + case)
    K, S = rng.choice(KS), rng.choice(SS)
    N = K * S
    off = rng.choice([0, 0, 1, 8])
    mode = rng.choice(H.MODES)
    x = [_spread_bf16(nrng, N, spread=12) for _ in range(K)]
    xin = [_dev_bf16(a, dev, off) for a in x]
    in_place = rng.random() < 0.5
    out = xin if in_place else [_dev_bf16(np.zeros(N, np.uint16), dev, off) for _ in range(K)]
    dpr.dpr_allreduce(xin, K, N, out, mode=mode, scale=1.0 / K)
    want, _ = ring.allreduce(x, K, mode, 1.0 / K)
    torch.cuda.synchronize()
    for r in range(K):
        H.assert_bf16_equal(H.bits(out[r]), want[r], f"AR K={K} S={S} replica {r}")
    shards = [nrng.integers(0, 65536, S, dtype=np.uint16) for _ in range(K)]
    full = [_dev_bf16(np.zeros(N, np.uint16), dev, off) for _ in range(K)]
    if rng.random() < 0.5:                      # in-place form: shard j inside replica j
        src = []
        for j in range(K):
            full[j][j * S:(j + 1) * S].copy_(syn.bits_to_bf16(shards[j]).to(dev))
            src.append(full[j][j * S:(j + 1) * S])
    else:
        src = [_dev_bf16(s, dev, rng.choice([0, 1])) for s in shards]
    dpr.dpr_allgather(src, K, N, full)
    want, _ = ring.allgather(shards, K)
    torch.cuda.synchronize()
    for r in range(K):
        H.assert_bf16_equal(H.bits(full[r]), want[r], f"AG K={K} S={S} replica {r}")


@pytest.mark.parametrize("case", range(20))
def test_fuzz_flatten_and_coalesced(case):
    dev = H.device()
    rng = random.Random(5000 + case)
    nrng = np.random.default_rng(200 + case)
    K = rng.choice([2, 3, 4, 8, 16])
    numel = [rng.choice([0, 1, 5, 16, 100, 4096, 4097, 8192 * 3 + 3, 20000]) for _ in range(rng.randint(1, 9))]
    grads = [[nrng.integers(0, 65536, n, dtype=np.uint16) if rng.random() < 0.5
              else _spread_bf16(nrng, n, spread=12) for n in numel] for _ in range(K)]
    dgr = [[_dev_bf16(g, dev, rng.choice([0, 1, 2, 8])) for g in row] for row in grads]
    # flatten with a gap after every gradient and padding at the end
    offsets, o = [], 0
    for n in numel:
        offsets.append(o)
        o += n + rng.choice([0, 0, 3, 16])
    bucket = o + rng.choice([0, 5])
    init = [nrng.integers(0, 65536, bucket, dtype=np.uint16) for _ in range(K)]
    dst = [_dev_bf16(i, dev, rng.choice([0, 1])) for i in init]
    with dpr.dpr_flatten_plan_create(dgr, numel, offsets, bucket) as plan:
        dpr.dpr_flatten_bucket(plan, dst)
        torch.cuda.synchronize()
    want = ofl.flatten_bucket(grads, numel, offsets, bucket, dst_init=init)
    for r in range(K):
        H.assert_bf16_equal(H.bits(dst[r]), want[r], f"flatten rank {r}")
    # the per-parameter reduce-scatter of the same gradients
    mode = rng.choice(H.MODES)
    with dpr.dpr_coalesced_plan_create(dgr, numel) as cplan:
        L = cplan.partition_numel
        out = [torch.empty(L, dtype=torch.float32, device=dev) for _ in range(K)]
        if L:
            dpr.dpr_reduce_scatter_coalesced(cplan, out, mode=mode)
            torch.cuda.synchronize()
            want = ring.reduce_scatter_coalesced(grads, numel, K, mode, 1.0 / K)
            for j in range(K):
                H.assert_f32_equal(out[j].cpu().numpy(), want[j], f"coalesced partition {j}")


@pytest.mark.parametrize("case", range(30))
def test_fuzz_reduce_scatter_fragments(case):
    """Random buckets: K, gradient count and sizes, gaps, end padding, source
    misalignment, mode, accumulate and scale; the fragments path against the
    oracle's gather followed by its ring reduce-scatter."""
    dev = H.device()
    rng = random.Random(5000 + case)
    nrng = np.random.default_rng(50 + case)
    K = rng.choice(KS)
    P = rng.randint(1, 7)
    sizes = [rng.choice([1, 7, 16, 100, 4095, 4096, 4097, 8192 + 16, 3 * 4096, 20000])
             for _ in range(P)]
    offset, at = [], 0
    for n in sizes:
        at += rng.choice([0, 0, 0, 1, 5, 16, 4096])
        offset.append(at)
        at += n
    order = list(range(P))
    rng.shuffle(order)                          # plan order need not be bucket order
    bucket = at + rng.choice([0, 3, 64])
    bucket += (-bucket) % K
    S = bucket // K
    host = [[_spread_bf16(nrng, n, spread=rng.choice([4, 12])) for n in sizes] for _ in range(K)]
    srcs = [[_dev_bf16(host[r][p], dev, rng.choice([0, 0, 1, 8])) for p in order] for r in range(K)]
    mode, acc = rng.choice(H.MODES), rng.random() < 0.5
    scale = rng.choice([1.0 / K, 1.0, 0.37])
    init = [nrng.standard_normal(S).astype(np.float32) for _ in range(K)]
    outs = [torch.from_numpy(i.copy()).to(dev) for i in init]
    with dpr.dpr_fragments_plan_create(srcs, [sizes[p] for p in order],
                                       [offset[p] for p in order], bucket) as plan:
        dpr.dpr_reduce_scatter_fragments(plan, outs, mode=mode, scale=scale, accumulate=acc)
        torch.cuda.synchronize()
    flat = ofl.flatten_bucket(host, sizes, offset, bucket)
    want, _ = ring.reduce_scatter(flat, K, 1, mode, scale, out_init=init if acc else None)
    for j in range(K):
        H.assert_f32_equal(outs[j].cpu().numpy(), want[j], f"K={K} P={P} shard {j}")


@pytest.mark.parametrize("case", range(16))
def test_fuzz_batched_calls(case):
    """Random batches of independent reduce-scatters and all-gathers: members of
    random chunk lengths (empty ones included) and alignments, one K, M and mode
    per batch, on a side stream (programmatic launches).  Every member equals
    the oracle bit for bit."""
    dev = H.device()
    rng = random.Random(11000 + case)
    nrng = np.random.default_rng(11000 + case)
    K, M = rng.choice([2, 3, 4, 8, 16]), rng.choice([1, 2])
    mode, acc = rng.choice(H.MODES), rng.random() < 0.5
    n = rng.randint(1, 12)
    Ss = [rng.choice([0] + SS) for _ in range(n)]
    xs, xin, init, outs = [], [], [], []
    for S in Ss:
        N = K * S
        x = [_spread_bf16(nrng, N, spread=rng.choice([4, 12])) for _ in range(M * K)]
        off = rng.choice([0, 0, 1, 8])
        xs.append(x)
        xin.append([_dev_bf16(a, dev, off) for a in x])
        i0 = [nrng.standard_normal(S).astype(np.float32) for _ in range(K)]
        init.append(i0)
        ooff = rng.choice([0, 0, 1, 4])
        row = []
        for a in i0:
            b = torch.empty(S + 8, dtype=torch.float32, device=dev)
            o = b[ooff:ooff + S]
            o.copy_(torch.from_numpy(a))
            row.append(o)
        outs.append(row)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    dpr.dpr_reduce_scatter_batch(xin, K, M, [K * S for S in Ss], outs, mode=mode,
                                 scale=1.0 / K, accumulate=acc, stream=s)
    # all-gather the first micro-batch's chunk j of rank j, member by member
    shards = [[xin[i][j][j * S:(j + 1) * S] for j in range(K)] for i, S in enumerate(Ss)]
    full = [[torch.empty(K * S, dtype=torch.bfloat16, device=dev) for _ in range(K)] for S in Ss]
    dpr.dpr_allgather_batch(shards, K, [K * S for S in Ss], full, stream=s)
    s.synchronize()
    for i, S in enumerate(Ss):
        if S == 0:
            continue
        want, _ = ring.reduce_scatter(xs[i], K, M, mode, 1.0 / K, out_init=init[i] if acc else None)
        for j in range(K):
            H.assert_f32_equal(outs[i][j].cpu().numpy(), want[j], f"member {i} shard {j}")
        want_ag, _ = ring.allgather([xs[i][j][j * S:(j + 1) * S] for j in range(K)], K)
        for r in range(K):
            H.assert_bf16_equal(H.bits(full[i][r]), want_ag[r], f"member {i} replica {r}")
