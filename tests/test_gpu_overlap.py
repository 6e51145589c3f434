"""Programmatic dependent launch and the batched reduce-scatters, on the GPU.

On a stream other than the legacy default stream every kernel of the library
may be scheduled while the kernel before it drains; it must not touch a
caller buffer before that kernel has completed.  These tests run chains of
calls in which each call reads (or overwrites) what the call before it wrote,
on a side stream with no synchronisation between the calls, with programmatic
launch on and off, and compare every result with the oracle bit for bit.

The batched reduce-scatters let independent members run beside one another.
They are compared with the same members issued one call at a time and with
the oracle, including members whose inputs the kernel just before the batch
wrote, and a batch that is refused must leave every output untouched.
"""
import numpy as np
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import flatten as ofl
from oracle import ring
from tests import gpu_helpers as H
from workloads import configs as C
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


def _host_bits(n, key, sigma=1e-3):
    return syn.bf16_bits(syn.gauss_bf16(0, n, key, sigma, 0.01, 100.0))


def _dev(a, dev):
    return syn.bits_to_bf16(a).to(dev)


@pytest.fixture
def launch_mode(request):
    prev = dpr.dpr_set_programmatic_launch(request.param)
    yield request.param
    dpr.dpr_set_programmatic_launch(prev)


@pytest.mark.parametrize("launch_mode", [True, False], indirect=True,
                         ids=["programmatic", "plain"])
def test_dependent_chain_matches_oracle(launch_mode):
    """flatten -> reduce-scatter (M=2, accumulate) -> in-place all-reduce of the
    bucket -> reduce-scatter of the all-reduced bucket -> all-gather from it ->
    flatten again (overwrites what the last two read) -> reduce-scatter, three
    times over, back to back on one side stream."""
    dev = H.device()
    K = 8
    numel = [5 * 4096 * 8, 4096 + 3, 8 * 4096 * 2 + 5, 77]
    offset = list(np.cumsum([0] + numel[:-1]))
    bucket = sum(numel)
    bucket += (-bucket) % (16 * K)
    S = bucket // K
    host_frags = [[_host_bits(n, syn.stream_key(31, r, 0, p)) for p, n in enumerate(numel)]
                  for r in range(K)]
    frags = [[_dev(a, dev) for a in row] for row in host_frags]
    host_g0 = [_host_bits(bucket, syn.stream_key(32, r, 1)) for r in range(K)]
    ipg0 = [_dev(a, dev) for a in host_g0]
    ipg1 = [torch.zeros(bucket, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    init = [syn.gauss_bf16(0, S, syn.stream_key(33, j), 1e-2).float().numpy() for j in range(K)]
    part = [torch.from_numpy(a.copy()).to(dev) for a in init]
    part2 = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
    part3 = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
    full = [torch.empty(bucket, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    iters = 3
    with dpr.dpr_flatten_plan_create(frags, numel, offset, bucket) as plan:
        with torch.cuda.stream(s):
            for _ in range(iters):
                dpr.dpr_flatten_bucket(plan, ipg1, stream=s)
                dpr.dpr_reduce_scatter(ipg0 + ipg1, K, 2, bucket, part, mode=ring.RING_FP32,
                                       accumulate=True, stream=s)
                dpr.dpr_allreduce(ipg1, K, bucket, ipg1, mode=ring.RING_FP32, stream=s)
                dpr.dpr_reduce_scatter(ipg1, K, 1, bucket, part2, mode=ring.HOP_BF16, stream=s)
                dpr.dpr_allgather([ipg1[j][j * S:(j + 1) * S] for j in range(K)], K, bucket,
                                  full, stream=s)
                dpr.dpr_flatten_bucket(plan, ipg1, stream=s)
                dpr.dpr_reduce_scatter(ipg1, K, 1, bucket, part3, mode=ring.RING_FP32, stream=s)
        s.synchronize()
    flat = ofl.flatten_bucket(host_frags, numel, offset, bucket)
    acc = init
    for _ in range(iters):
        acc, _ = ring.reduce_scatter(host_g0 + flat, K, 2, ring.RING_FP32, 1.0 / K, out_init=acc)
    ar, _ = ring.allreduce(flat, K, ring.RING_FP32, 1.0 / K)
    want2, _ = ring.reduce_scatter(ar, K, 1, ring.HOP_BF16, 1.0 / K)
    want_full, _ = ring.allgather([ar[j][j * S:(j + 1) * S] for j in range(K)], K)
    want3, _ = ring.reduce_scatter(flat, K, 1, ring.RING_FP32, 1.0 / K)
    for j in range(K):
        H.assert_f32_equal(part[j].cpu().numpy(), acc[j], f"accumulated shard {j}")
        H.assert_f32_equal(part2[j].cpu().numpy(), want2[j], f"shard {j} of the all-reduced bucket")
        H.assert_f32_equal(part3[j].cpu().numpy(), want3[j], f"shard {j} after the re-gather")
        H.assert_bf16_equal(H.bits(full[j]), want_full[j], f"all-gather replica {j}")
        H.assert_bf16_equal(H.bits(ipg1[j]), flat[j], f"re-gathered bucket {j}")


def _batch_case(K, M, sizes, seed, dev):
    """Member inputs laid out in one buffer per rank, written there by one
    flatten launch (the kernel right before the batch).  Member i, micro m,
    starts at an element offset that is a multiple of 16, or of 16 plus one
    for members whose size is odd (the element-wise kernels)."""
    n = len(sizes)
    off, at = {}, 0
    for i, N in enumerate(sizes):
        for m in range(M):
            at += (-at) % 16
            if N % 2:
                at += 1
            off[i, m] = at
            at += N
    total = at + 16
    host = {(r, i, m): _host_bits(sizes[i], syn.stream_key(seed, r, m, i))
            for r in range(K) for i in range(n) for m in range(M)}
    srcs = [[_dev(host[r, i, m], dev) for i in range(n) for m in range(M)] for r in range(K)]
    numel = [sizes[i] for i in range(n) for m in range(M)]
    offsets = [off[i, m] for i in range(n) for m in range(M)]
    big = [torch.zeros(total, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    inputs = [[big[r][off[i, m]:off[i, m] + sizes[i]] for m in range(M) for r in range(K)]
              for i in range(n)]
    host_in = [[host[r, i, m] for m in range(M) for r in range(K)] for i in range(n)]
    return srcs, numel, offsets, total, big, inputs, host_in


BATCHES = [  # (K, M, mode, accumulate, member sizes)
    (8, 2, ring.RING_FP32, False, [8 * 16 * 700, 0, 8 * 8 * 33, 8 * 13, 8 * 4096 * 9 + 8 * 16, 8 * 16]),
    (8, 1, ring.HOP_BF16, True, [8 * 16 * 4096] * 6 + [8 * 3]),
    (4, 1, ring.RING_FP32, True, [4 * 16 * 999, 4 * 7, 4 * 8 * 4097]),
    (5, 2, ring.HOP_BF16, False, [5 * 16 * 301, 5 * 9, 5 * 16 * 4096]),
    (64, 1, ring.RING_FP32, False, [64 * 16 * 40, 64 * 16 * 3]),
]


@pytest.mark.parametrize("K,M,mode,accumulate,sizes", BATCHES)
def test_reduce_scatter_batch_matches_single_calls_and_oracle(K, M, mode, accumulate, sizes):
    dev = H.device()
    srcs, numel, offsets, total, big, inputs, host_in = _batch_case(K, M, sizes, 60 + K, dev)
    init = [[syn.gauss_bf16(0, N // K, syn.stream_key(61, i, 0, j), 1e-2).float().numpy()
             for j in range(K)] for i, N in enumerate(sizes)]
    outs = [[torch.from_numpy(a.copy()).to(dev) for a in row] for row in init]
    ref = [[torch.from_numpy(a.copy()).to(dev) for a in row] for row in init]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    iters = 2
    with dpr.dpr_flatten_plan_create(srcs, numel, offsets, total) as plan:
        for _ in range(iters):
            dpr.dpr_flatten_bucket(plan, big, stream=s)
            dpr.dpr_reduce_scatter_batch(inputs, K, M, sizes, outs, mode=mode,
                                         accumulate=accumulate, stream=s)
        s.synchronize()
        for _ in range(iters):
            for i, N in enumerate(sizes):
                dpr.dpr_reduce_scatter(inputs[i], K, M, N, ref[i], mode=mode,
                                       accumulate=accumulate, stream=s)
        s.synchronize()
    for i, N in enumerate(sizes):
        if N == 0:                    # an empty member launches nothing
            continue
        want = init[i]
        for _ in range(iters if accumulate else 1):
            want, _ = ring.reduce_scatter(host_in[i], K, M, mode, 1.0 / K,
                                          out_init=want if accumulate else None)
        for j in range(K):
            assert torch.equal(outs[i][j].view(torch.int32), ref[i][j].view(torch.int32)), \
                f"member {i} shard {j}: batch differs from single calls"
            H.assert_f32_equal(outs[i][j].cpu().numpy(), want[j], f"member {i} shard {j}")


def test_refused_batch_leaves_every_output_untouched():
    dev = H.device()
    K, N = 4, 4 * 16 * 64
    x = [torch.ones(N, dtype=torch.bfloat16, device=dev) for _ in range(2 * K)]
    outs = [[torch.full((N // K,), 3.0, device=dev) for _ in range(K)] for _ in range(2)]
    # member 1 writes member 0's shard 1
    clash = [outs[0], [outs[1][0], outs[0][1], outs[1][2], outs[1][3]]]
    # member 1 writes into member 0's input (x[0] holds N bf16 = N/2 fp32 slots)
    into_input = [outs[0], [outs[1][0], outs[1][1], outs[1][2],
                            x[0].view(torch.float32)[: N // K]]]
    for bad in (clash, into_input):
        with pytest.raises(dpr.DprError) as e:
            dpr.dpr_reduce_scatter_batch([x[:K], x[K:]], K, 1, [N, N], bad)
        assert e.value.status == 5
    torch.cuda.synchronize()
    for row in outs:
        for t in row:
            assert bool((t == 3.0).all())
    assert all(bool((t == 1.0).all()) for t in x)


def _fragment_buckets(dev, K):
    cfg = C.Fragmented("batch", 13, K=K, layers=3, dist=C.Dist("gauss", 1e-3), bucket_cap=20_000,
                       hidden=96, ffn=256)
    arr = cfg.arrival_order()
    numel = [n for *_, n in arr]
    buckets = ofl.assign_buckets(numel, cfg.bucket_cap, pad_to=K)
    grads = [[cfg.grad(r, p, device=dev) for p in range(len(arr))] for r in range(K)]
    return numel, buckets, grads


@pytest.mark.parametrize("mode,accumulate", [(ring.RING_FP32, False), (ring.HOP_BF16, True)])
@pytest.mark.parametrize("launch_mode", [True, False], indirect=True,
                         ids=["programmatic", "plain"])
def test_fragments_batch_matches_single_calls_and_oracle(mode, accumulate, launch_mode):
    dev = H.device()
    K = 4
    numel, buckets, grads = _fragment_buckets(dev, K)
    assert len(buckets) >= 3
    plans = [dpr.dpr_fragments_plan_create([[grads[r][p] for p in b.params] for r in range(K)],
                                           [numel[p] for p in b.params], b.offsets, b.numel)
             for b in buckets]
    init = [[syn.gauss_bf16(0, b.numel // K, syn.stream_key(62, bi, 0, j), 1e-2).float().numpy()
             for j in range(K)] for bi, b in enumerate(buckets)]
    outs = [[torch.from_numpy(a.copy()).to(dev) for a in row] for row in init]
    ref = [[torch.from_numpy(a.copy()).to(dev) for a in row] for row in init]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    dpr.dpr_reduce_scatter_fragments_batch(plans, outs, mode=mode, accumulate=accumulate, stream=s)
    for pl, o in zip(plans, ref):
        dpr.dpr_reduce_scatter_fragments(pl, o, mode=mode, accumulate=accumulate, stream=s)
    s.synchronize()
    for bi, b in enumerate(buckets):
        flat = ofl.flatten_bucket([[H.bits(grads[r][p]) for p in b.params] for r in range(K)],
                                  [numel[p] for p in b.params], b.offsets, b.numel)
        want, _ = ring.reduce_scatter(flat, K, 1, mode, 1.0 / K,
                                      out_init=init[bi] if accumulate else None)
        for j in range(K):
            assert torch.equal(outs[bi][j].view(torch.int32), ref[bi][j].view(torch.int32)), \
                f"bucket {bi} shard {j}: batch differs from single calls"
            H.assert_f32_equal(outs[bi][j].cpu().numpy(), want[j], f"bucket {bi} shard {j}")
    for pl in plans:
        pl.close()


def test_fragments_batch_refuses_an_output_inside_a_source():
    """Member 1's first shard placed over a gradient that member 0 reads."""
    dev = H.device()
    K = 4
    numel, buckets, grads = _fragment_buckets(dev, K)
    plans = [dpr.dpr_fragments_plan_create([[grads[r][p] for p in b.params] for r in range(K)],
                                           [numel[p] for p in b.params], b.offsets, b.numel)
             for b in buckets[:2]]
    outs = [[torch.full((b.numel // K,), 3.0, device=dev) for _ in range(K)] for b in buckets[:2]]
    n1 = buckets[1].numel // K
    g = max((grads[0][p] for p in buckets[0].params), key=lambda t: t.numel())
    assert g.numel() % 2 == 0 and g.numel() // 2 >= n1
    bad = [outs[0], [g.view(torch.float32)[:n1]] + outs[1][1:]]
    with pytest.raises(dpr.DprError) as e:
        dpr.dpr_reduce_scatter_fragments_batch(plans, bad)
    assert e.value.status == 5
    torch.cuda.synchronize()
    assert all(bool((t == 3.0).all()) for row in outs for t in row)
    for pl in plans:
        pl.close()


@pytest.mark.parametrize("K,n_buckets", [(4, 300), (64, 40), (3, 5)])
def test_fragments_batch_over_several_launches(K, n_buckets):
    """Batches larger than one launch holds (128 buckets, or 2048 shard
    pointers: 32 buckets at K=64), and a K without a compiled template (3):
    every bucket matches its single call and the oracle."""
    dev = H.device()
    rng = np.random.default_rng(K * 1000 + n_buckets)
    plans, outs, ref, host = [], [], [], []
    for b in range(n_buckets):
        sizes = [int(x) for x in rng.integers(1, 3000, size=int(rng.integers(1, 3)))]
        offset, at = [], 0
        for n in sizes:
            at += int(rng.integers(0, 20))
            offset.append(at)
            at += n
        bucket = at + (-at) % K + K * int(rng.integers(0, 3))
        hb = [[_host_bits(n, syn.stream_key(70 + b, r, 0, p)) for p, n in enumerate(sizes)]
              for r in range(K)]
        views = [[_dev(a, dev) for a in row] for row in hb]
        plans.append(dpr.dpr_fragments_plan_create(views, sizes, offset, bucket))
        outs.append([torch.full((bucket // K,), 2.0, device=dev) for _ in range(K)])
        ref.append([torch.full((bucket // K,), 2.0, device=dev) for _ in range(K)])
        host.append((hb, sizes, offset, bucket))
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    dpr.dpr_reduce_scatter_fragments_batch(plans, outs, mode=ring.HOP_BF16, accumulate=True,
                                           stream=s)
    for pl, o in zip(plans, ref):
        dpr.dpr_reduce_scatter_fragments(pl, o, mode=ring.HOP_BF16, accumulate=True, stream=s)
    s.synchronize()
    for b in range(n_buckets):
        for j in range(K):
            assert torch.equal(outs[b][j].view(torch.int32), ref[b][j].view(torch.int32)), \
                f"bucket {b} shard {j}: batch differs from single calls"
    for b in range(0, n_buckets, max(1, n_buckets // 7)):
        hb, sizes, offset, bucket = host[b]
        flat = ofl.flatten_bucket(hb, sizes, offset, bucket)
        init = [np.full(bucket // K, 2.0, np.float32) for _ in range(K)]
        want, _ = ring.reduce_scatter(flat, K, 1, ring.HOP_BF16, 1.0 / K, out_init=init)
        for j in range(K):
            H.assert_f32_equal(outs[b][j].cpu().numpy(), want[j], f"bucket {b} shard {j}")
    for pl in plans:
        pl.close()


def test_stacked_tensor_arguments_equal_lists():
    """The binding takes one tensor of contiguous rows in place of a list of
    rank buffers (checked once, not buffer by buffer): same pointers, same
    bits; rows that are not contiguous are refused on the host."""
    dev = H.device()
    K, M, N = 8, 2, 8 * 16 * 4096
    S = N // K
    g = torch.Generator(device=dev)
    g.manual_seed(5)
    x = torch.empty(M * K, N, dtype=torch.bfloat16, device=dev).normal_(0, 1e-3, generator=g)
    a = torch.empty(K, S, device=dev)
    b = torch.empty(K, S, device=dev)
    dpr.dpr_reduce_scatter(x, K, M, N, a, mode=ring.HOP_BF16)
    dpr.dpr_reduce_scatter(list(x.unbind(0)), K, M, N, list(b.unbind(0)), mode=ring.HOP_BF16)
    full_a = torch.empty(K, N, dtype=torch.bfloat16, device=dev)
    full_b = torch.empty(K, N, dtype=torch.bfloat16, device=dev)
    shards = x[:K, :S]                    # rows of S elements, N apart
    dpr.dpr_allgather(shards, K, N, full_a)
    dpr.dpr_allgather([shards[j] for j in range(K)], K, N, list(full_b.unbind(0)))
    ar_a = torch.empty(K, N, dtype=torch.bfloat16, device=dev)
    dpr.dpr_allreduce(x[K:], K, N, ar_a)
    ar_b = [torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    dpr.dpr_allreduce(list(x[K:].unbind(0)), K, N, ar_b)
    # a batch of 3 members as one [3, M*K, N] tensor and one [3, K, S] tensor
    xb = x.unsqueeze(0).repeat(3, 1, 1)
    ob = torch.empty(3, K, S, device=dev)
    dpr.dpr_reduce_scatter_batch(xb, K, M, [N] * 3, ob, mode=ring.HOP_BF16)
    # members whose rows cannot merge with the member dimension: shard j of
    # member i is chunk j of rank j's buffer, rows N + S apart, members
    # M*K*N apart; the batch must equal single calls given lists
    sh3 = torch.as_strided(xb, (3, K, S), (M * K * N, N + S, 1))
    fb = torch.empty(3, K, N, dtype=torch.bfloat16, device=dev)
    dpr.dpr_allgather_batch(sh3, K, [N] * 3, fb)
    fs = [torch.empty(K, N, dtype=torch.bfloat16, device=dev) for _ in range(3)]
    for i in range(3):
        dpr.dpr_allgather([sh3[i, j] for j in range(K)], K, N, list(fs[i].unbind(0)))
    torch.cuda.synchronize()
    for i in range(3):
        assert torch.equal(fb[i].view(torch.int16), fs[i].view(torch.int16)), i
        want = torch.cat([xb[i, j, j * S:(j + 1) * S] for j in range(K)])
        for r in range(K):
            assert torch.equal(fb[i, r].view(torch.int16), want.view(torch.int16)), (i, r)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    assert torch.equal(full_a.view(torch.int16), full_b.view(torch.int16))
    for r in range(K):
        assert torch.equal(ar_a[r].view(torch.int16), ar_b[r].view(torch.int16))
    for i in range(3):
        assert torch.equal(ob[i].view(torch.int32), a.view(torch.int32))
    with pytest.raises(ValueError):
        dpr.dpr_reduce_scatter(x.t(), K, M, N, a)                        # rows not contiguous
    with pytest.raises(ValueError):
        dpr.dpr_reduce_scatter(x[: M * K - 1], K, M, N, a)               # too few rows
    with pytest.raises(ValueError):
        dpr.dpr_reduce_scatter(x, K, M, N, a[:, : S - 1])                # rows too short
    with pytest.raises(ValueError):
        dpr.dpr_reduce_scatter_batch(xb.transpose(0, 1), K, M, [N] * 3, ob)


AG_BATCHES = [  # (K, member sizes, in-place members)
    (8, [8 * 16 * 600, 0, 8 * 8 * 33, 8 * 13, 8 * 8192 * 3 + 8 * 16], {0, 4}),
    (4, [4 * 16 * 4096] * 5 + [4 * 5], {2}),
    (5, [5 * 16 * 301, 5 * 9, 5 * 8192 * 2], set()),
]


@pytest.mark.parametrize("K,sizes,in_place", AG_BATCHES)
def test_allgather_batch_after_the_reduce_scatter_that_wrote_its_shards(K, sizes, in_place):
    """bf16 partition shards written by reduce-scatters on the same stream, then
    all-gathered in one batched call (members in place or not): the result
    equals single calls and the oracle's reduce-scatter followed by its
    all-gather."""
    dev = H.device()
    s = torch.cuda.Stream()
    host_x, outs, shards, ref = [], [], [], []
    for i, N in enumerate(sizes):
        S = N // K
        hx = [_host_bits(N, syn.stream_key(80 + i, r)) for r in range(K)]
        host_x.append(hx)
        xi = [_dev(a, dev) for a in hx]
        o = [torch.full((N,), 1.0, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        if i in in_place:
            sh = [o[j][j * S:(j + 1) * S] for j in range(K)]
        else:
            sh = [torch.empty(S, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        if N > 0:
            dpr.dpr_reduce_scatter_bf16(xi, K, 1, N, sh, stream=s)
        outs.append(o)
        shards.append(sh)
        ref.append([torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(K)])
    dpr.dpr_allgather_batch(shards, K, sizes, outs, stream=s)
    for i, N in enumerate(sizes):
        dpr.dpr_allgather(shards[i], K, N, ref[i], stream=s)
    s.synchronize()
    for i, N in enumerate(sizes):
        if N == 0:
            continue
        want_sh, _ = ring.reduce_scatter_bf16(host_x[i], K, 1, ring.RING_FP32, 1.0 / K)
        want, _ = ring.allgather(want_sh, K)
        for r in range(K):
            assert torch.equal(outs[i][r].view(torch.int16), ref[i][r].view(torch.int16)), \
                f"member {i} replica {r}: batch differs from single calls"
            H.assert_bf16_equal(H.bits(outs[i][r]), want[r], f"member {i} replica {r}")


def test_deep_batches_complete_in_order():
    """4096 one-block members in each batched call (the deepest chain of grids
    the calls accept), followed on the stream by work that reads every
    member's output: every member has completed before it."""
    dev = H.device()
    K, n = 4, 4096
    N = K * 16
    x = torch.empty(n, K, N, dtype=torch.bfloat16, device=dev).normal_(0, 1.0)
    out = torch.zeros(n, K, N // K, device=dev)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    dpr.dpr_reduce_scatter_batch(x, K, 1, [N] * n, out, stream=s)
    with torch.cuda.stream(s):
        total = out.sum(dim=(1, 2))             # reads every member's output after the batch
    full = torch.zeros(n, K, N, dtype=torch.bfloat16, device=dev)
    shards = torch.as_strided(x, (n, K, N // K), (K * N, N, 1))    # rank j's first chunk
    dpr.dpr_allgather_batch(shards, K, [N] * n, full, stream=s)
    with torch.cuda.stream(s):
        copied = full.float().sum(dim=(1, 2))
    s.synchronize()
    # what the stream read right after each batch is what the members finally wrote
    assert torch.equal(total, out.sum(dim=(1, 2)))
    assert torch.equal(copied, full.float().sum(dim=(1, 2)))
    ref = torch.empty(K, N // K, device=dev)
    for i in (0, 1, n // 2, n - 2, n - 1):
        dpr.dpr_reduce_scatter(x[i], K, 1, N, ref)
        torch.cuda.synchronize()
        assert torch.equal(out[i].view(torch.int32), ref.view(torch.int32)), i
    cat = shards.reshape(n, 1, N).expand(n, K, N)       # every replica: the K shards in order
    assert torch.equal(full.view(torch.int16), cat.contiguous().view(torch.int16))


def test_batched_calls_replay_from_a_cuda_graph():
    """The batched calls captured in a CUDA graph (their programmatic launches
    become programmatic edges) replay to the eager results, twice in a row."""
    dev = H.device()
    K, M, n, N = 8, 1, 6, 8 * 16 * 1024
    S = N // K
    g = torch.Generator(device=dev)
    g.manual_seed(21)
    x = torch.empty(n, M * K, N, dtype=torch.bfloat16, device=dev).normal_(0, 1e-3, generator=g)
    eager_rs = torch.empty(n, K, S, device=dev)
    eager_ag = torch.empty(n, K, N, dtype=torch.bfloat16, device=dev)
    shards = torch.as_strided(x, (n, K, S), (M * K * N, N, 1))
    dpr.dpr_reduce_scatter_batch(x, K, M, [N] * n, eager_rs)
    dpr.dpr_allgather_batch(shards, K, [N] * n, eager_ag)
    numel, buckets, grads = _fragment_buckets(dev, 4)
    plans = [dpr.dpr_fragments_plan_create([[grads[r][p] for p in b.params] for r in range(4)],
                                           [numel[p] for p in b.params], b.offsets, b.numel)
             for b in buckets]
    eager_fr = [torch.empty(4, b.numel // 4, device=dev) for b in buckets]
    dpr.dpr_reduce_scatter_fragments_batch(plans, eager_fr)
    torch.cuda.synchronize()
    rs = torch.zeros_like(eager_rs)
    ag = torch.zeros_like(eager_ag)
    fr = [torch.zeros_like(t) for t in eager_fr]
    s = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        dpr.dpr_reduce_scatter_batch(x, K, M, [N] * n, rs, stream=s)
        dpr.dpr_allgather_batch(shards, K, [N] * n, ag, stream=s)
        dpr.dpr_reduce_scatter_fragments_batch(plans, fr, stream=s)
    for _ in range(2):
        rs.zero_()
        ag.zero_()
        for t in fr:
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(rs.view(torch.int32), eager_rs.view(torch.int32))
        assert torch.equal(ag.view(torch.int16), eager_ag.view(torch.int16))
        for a, b in zip(fr, eager_fr):
            assert torch.equal(a.view(torch.int32), b.view(torch.int32))
    del graph
    for pl in plans:
        pl.close()
