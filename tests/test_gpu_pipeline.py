"""The stream-overlapped bucket pipeline, checked against the validation list
of the issue "ZeRO-1/2 average_tensor serializes backward compute behind the
preceding reduction" (DeepSpeed issue 8364):
  - gradient parity against overlap off (gather and reduce on one stream),
    and against the CPU oracle, for both wait policies and 1-3 buffers;
  - rapid reuse of both physical buffers while the producer rewrites the
    gradients for every bucket (the ping-pong reuse race);
  - gradients produced on several streams (the multi-producer case);
  - a timing comparison: with per-buffer completion events the compute stream
    is never slower than with the reverse wait on the whole reduction stream."""
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


def _small_model(dev):
    cfg = C.Fragmented("pipe", 11, K=4, layers=4, dist=C.Dist("gauss", 1e-3), bucket_cap=12_000,
                       hidden=64, ffn=176)
    arr = cfg.arrival_order()
    numel = [n for *_, n in arr]
    buckets = ofl.assign_buckets(numel, cfg.bucket_cap, pad_to=8 * cfg.K)
    grads = [[cfg.grad(r, p, device=dev) for p in range(len(arr))] for r in range(cfg.K)]
    plans = [dpr.dpr_flatten_plan_create([[grads[r][p] for p in b.params] for r in range(cfg.K)],
                                         [numel[p] for p in b.params], b.offsets, b.numel)
             for b in buckets]
    return cfg, numel, buckets, grads, plans


def _serial(K, buckets, plans, dev):
    outs = []
    ipg = [torch.zeros(max(b.numel for b in buckets), dtype=torch.bfloat16, device=dev) for _ in range(K)]
    for b, plan in zip(buckets, plans):
        views = [t[:b.numel] for t in ipg]
        for v in views:
            v.zero_()
        dpr.dpr_flatten_bucket(plan, views)
        o = [torch.empty(b.numel // K, dtype=torch.float32, device=dev) for _ in range(K)]
        dpr.dpr_reduce_scatter(views, K, 1, b.numel, o)
        outs.append(o)
    torch.cuda.synchronize()
    return outs


@pytest.mark.parametrize("policy", [dpr.WAIT_PER_BUFFER, dpr.WAIT_REDUCTION_STREAM])
@pytest.mark.parametrize("n_buffers", [1, 2, 3])
def test_parity_against_overlap_off_and_oracle(policy, n_buffers):
    dev = H.device()
    cfg, numel, buckets, grads, plans = _small_model(dev)
    K = cfg.K
    serial = _serial(K, buckets, plans, dev)
    cur = torch.cuda.Stream()
    outs = [[torch.full((b.numel // K,), 7.0, device=dev) for _ in range(K)] for b in buckets]
    with dpr.BucketPipeline(K, max(b.numel for b in buckets), n_buffers, policy) as pipe:
        for plan, o in zip(plans, outs):
            pipe.submit(plan, o, stream=cur)
        pipe.flush(stream=cur)
        cur.synchronize()
    for bi, (b, o, so) in enumerate(zip(buckets, outs, serial)):
        flat = ofl.flatten_bucket([[H.bits(grads[r][p]) for p in b.params] for r in range(K)],
                                  [numel[p] for p in b.params], b.offsets, b.numel)
        want, _ = ring.reduce_scatter(flat, K, 1, ring.RING_FP32, 1.0 / K)
        for j in range(K):
            assert torch.equal(o[j], so[j]), f"bucket {bi} shard {j} differs from overlap off"
            H.assert_f32_equal(o[j].cpu().numpy(), want[j], f"bucket {bi} shard {j}")
    for p in plans:
        p.close()


@pytest.mark.parametrize("max_blocks", [0, 24])
def test_hop_mode_accumulate_and_block_budget(max_blocks):
    """Per-hop bf16 sums accumulated into existing partitions, with the
    reductions unbounded or held to a small block budget (grid-stride):
    bit-exact against the oracle."""
    dev = H.device()
    cfg, numel, buckets, grads, plans = _small_model(dev)
    K = cfg.K
    init = [[syn.gauss_bf16(0, b.numel // K, syn.stream_key(77, bi, 0, j), 1e-2).float()
             for j in range(K)] for bi, b in enumerate(buckets)]
    outs = [[t.clone().to(dev) for t in row] for row in init]
    cur = torch.cuda.Stream()
    with dpr.BucketPipeline(K, max(b.numel for b in buckets), 2, dpr.WAIT_PER_BUFFER,
                            max_blocks=max_blocks) as pipe:
        for plan, o in zip(plans, outs):
            pipe.submit(plan, o, mode=ring.HOP_BF16, scale=1.0 / K, accumulate=True, stream=cur)
        pipe.flush(stream=cur)
        cur.synchronize()
    for bi, b in enumerate(buckets):
        flat = ofl.flatten_bucket([[H.bits(grads[r][p]) for p in b.params] for r in range(K)],
                                  [numel[p] for p in b.params], b.offsets, b.numel)
        want, _ = ring.reduce_scatter(flat, K, 1, ring.HOP_BF16, 1.0 / K,
                                      out_init=[t.numpy() for t in init[bi]])
        for j in range(K):
            H.assert_f32_equal(outs[bi][j].cpu().numpy(), want[j], f"bucket {bi} shard {j}")
    for p in plans:
        p.close()


def test_reduction_stream_orders_other_work():
    """dpr_bucket_pipeline_stream returns the pipeline's own reduction stream:
    work ordered behind it sees every submitted reduction complete."""
    dev = H.device()
    cfg, numel, buckets, grads, plans = _small_model(dev)
    K = cfg.K
    serial = _serial(K, buckets, plans, dev)
    cur = torch.cuda.Stream()
    other = torch.cuda.Stream()
    outs = [[torch.zeros(b.numel // K, device=dev) for _ in range(K)] for b in buckets]
    copies = []
    with dpr.BucketPipeline(K, max(b.numel for b in buckets), 2) as pipe:
        rs = pipe.reduction_stream()
        assert rs.cuda_stream not in (0, cur.cuda_stream, other.cuda_stream)
        for plan, o in zip(plans, outs):
            pipe.submit(plan, o, stream=cur)
        other.wait_stream(rs)            # ordered behind the reductions, not behind a flush
        with torch.cuda.stream(other):
            copies = [[t.clone() for t in o] for o in outs]
        other.synchronize()
        pipe.flush(stream=cur)
        cur.synchronize()
    for bi, (c, so) in enumerate(zip(copies, serial)):
        for j in range(K):
            assert torch.equal(c[j], so[j]), f"bucket {bi} shard {j}"
    for p in plans:
        p.close()


def test_rapid_reuse_of_both_buffers():
    """The producer rewrites the same gradient tensors for every bucket on the
    compute stream; 48 buckets go through 2 physical buffers back to back."""
    dev = H.device()
    K, sizes = 8, [300_000, 4096, 131_072, 77]
    offsets = list(np.cumsum([0] + sizes[:-1]))
    bucket = sum(sizes) + (-sum(sizes)) % (8 * K)
    grads = [[torch.empty(n, dtype=torch.bfloat16, device=dev) for n in sizes] for _ in range(K)]
    plan = dpr.dpr_flatten_plan_create(grads, sizes, offsets, bucket)
    cur = torch.cuda.Stream()
    n_iter = 48
    outs = [[torch.empty(bucket // K, dtype=torch.float32, device=dev) for _ in range(K)]
            for _ in range(n_iter)]

    def produce(i):
        for r in range(K):
            for p, n in enumerate(sizes):
                syn.gauss_bf16(0, n, syn.stream_key(1000 + i, r, 0, p), 1e-3, device=dev,
                               out=grads[r][p])

    with dpr.BucketPipeline(K, bucket, 2, dpr.WAIT_PER_BUFFER) as pipe:
        with torch.cuda.stream(cur):
            for i in range(n_iter):
                produce(i)
                pipe.submit(plan, outs[i], stream=cur)
            pipe.flush(stream=cur)
        cur.synchronize()
    ipg = [torch.zeros(bucket, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    for i in range(n_iter):
        produce(i)
        dpr.dpr_flatten_bucket(plan, ipg)
        ref = [torch.empty(bucket // K, dtype=torch.float32, device=dev) for _ in range(K)]
        dpr.dpr_reduce_scatter(ipg, K, 1, bucket, ref)
        torch.cuda.synchronize()
        for j in range(K):
            assert torch.equal(outs[i][j], ref[j]), f"bucket {i} shard {j}"
    plan.close()


def test_multi_producer_streams():
    """Half of the gradients are written on one side stream behind a long
    matmul, half on another; the bucket lists both producers and must see
    the final gradients."""
    dev = H.device()
    K, sizes = 4, [1 << 20, 1 << 19, 4096, 1 << 20]
    offsets = list(np.cumsum([0] + sizes[:-1]))
    bucket = sum(sizes)
    grads = [[torch.zeros(n, dtype=torch.bfloat16, device=dev) for n in sizes] for _ in range(K)]
    plan = dpr.dpr_flatten_plan_create(grads, sizes, offsets, bucket)
    a = torch.randn(8192, 8192, device=dev).to(torch.bfloat16)
    torch.cuda.synchronize()
    sa, sb, cur = torch.cuda.Stream(), torch.cuda.Stream(), torch.cuda.Stream()
    want = [[syn.gauss_bf16(0, n, syn.stream_key(7, r, 0, p), 1e-3, device=dev)
             for p, n in enumerate(sizes)] for r in range(K)]
    torch.cuda.synchronize()
    out = [torch.empty(bucket // K, dtype=torch.float32, device=dev) for _ in range(K)]
    with dpr.BucketPipeline(K, bucket, 2) as pipe:
        with torch.cuda.stream(sa):
            for _ in range(6):
                a = a @ a * 1e-3                       # delay before the writes
            for r in range(K):
                for p in (0, 1):
                    grads[r][p].copy_(want[r][p])
        with torch.cuda.stream(sb):
            for r in range(K):
                for p in (2, 3):
                    grads[r][p].copy_(want[r][p])
        pipe.submit(plan, out, producers=[sa, sb], stream=cur)
        pipe.flush(stream=cur)
        cur.synchronize()
    torch.cuda.synchronize()
    flat = ofl.flatten_bucket([[H.bits(t) for t in want[r]] for r in range(K)], sizes, offsets, bucket)
    ref, _ = ring.reduce_scatter(flat, K, 1, ring.RING_FP32, 1.0 / K)
    for j in range(K):
        H.assert_f32_equal(out[j].cpu().numpy(), ref[j], f"shard {j}")
    plan.close()


def test_compute_is_not_held_behind_the_previous_reduction():
    """With the reductions on a small grid (152 blocks, as a collective library
    leaves most SMs to compute), the reverse wait stalls the compute stream at
    every bucket enqueue until the previous bucket's reduction ends; the
    per-buffer events do not, and the backward finishes measurably earlier.
    Both produce the same partitions as overlap off."""
    dev = H.device()
    import bench
    pb = bench.PipelineBackward(dev)
    pb.run("serial")
    ref = [[o.clone() for o in oo] for oo in pb.outs]
    t = {}
    for pol in ("reverse_wait", "per_buffer"):
        pb.run(pol, 152)
        t[pol] = min(pb.run(pol, 152) for _ in range(3))
        for oo, rr in zip(pb.outs, ref):
            for o, r in zip(oo, rr):
                assert torch.equal(o, r), pol
    pb.close()
    print(t)
    assert t["per_buffer"] <= 0.95 * t["reverse_wait"]


def test_refused_submits_enqueue_nothing():
    """Every check of a submit runs before anything is enqueued: outputs that
    overlap each other and more producer streams than the pipeline holds
    events for are refused, nothing is written, and the buckets submitted
    around them still match overlap off."""
    dev = H.device()
    cfg, numel, buckets, grads, plans = _small_model(dev)
    K = cfg.K
    serial = _serial(K, buckets, plans, dev)
    cur = torch.cuda.Stream()
    outs = [[torch.full((b.numel // K,), 7.0, device=dev) for _ in range(K)] for b in buckets]
    spare = torch.full((buckets[1].numel // K + 1,), 5.0, device=dev)
    producers = [torch.cuda.Stream() for _ in range(9)]
    with dpr.BucketPipeline(K, max(b.numel for b in buckets), 2) as pipe:
        for bi, (plan, o) in enumerate(zip(plans, outs)):
            if bi == 1:
                with pytest.raises(dpr.DprError) as e:
                    pipe.submit(plan, [o[0], o[0]] + o[2:], stream=cur)
                assert e.value.status == 5
                with pytest.raises(dpr.DprError) as e:       # shards 0 and 1 overlap
                    pipe.submit(plan, [spare[:-1], spare[1:]] + o[2:], stream=cur)
                assert e.value.status == 5
                with pytest.raises(dpr.DprError) as e:
                    pipe.submit(plan, o, producers=producers, stream=cur)
                assert e.value.status == 3
            pipe.submit(plan, o, stream=cur)
        pipe.flush(stream=cur)
        cur.synchronize()
    assert bool((spare == 5.0).all())
    for bi, (o, so) in enumerate(zip(outs, serial)):
        for j in range(K):
            assert torch.equal(o[j], so[j]), f"bucket {bi} shard {j}"
    for p in plans:
        p.close()
