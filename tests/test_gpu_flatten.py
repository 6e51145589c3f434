"""GPU parity of the flat-bucket gather (and of flatten followed by the
reduce-scatter, bucket by bucket) against the CPU oracle, bit-exact."""
import numpy as np
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import flatten as ofl
from oracle import ring
from tests import gpu_helpers as H
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


def _grad(n, key, dev, misalign=0):
    base = torch.empty(n + 8, dtype=torch.bfloat16, device=dev)
    t = base[misalign:misalign + n]
    t.copy_(syn.gauss_bf16(0, n, key, 1e-3).to(dev))
    return t


@pytest.mark.parametrize("dst_misalign", [0, 1, 3])
def test_flatten_parity_mixed_alignment(dst_misalign):
    dev = H.device()
    K = 3
    numel = [1, 7, 8, 13, 8192, 9000, 20001, 0, 64]
    b = ofl.assign_buckets([n for n in numel if n], cap=10 ** 9, pad_to=8)[0]
    # offsets over the non-empty gradients; the empty one sits anywhere
    offsets, k = [], 0
    for n in numel:
        if n:
            offsets.append(b.offsets[k])
            k += 1
        else:
            offsets.append(0)
    bucket = b.numel + 5
    srcs = [[_grad(n, syn.stream_key(7, r, 0, p), dev, misalign=(p + r) % 4)
             for p, n in enumerate(numel)] for r in range(K)]
    rng = np.random.default_rng(dst_misalign)
    init = [rng.integers(0, 65536, bucket, dtype=np.uint16) for _ in range(K)]
    bases = [torch.empty(bucket + 8, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    dst = [bb[dst_misalign:dst_misalign + bucket] for bb in bases]
    for r in range(K):
        dst[r].copy_(syn.bits_to_bf16(init[r]).to(dev))
    with dpr.dpr_flatten_plan_create(srcs, numel, offsets, bucket) as plan:
        dpr.dpr_flatten_bucket(plan, dst)
        torch.cuda.synchronize()
    want = ofl.flatten_bucket([[H.bits(t) for t in srcs[r]] for r in range(K)], numel, offsets,
                              bucket, dst_init=init)
    for r in range(K):
        H.assert_bf16_equal(H.bits(dst[r]), want[r], f"rank {r}")


@pytest.mark.parametrize("mode", H.MODES)
def test_flatten_then_reduce_scatter_small_transformer(mode):
    """Gradients of a small 3-layer transformer (hidden 64, MLP 176) in arrival
    order, bucketed with a cap, flattened and reduce-scattered bucket by bucket
    into one fp32 partition per rank."""
    dev = H.device()
    from workloads import configs as C
    cfg = C.Fragmented("small", 9, K=4, layers=3, dist=C.Dist("gauss", 1e-3),
                       bucket_cap=10_000, hidden=64, ffn=176)
    K = cfg.K
    arr = cfg.arrival_order()
    numel = [n for *_, n in arr]
    buckets = ofl.assign_buckets(numel, cfg.bucket_cap, pad_to=8 * K)
    grads = [[cfg.grad(r, p, device=dev) for p in range(len(arr))] for r in range(K)]
    for bi, bk in enumerate(buckets):
        P = len(bk.params)
        srcs = [[grads[r][p] for p in bk.params] for r in range(K)]
        ipg = [torch.zeros(bk.numel, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        with dpr.dpr_flatten_plan_create(srcs, [numel[p] for p in bk.params], bk.offsets,
                                         bk.numel) as plan:
            dpr.dpr_flatten_bucket(plan, ipg)
            S = bk.numel // K
            out = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
            dpr.dpr_reduce_scatter(ipg, K, 1, bk.numel, out, mode=mode)
            torch.cuda.synchronize()
        flat = ofl.flatten_bucket([[H.bits(t) for t in srcs[r]] for r in range(K)],
                                  [numel[p] for p in bk.params], bk.offsets, bk.numel)
        for r in range(K):
            H.assert_bf16_equal(H.bits(ipg[r]), flat[r], f"bucket {bi} rank {r}")
        want, _ = ring.reduce_scatter(flat, K, 1, mode, 1.0 / K)
        for j in range(K):
            H.assert_f32_equal(out[j].cpu().numpy(), want[j], f"bucket {bi} shard {j}")
        del P


def test_flatten_plan_reuse_and_destroy():
    dev = H.device()
    srcs = [[_grad(100, syn.stream_key(1, r, 0, p), dev) for p in range(2)] for r in range(2)]
    plan = dpr.dpr_flatten_plan_create(srcs, [100, 100], [0, 100], 200)
    for _ in range(3):
        dst = [torch.zeros(200, dtype=torch.bfloat16, device=dev) for _ in range(2)]
        dpr.dpr_flatten_bucket(plan, dst)
        for r in range(2):
            assert torch.equal(dst[r], torch.cat(srcs[r]))
    dpr.dpr_flatten_plan_destroy(plan)
    dpr.dpr_flatten_plan_destroy(plan)     # second destroy is a no-op
    with pytest.raises(dpr.DprError):
        dpr.dpr_flatten_bucket(plan, dst)   # a destroyed plan is rejected
