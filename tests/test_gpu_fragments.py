"""GPU parity of the reduce-scatter straight from a bucket's fragments.

The reference result is the oracle's gather of the bucket (zeros where no
gradient lies) followed by its ring reduce-scatter.  Every case must also be
bit-identical to the library's own gather followed by its reduce-scatter.
Cases cover:
- odd gradient sizes, gaps, and gradients that cross tile and chunk
  boundaries;
- misaligned sources;
- both summation modes, copy and accumulate;
- every K template and the run-time-K kernel;
- guard bytes around every buffer;
- configuration 3's 42 buckets at full size.
"""
import numpy as np
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import flatten as ofl
from oracle import ring
from tests import gpu_helpers as H
from tests.gpu_helpers import Arena
from workloads import configs as C
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


def _layout(sizes, gaps, K, pad):
    offset, at = [], 0
    for n, g in zip(sizes, gaps):
        at += g
        offset.append(at)
        at += n
    bucket = at + pad
    bucket += (-bucket) % K
    return offset, bucket


CASES = [  # (K, sizes, gaps before each, padding at the end)
    (2, [4096 * 3, 16], [0, 0], 0),
    (3, [7, 9000, 4097, 1], [5, 0, 3, 2], 11),
    (4, [8192 * 4, 300, 4096 * 4 + 16], [0, 16, 0], 64),
    (5, [5 * 4096 * 2, 77, 5], [0, 1, 0], 0),
    (8, [8 * 4096 * 3, 8 * 16 * 33, 4095, 13], [0, 0, 1, 0], 8 * 16),
    (16, [16 * 4096, 16 * 100 + 3], [0, 0], 13),
    (64, [64 * 4096 + 64 * 8], [0], 0),
]


def _grads(K, sizes, seed, dev, misalign):
    views, host = [], []
    for r in range(K):
        rv, rh = [], []
        for p, n in enumerate(sizes):
            shift = (r + p) % 3 if misalign else 0
            b = torch.empty(n + 8, dtype=torch.bfloat16, device=dev)
            v = b[shift:shift + n]
            a = syn.bf16_bits(syn.gauss_bf16(0, n, syn.stream_key(seed, r, 0, p), 1e-3, 0.01, 100.0))
            v.copy_(syn.bits_to_bf16(a).to(dev))
            rv.append(v)
            rh.append(a)
        views.append(rv)
        host.append(rh)
    return views, host


@pytest.mark.parametrize("K,sizes,gaps,pad", CASES)
@pytest.mark.parametrize("mode", H.MODES)
@pytest.mark.parametrize("misalign", [False, True])
def test_reduce_scatter_fragments_parity(K, sizes, gaps, pad, mode, misalign):
    dev = H.device()
    offset, bucket = _layout(sizes, gaps, K, pad)
    S = bucket // K
    views, host = _grads(K, sizes, 40 + K, dev, misalign)
    flat = ofl.flatten_bucket(host, sizes, offset, bucket)
    init = [syn.gauss_bf16(0, S, syn.stream_key(9, j), 1e-2).float() for j in range(K)]
    ipg = [torch.zeros(bucket, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    with dpr.dpr_fragments_plan_create(views, sizes, offset, bucket) as plan, \
            dpr.dpr_flatten_plan_create(views, sizes, offset, bucket) as fplan:
        dpr.dpr_flatten_bucket(fplan, ipg)
        for acc in (False, True):
            out = [i.clone().to(dev) for i in init]
            ref = [i.clone().to(dev) for i in init]
            dpr.dpr_reduce_scatter_fragments(plan, out, mode=mode, scale=1.0 / K, accumulate=acc)
            dpr.dpr_reduce_scatter(ipg, K, 1, bucket, ref, mode=mode, scale=1.0 / K, accumulate=acc)
            torch.cuda.synchronize()
            want, _ = ring.reduce_scatter(flat, K, 1, mode, 1.0 / K,
                                          out_init=[i.numpy() for i in init] if acc else None)
            for j in range(K):
                H.assert_f32_equal(out[j].cpu().numpy(), want[j], f"acc={acc} shard {j}")
                assert torch.equal(out[j].view(torch.int32), ref[j].view(torch.int32)), (acc, j)


def test_reduce_scatter_fragments_guards():
    """Every buffer in one allocation behind guard gaps; nothing outside the
    shards changes, including the source gradients."""
    dev = H.device()
    K, sizes, gaps, pad = 4, [4096 * 4 + 8, 1000, 37], [3, 0, 9], 20
    offset, bucket = _layout(sizes, gaps, K, pad)
    S = bucket // K
    for shift in (0, 2):
        a = Arena()
        src = [[a.add(n, torch.bfloat16, shift if p else 0) for p, n in enumerate(sizes)]
               for _ in range(K)]
        outs = [a.add(S, torch.float32, 2 * shift) for _ in range(K)]
        v = a.build(dev)
        host = [[syn.bf16_bits(syn.gauss_bf16(0, n, syn.stream_key(5, r, 0, p), 1e-3))
                 for p, n in enumerate(sizes)] for r in range(K)]
        for r in range(K):
            for p in range(len(sizes)):
                v[src[r][p]].copy_(syn.bits_to_bf16(host[r][p]).to(dev))
        a.snapshot()
        with dpr.dpr_fragments_plan_create([[v[i] for i in row] for row in src], sizes, offset,
                                           bucket) as plan:
            dpr.dpr_reduce_scatter_fragments(plan, [v[o] for o in outs], mode=ring.HOP_BF16)
        a.check_untouched([(o, 0, S) for o in outs])
        want, _ = ring.reduce_scatter(ofl.flatten_bucket(host, sizes, offset, bucket), K, 1,
                                      ring.HOP_BF16, 1.0 / K)
        for j in range(K):
            H.assert_f32_equal(v[outs[j]].cpu().numpy(), want[j], f"shift {shift} shard {j}")


def test_cfg3_fragments_full_size():
    """Configuration 3's 42 buckets: each bucket reduced straight from its
    gradients equals the gather + reduce-scatter of that bucket, bit for bit,
    and the oracle's C ring simulation on the gathered bucket at every element;
    three buckets are also checked against the numpy oracle at sampled
    positions."""
    dev = H.device()
    cfg = C.CFG3
    K = cfg.K
    arr = cfg.arrival_order()
    numel = [n for *_, n in arr]
    total = sum(numel)
    free, _ = torch.cuda.mem_get_info()
    if free / 2 ** 30 < (total * 2 * K + total * 8) / 2 ** 30 + 4:
        pytest.skip("not enough free device memory")
    buckets = ofl.assign_buckets(numel, cfg.bucket_cap, pad_to=8 * K)
    grads = [[cfg.grad(r, p, device=dev) for p in range(len(arr))] for r in range(K)]
    ipg = [torch.zeros(max(b.numel for b in buckets), dtype=torch.bfloat16, device=dev)
           for _ in range(K)]
    for bi, b in enumerate(buckets):
        S = b.numel // K
        srcs = [[grads[r][p] for p in b.params] for r in range(K)]
        sizes = [numel[p] for p in b.params]
        out = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
        ref = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
        views = [t[:b.numel] for t in ipg]
        for t in views:
            t.zero_()
        with dpr.dpr_fragments_plan_create(srcs, sizes, b.offsets, b.numel) as plan, \
                dpr.dpr_flatten_plan_create(srcs, sizes, b.offsets, b.numel) as fplan:
            dpr.dpr_reduce_scatter_fragments(plan, out)
            dpr.dpr_flatten_bucket(fplan, views)
            dpr.dpr_reduce_scatter(views, K, 1, b.numel, ref)
            torch.cuda.synchronize()
        for j in range(K):
            assert torch.equal(out[j].view(torch.int32), ref[j].view(torch.int32)), (bi, j)
        # every element, against the C ring simulation on the gathered bucket
        H.assert_rs_every_element(views, out, K, 1, ring.RING_FP32, 1.0 / K, f"bucket {bi}")
        if bi in (0, 17, 41):
            T = H.sample_positions(S, 32, bi)
            idx = H.chunk_positions(K, S, T)
            x = []
            for r in range(K):
                v = np.zeros(len(idx), np.uint16)
                for p, o, n in zip(b.params, b.offsets, sizes):
                    sel = np.flatnonzero((idx >= o) & (idx < o + n))
                    if len(sel):
                        v[sel] = H.bits(cfg.grad_at(r, p, idx[sel] - o))
                x.append(v)
            want, _ = ring.reduce_scatter(x, K, 1, ring.RING_FP32, 1.0 / K)
            T_d = torch.as_tensor(T, device=dev)
            for j in range(K):
                H.assert_f32_equal(out[j][T_d].cpu().numpy(), want[j], f"bucket {bi} shard {j}")
    del grads, ipg
    torch.cuda.empty_cache()
