"""GPU parity of the per-parameter (ZeRO-3 discrete path) reduce-scatter and
all-gather against the CPU oracle, bit-exact: odd and empty parameters, zero
padding, mixed alignments, both summation modes, accumulate, canaries around
every written tensor, and config 3's 56 gradients at full size (sampled against the numpy
oracle, and at every element against the oracle's C ring simulation)."""
import numpy as np
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import ring
from oracle import ring_c
from tests import gpu_helpers as H
from workloads import configs as C
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu

CANARY = 0x7E57


def _tensors(K, numel, seed, dev, misalign):
    """Per-rank tensors inside larger buffers with canaries on both sides."""
    bases, views, host = [], [], []
    for r in range(K):
        rb, rv, rh = [], [], []
        for p, n in enumerate(numel):
            off = 8 + ((r + p) % 3 if misalign else 0)
            b = torch.full((n + 24,), 0, dtype=torch.int16, device=dev)
            b.fill_(CANARY)
            v = b[off:off + n].view(torch.bfloat16)
            a = syn.bf16_bits(syn.gauss_bf16(0, n, syn.stream_key(seed, r, 0, p), 1e-3, 0.01, 100.0))
            v.copy_(syn.bits_to_bf16(a).to(dev))
            rb.append((b, off))
            rv.append(v)
            rh.append(a)
        bases.append(rb)
        views.append(rv)
        host.append(rh)
    return bases, views, host


def _canaries_intact(bases, numel):
    for rb in bases:
        for (b, off), n in zip(rb, numel):
            h = b.cpu().numpy()
            assert np.all(h[:off] == CANARY) and np.all(h[off + n:] == CANARY)


CASES = [
    (2, [16, 1, 0, 4096 * 16]),
    (3, [7, 9000, 3 * 4096 * 2, 1]),
    (4, [4096 * 4 * 3, 11, 4 * 16 * 100, 5]),
    (8, [8 * 16 * 4096 + 8 * 16 * 7, 4096, 8, 13, 8 * 16 * 33]),
    (5, [5 * 16 * 4096 * 2, 77]),
]


@pytest.mark.parametrize("K,numel", CASES)
@pytest.mark.parametrize("mode", H.MODES)
@pytest.mark.parametrize("misalign", [False, True])
def test_reduce_scatter_coalesced_parity(K, numel, mode, misalign):
    dev = H.device()
    bases, views, host = _tensors(K, numel, 31 + K, dev, misalign)
    with dpr.dpr_coalesced_plan_create(views, numel) as plan:
        L = plan.partition_numel
        assert L == ring.shard_layout(numel, K)[2]
        init = [syn.gauss_bf16(0, L, syn.stream_key(5, j), 1e-2).float() for j in range(K)]
        for acc in (False, True):
            out = [i.clone().to(dev) for i in init]
            dpr.dpr_reduce_scatter_coalesced(plan, out, mode=mode, scale=1.0 / K, accumulate=acc)
            torch.cuda.synchronize()
            want = ring.reduce_scatter_coalesced(host, numel, K, mode, 1.0 / K,
                                                 out_init=[i.numpy() for i in init] if acc else None)
            for j in range(K):
                H.assert_f32_equal(out[j].cpu().numpy(), want[j], f"acc={acc} partition {j}")
    _canaries_intact(bases, numel)


@pytest.mark.parametrize("K,numel", CASES)
@pytest.mark.parametrize("misalign", [False, True])
def test_allgather_coalesced_parity(K, numel, misalign):
    dev = H.device()
    bases, views, _ = _tensors(K, numel, 77 + K, dev, misalign)
    for v in views:
        for t in v:
            t.zero_()
    L = ring.shard_layout(numel, K)[2]
    rng = np.random.default_rng(K)
    shards = [rng.integers(0, 65536, L, dtype=np.uint16) for _ in range(K)]
    with dpr.dpr_coalesced_plan_create(views, numel) as plan:
        dpr.dpr_allgather_coalesced(plan, [syn.bits_to_bf16(s).to(dev) for s in shards])
        torch.cuda.synchronize()
    want = ring.allgather_coalesced(shards, numel, K)
    for r in range(K):
        for p in range(len(numel)):
            H.assert_bf16_equal(H.bits(views[r][p]), want[r][p], f"rank {r} param {p}")
    _canaries_intact(bases, numel)


@pytest.mark.parametrize("mode", H.MODES)
def test_cfg3_per_parameter_full_size(mode):
    """Config 3 (56 gradients of the hidden-4096 transformer, K=8) through the
    discrete path at full size; oracle on sampled shard positions of four
    parameters (a norm, q, fc1, fc2); every partition element checked against
    the error bound of the exact sum."""
    dev = H.device()
    cfg = C.CFG3
    K = cfg.K
    arr = cfg.arrival_order()
    numel = [n for *_, n in arr]
    grads = [[cfg.grad(r, p, device=dev) for p in range(len(arr))] for r in range(K)]
    sizes, offs, L = ring.shard_layout(numel, K)
    with dpr.dpr_coalesced_plan_create(grads, numel) as plan:
        out = [torch.empty(L, dtype=torch.float32, device=dev) for _ in range(K)]
        dpr.dpr_reduce_scatter_coalesced(plan, out, mode=mode)
        torch.cuda.synchronize()
        for p in (0, 2, 6, 7):
            s, o, n = sizes[p], offs[p], numel[p]
            T = H.sample_positions(s, 32, p)

            def at(r, _m, idx, p=p, n=n):
                idx = np.asarray(idx)
                v = torch.zeros(len(idx), dtype=torch.bfloat16)
                ok = np.flatnonzero(idx < n)
                if len(ok):
                    v[torch.from_numpy(ok)] = cfg.grad_at(r, p, idx[ok])
                return v
            want = H.oracle_rs_sampled(at, K, 1, s, T, mode, 1.0 / K)
            idx = torch.from_numpy(o + T).to(dev)
            for j in range(K):
                H.assert_f32_equal(out[j].index_select(0, idx).cpu().numpy(), want[j], f"p{p} j{j}")
        # every element of every parameter's shards: the C ring simulation on each
        # gradient copied back from the device and zero-padded to K * s
        for p, (s, o, n) in enumerate(zip(sizes, offs, numel)):
            x = []
            for r in range(K):
                a = np.zeros(K * s, dtype=np.uint16)
                a[:n] = H.bits(grads[r][p].reshape(-1))
                x.append(a)
            want, _ = ring_c.reduce_scatter(x, K, 1, mode, 1.0 / K)
            for j in range(K):
                H.assert_f32_equal(out[j][o:o + s].cpu().numpy(), want[j], f"every p{p} j{j}")
        # the all-gather of the bf16-rounded partitions rebuilds every gradient's
        # all-reduce: compare parameter 2 (q) with dpr_allreduce of the same grads
        with dpr.dpr_coalesced_plan_create(
                [[torch.empty_like(grads[r][p]) for p in range(len(arr))] for r in range(K)],
                numel) as agp:
            dpr.dpr_allgather_coalesced(agp, [o_.to(torch.bfloat16) for o_ in out])
            p = 2
            ar = [torch.empty_like(grads[r][p]) for r in range(K)]
            dpr.dpr_allreduce([grads[r][p] for r in range(K)], K, numel[p], ar, mode=mode)
            torch.cuda.synchronize()
            for r in range(K):
                assert torch.equal(agp._tensors[r * len(arr) + p].view(torch.int16),
                                   ar[r].view(torch.int16))
            # and every parameter of every replica is its shards laid end to end,
            # padding dropped
            for q, (sq, oq, nq) in enumerate(zip(sizes, offs, numel)):
                full = torch.cat([out[j][oq:oq + sq].to(torch.bfloat16) for j in range(K)])[:nq]
                for r in range(K):
                    got = agp._tensors[r * len(arr) + q].reshape(-1)
                    assert torch.equal(got.view(torch.int16), full.view(torch.int16)), (q, r)
    del grads
    torch.cuda.empty_cache()
