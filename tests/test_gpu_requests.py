"""Persistent collectives (dpr_reduce_scatter_init, dpr_allgather_init,
dpr_allreduce_init, dpr_start): started any number of times, a request gives
what the one-shot call gives, bit for bit, and the oracle's result; starts
on a side stream are programmatic launches ordered behind the work before
them."""
import numpy as np
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import ring
from tests import gpu_helpers as H
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("K,S,M,mode", [(8, 16 * 512, 2, ring.HOP_BF16), (4, 8 * 33, 1, ring.RING_FP32),
                                        (5, 13, 2, ring.RING_FP32)])
def test_requests_match_one_shot_calls_and_the_oracle(K, S, M, mode):
    dev = H.device()
    N = K * S
    hx = [syn.bf16_bits(syn.gauss_bf16(0, N, syn.stream_key(90, i), 1e-3, 0.01, 100.0))
          for i in range(M * K)]
    x = torch.stack([syn.bits_to_bf16(a) for a in hx]).to(dev)
    init = np.stack([syn.gauss_bf16(0, S, syn.stream_key(91, j), 1e-2).float().numpy()
                     for j in range(K)])
    part = torch.from_numpy(init.copy()).to(dev)
    full = torch.empty(K, N, dtype=torch.bfloat16, device=dev)
    ar = torch.empty(K, N, dtype=torch.bfloat16, device=dev)
    shards = x[:K, :S]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with dpr.dpr_reduce_scatter_init(x, K, M, N, part, mode=mode, accumulate=True) as rs, \
            dpr.dpr_allgather_init(shards, K, N, full) as ag, \
            dpr.dpr_allreduce_init(x[:K], K, N, ar, mode=mode) as arq:
        for _ in range(3):                 # accumulates three times
            rs.start(s)
        ag.start(s)
        arq.start(s)
        s.synchronize()
    want = init
    for _ in range(3):
        want, _ = ring.reduce_scatter(hx, K, M, mode, 1.0 / K, out_init=want)
    for j in range(K):
        H.assert_f32_equal(part[j].cpu().numpy(), want[j], f"shard {j}")
    want_ag, _ = ring.allgather([a[:S] for a in hx[:K]], K)
    want_ar, _ = ring.allreduce(hx[:K], K, mode, 1.0 / K)
    ref_ag = torch.empty_like(full)
    ref_ar = torch.empty_like(ar)
    dpr.dpr_allgather(shards, K, N, ref_ag)
    dpr.dpr_allreduce(x[:K], K, N, ref_ar, mode=mode)
    torch.cuda.synchronize()
    for r in range(K):
        H.assert_bf16_equal(H.bits(full[r]), want_ag[r], f"all-gather replica {r}")
        H.assert_bf16_equal(H.bits(ar[r]), want_ar[r], f"all-reduce replica {r}")
        assert torch.equal(full[r].view(torch.int16), ref_ag[r].view(torch.int16))
        assert torch.equal(ar[r].view(torch.int16), ref_ar[r].view(torch.int16))


def test_request_refused_at_init_and_empty_requests():
    dev = H.device()
    x = torch.zeros(4, 64, dtype=torch.bfloat16, device=dev)
    out = torch.zeros(4, 16, device=dev)
    with pytest.raises(dpr.DprError) as e:          # an output inside an input
        dpr.dpr_reduce_scatter_init(x, 4, 1, 64, x.view(torch.float32)[:, :16])
    assert e.value.status == 5
    with dpr.dpr_reduce_scatter_init(x, 4, 1, 0, out) as rq:   # N == 0: starts launch nothing
        rq.start()
    torch.cuda.synchronize()
    assert int(out.abs().sum()) == 0
