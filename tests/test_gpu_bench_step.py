"""One step of the bench workload at its full size (K = 8, 1 GiB per rank,
N = 2**29), run through the bench's own launch sequence, against the oracle.

Every result is compared with the oracle at sampled positions of every chunk:
the first and last 64, 64 random ones, and both sides of every fragment
boundary.  Three results are also checked in full, on the device, against what
fixes them whatever the values:
- the bucket gather against the fragments it copies
  (dst[offset_p + t] = src_p[t]);
- every all-gather replica against the concatenated shards;
- every all-reduce replica against replica 0.
"""
import numpy as np
import pytest
import torch

from oracle import ring
from tests import gpu_helpers as H
from workloads import configs as C
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


def _flat_at(w, r, idx):
    """Host values of rank r's flat bucket (the 32 fragments back to back) at idx."""
    F = w.frag_numel
    out = np.empty(len(idx), np.uint16)
    for p in np.unique(idx // F):
        sel = (idx // F) == p
        out[sel] = H.bits(w.dist.at(idx[sel] % F, w.frag_key(r, int(p))))
    return out


def test_bench_step_full_size_sampled():
    dev = H.device()
    import bench
    torch.cuda.empty_cache()
    w = C.BENCH
    K, N, F, P = w.K, w.N, w.frag_numel, w.n_frag
    S = N // K
    stream = torch.cuda.Stream()
    wl = bench.Workload(dev, stream)
    assert (wl.K, wl.N) == (K, N)
    wl.step(bench.STEP_KERNELS)
    stream.synchronize()

    edges = [e for b in range(F, S, F) for e in (b - 1, b)]
    T = np.union1d(H.sample_positions(S, 64, 7), np.array(edges, np.int64))
    idx = H.chunk_positions(K, S, T)
    idx_d = torch.as_tensor(idx, device=dev)
    T_d = torch.as_tensor(T, device=dev)

    ipg0 = [H.bits(w.dist.at(idx, w.micro0_key(r))) for r in range(K)]
    flat = [_flat_at(w, r, idx) for r in range(K)]
    x = ipg0 + flat                                     # x[m*K + r]

    # bucket gather: sampled against the generator, in full against the fragments
    for r in range(K):
        H.assert_bf16_equal(H.bits(wl.ipg1_all[r][idx_d]), flat[r], f"flatten rank {r}")
        for p in range(P):
            assert torch.equal(wl.ipg1_all[r, p * F:(p + 1) * F].view(torch.int16),
                               wl.frag_all[r * P + p].view(torch.int16)), (r, p)

    # reduce-scatter, ring fp32, two micro-batches, copy into the partitions
    want, _ = ring.reduce_scatter(x, K, 2, ring.RING_FP32, 1.0 / K)
    for j in range(K):
        H.assert_f32_equal(wl.part_f32_all[j][T_d].cpu().numpy(), want[j], f"rs fp32 shard {j}")

    # reduce-scatter, per-hop bf16, accumulating into the previous partitions
    prev = [syn.gauss_bf16_at(T, w.prev_grad_key(j), 1e-3).float().numpy() for j in range(K)]
    want, _ = ring.reduce_scatter(x, K, 2, ring.HOP_BF16, 1.0 / K, out_init=prev)
    for j in range(K):
        H.assert_f32_equal(wl.part_hop_all[j][T_d].cpu().numpy(), want[j], f"rs hop shard {j}")

    # all-gather: sampled against the generator, in full against the shards
    shards = [H.bits(w.param_dist.at(j * S + T, w.param_key())) for j in range(K)]
    cat = np.concatenate(shards)
    whole = wl.shards_all.view(-1).view(torch.int16)
    for r in range(K):
        H.assert_bf16_equal(H.bits(wl.params_all[r][idx_d]), cat, f"allgather replica {r}")
        assert torch.equal(wl.params_all[r].view(torch.int16), whole), r

    # all-reduce of the flat buckets, ring fp32, x1/K, bf16 replicas
    outs, _ = ring.allreduce(flat, K, ring.RING_FP32, 1.0 / K)
    for r in range(K):
        H.assert_bf16_equal(H.bits(wl.ar_all[r][idx_d]), outs[r], f"allreduce replica {r}")
        assert torch.equal(wl.ar_all[r].view(torch.int16), wl.ar_all[0].view(torch.int16)), r

    wl.plan.close()
    del wl
    torch.cuda.empty_cache()
