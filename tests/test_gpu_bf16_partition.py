"""GPU parity of the bf16 partition path (reduce-scatter into bf16 shards with
copy_ / bf16 add_, and the step()-time cast) against the CPU oracle,
bit-exact, plus config 2 at full size over two micro steps (at every element
against the oracle's C ring simulation)."""
import numpy as np
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import bf16 as obf
from oracle import ring
from oracle import ring_c
from tests import gpu_helpers as H
from tests.test_gpu_collectives import _inputs, _upload
from workloads import configs as C
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu

CASES = [(2, 16), (3, 304), (4, 1), (5, 8003), (8, 8008), (8, 4096), (16, 40), (64, 16)]


@pytest.mark.parametrize("K,S", CASES)
@pytest.mark.parametrize("mode", H.MODES)
@pytest.mark.parametrize("M", [1, 2])
def test_reduce_scatter_bf16_parity(K, S, mode, M):
    dev = H.device()
    N = K * S
    for offset in (0, 1):
        x = _inputs(K, M, N, 300 + K + S + M + mode, "spread")
        xin = _upload(x, dev, offset)
        init = _inputs(K, 1, S, 9 + K, "gauss")
        for acc in (False, True):
            bases = [torch.empty(S + 16, dtype=torch.bfloat16, device=dev) for _ in range(K)]
            out = [b[offset:offset + S] for b in bases]
            for o, i in zip(out, init):
                o.copy_(syn.bits_to_bf16(i).to(dev))
            dpr.dpr_reduce_scatter_bf16(xin, K, M, N, out, mode=mode, scale=1.0 / K, accumulate=acc)
            want, _ = ring.reduce_scatter_bf16(x, K, M, mode, 1.0 / K, out_init=init if acc else None)
            torch.cuda.synchronize()
            for j in range(K):
                H.assert_bf16_equal(H.bits(out[j]), want[j], f"offset {offset} acc {acc} shard {j}")


@pytest.mark.parametrize("n", [1, 15, 16, 17, 4096, 100_003, 1 << 22])
@pytest.mark.parametrize("offset", [0, 1])
def test_cast_parity(n, offset):
    dev = H.device()
    rng = np.random.default_rng(n)
    bits = rng.integers(0, 65536, n, dtype=np.uint16)
    src_base = torch.empty(n + 16, dtype=torch.bfloat16, device=dev)
    src = src_base[offset:offset + n]
    src.copy_(syn.bits_to_bf16(bits).to(dev))
    out_base = torch.full((n + 16,), -1.0, device=dev)
    out = out_base[offset:offset + n]
    dpr.dpr_cast_bf16_to_fp32(src, out)
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy().view(np.uint32),
                          ring.cast_partition(bits).view(np.uint32))
    rest = out_base.cpu().numpy()
    assert np.all(rest[:offset] == -1.0) and np.all(rest[offset + n:] == -1.0)


@pytest.mark.parametrize("mode", H.MODES)
def test_cfg2_two_micro_steps_then_cast(mode):
    """Config 2 (K=8, 25 M elements): micro step 0 copies the shard into the
    bf16 partition, micro step 1 adds the next micro-batch's shard in bf16,
    step() casts to fp32.  Sampled numpy-oracle check, and every element
    against the C ring simulation; over every element the copy also equals
    bf16 of the fp32 reduce-scatter."""
    dev = H.device()
    cfg = C.CFG2
    K, N = cfg.K, cfg.N
    S = N // K
    x0 = [cfg.buffer(r, 0, device=dev) for r in range(K)]
    x1 = [cfg.buffer(r, 1, device=dev) for r in range(K)]
    part = [torch.empty(S, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    dpr.dpr_reduce_scatter_bf16(x0, K, 1, N, part, mode=mode)
    f32 = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
    dpr.dpr_reduce_scatter(x0, K, 1, N, f32, mode=mode)
    torch.cuda.synchronize()
    for j in range(K):
        assert torch.equal(part[j].view(torch.int16), f32[j].to(torch.bfloat16).view(torch.int16))
    dpr.dpr_reduce_scatter_bf16(x1, K, 1, N, part, mode=mode, accumulate=True)
    cast = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
    for j in range(K):
        dpr.dpr_cast_bf16_to_fp32(part[j], cast[j])
    torch.cuda.synchronize()
    T = H.sample_positions(S, 64, 21 + mode)
    x0h = H.gather_inputs(cfg.at, K, 1, S, T)
    x1h = H.gather_inputs(lambda r, m, idx: cfg.at(r, 1, idx), K, 1, S, T)
    p0, _ = ring.reduce_scatter_bf16(x0h, K, 1, mode, 1.0 / K)
    p1, _ = ring.reduce_scatter_bf16(x1h, K, 1, mode, 1.0 / K, out_init=p0)
    idx = torch.from_numpy(T).to(dev)
    for j in range(K):
        H.assert_bf16_equal(H.bits(part[j].index_select(0, idx)), p1[j], f"shard {j}")
        assert np.array_equal(cast[j].index_select(0, idx).cpu().numpy().view(np.uint32),
                              ring.cast_partition(p1[j]).view(np.uint32))
    # every element: the C ring simulation's fp32 shards of both micro steps,
    # rounded to bf16 and added in bf16 (copy_, then add_), then widened
    s0, _ = ring_c.reduce_scatter([H.bits(t) for t in x0], K, 1, mode, 1.0 / K)
    s1, _ = ring_c.reduce_scatter([H.bits(t) for t in x1], K, 1, mode, 1.0 / K)
    for j in range(K):
        want = obf.add(obf.from_f32(s0[j]), obf.from_f32(s1[j]))
        H.assert_bf16_equal(H.bits(part[j]), want, f"every shard {j}")
        assert np.array_equal(cast[j].cpu().numpy().view(np.uint32),
                              obf.to_f32(want).view(np.uint32)), j
