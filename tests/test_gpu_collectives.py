"""GPU parity, element by element, of the C-ABI reduce-scatter, all-reduce and
all-gather against the CPU oracle, at sizes the oracle finishes in seconds:
every K kernel specialisation and the run-time-K kernels, vector and
element-wise layouts, ragged tails, several blocks per chunk, the grid-stride
wrap, both summation modes, 1 and 2 micro-batches, copy and accumulate,
in-place forms, special values and empty calls.  Results must be bit-exact
(NaN compared as NaN)."""
import numpy as np
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import bf16 as obf
from oracle import ring
from tests import gpu_helpers as H
from workloads import synthetic as syn

pytestmark = pytest.mark.gpu


def _spread_bf16(rng, n, spread=20):
    """Finite bf16 bit patterns with exponents over +-spread: order-sensitive sums."""
    s = rng.integers(0, 2, n, dtype=np.uint32)
    e = (127 + rng.integers(-spread, spread + 1, n)).astype(np.uint32)
    m = rng.integers(0, 128, n, dtype=np.uint32)
    return ((s << 15) | (e << 7) | m).astype(np.uint16)


def _inputs(K, M, N, seed, kind):
    if kind == "spread":
        rng = np.random.default_rng(seed)
        return [_spread_bf16(rng, N) for _ in range(M * K)]
    return [syn.bf16_bits(syn.gauss_bf16(0, N, syn.stream_key(seed, i), 1e-3, 0.01, 100.0))
            for i in range(M * K)]


def _upload(arrs, dev, offset=0):
    """bf16 device tensors holding `arrs`; offset > 0 shifts each buffer by that
    many elements off its allocation's alignment."""
    out = []
    for a in arrs:
        base = torch.empty(len(a) + 8, dtype=torch.bfloat16, device=dev)
        t = base[offset:offset + len(a)]
        t.copy_(syn.bits_to_bf16(a).to(dev))
        out.append(t)
    return out


RS_CASES = [  # (K, S): S % 8 == 0 takes the vector kernels, otherwise element-wise
    (2, 8), (2, 4104), (3, 304), (4, 1024), (4, 1), (5, 8003), (7, 13), (8, 8008),
    (8, 1000), (16, 2056), (32, 136), (64, 264), (64, 8), (6, 4096), (12, 40),
]


@pytest.mark.parametrize("K,S", RS_CASES)
@pytest.mark.parametrize("mode", H.MODES)
@pytest.mark.parametrize("M", [1, 2])
def test_reduce_scatter_parity(K, S, mode, M):
    dev = H.device()
    N = K * S
    for kind, acc in (("spread", False), ("gauss", True)):
        seed = 1000 * K + S + 7 * M + 3 * mode + (kind == "gauss")
        x = _inputs(K, M, N, seed, kind)
        xin = _upload(x, dev)
        init = [obf.to_f32(a[:S]).copy() for a in _inputs(K, 1, S, seed + 1, "gauss")]
        out = [torch.from_numpy(i.copy()).to(dev) for i in init]
        dpr.dpr_reduce_scatter(xin, K, M, N, out, mode=mode, scale=1.0 / K, accumulate=acc)
        want, _ = ring.reduce_scatter(x, K, M, mode, 1.0 / K, out_init=init if acc else None)
        torch.cuda.synchronize()
        for j in range(K):
            H.assert_f32_equal(out[j].cpu().numpy(), want[j], f"{kind} shard {j}")


def test_reduce_scatter_grid_stride_wrap():
    """A chunk larger than one wave of blocks covers (several loop trips)."""
    dev = H.device()
    K, S = 2, 8 * 1_000_003
    N = K * S
    x = _inputs(K, 1, N, 99, "gauss")
    out = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
    dpr.dpr_reduce_scatter(_upload(x, dev), K, 1, N, out, mode=ring.RING_FP32, scale=0.5)
    want, _ = ring.reduce_scatter(x, K, 1, ring.RING_FP32, 0.5)
    for j in range(K):
        H.assert_f32_equal(out[j].cpu().numpy(), want[j], f"shard {j}")


@pytest.mark.parametrize("mode", H.MODES)
def test_reduce_scatter_unaligned_buffers(mode):
    """2-byte aligned inputs and 4-byte aligned outputs take the element-wise
    kernel and give the same bits."""
    dev = H.device()
    K, S = 8, 1024
    N = K * S
    x = _inputs(K, 2, N, 5, "spread")
    xin = _upload(x, dev, offset=1)
    out_base = [torch.empty(S + 4, dtype=torch.float32, device=dev) for _ in range(K)]
    out = [b[1:1 + S] for b in out_base]
    dpr.dpr_reduce_scatter(xin, K, 2, N, out, mode=mode, scale=0.125)
    want, _ = ring.reduce_scatter(x, K, 2, mode, 0.125)
    for j in range(K):
        H.assert_f32_equal(out[j].cpu().numpy(), want[j], f"shard {j}")


def test_worked_example_integer_4gpu():
    """Ring All-Reduce illustrated: final chunk sums 15 (j + 1), averaged by 1/4."""
    dev = H.device()
    bufs = [b.to(dev) for b in syn.integer_example(4, 4)]
    out = [torch.empty(1, dtype=torch.float32, device=dev) for _ in range(4)]
    dpr.dpr_reduce_scatter(bufs, 4, 1, 4, out, scale=0.25)
    assert [o.item() for o in out] == [15 * (j + 1) / 4 for j in range(4)]
    ar = [torch.empty(4, dtype=torch.bfloat16, device=dev) for _ in range(4)]
    dpr.dpr_allreduce(bufs, 4, 4, ar, scale=1.0)
    for r in range(4):
        assert ar[r].float().tolist() == [15.0, 30.0, 45.0, 60.0]


def test_special_values():
    dev = H.device()
    K, S = 4, 16
    N = K * S
    for vec_offset in (0, 1):
        x = [np.full(N, 0x3F80, np.uint16) for _ in range(K)]        # 1.0
        x[2][1] = 0x7FC0                                             # NaN
        x[1][S + 3] = 0x7F80                                         # +Inf
        x[3][2 * S + 5] = 0x7F7F                                     # max bf16 ...
        x[0][2 * S + 5] = 0x7B00                                     # + 2**119 (bf16 tie -> Inf)
        x[1][3 * S] = 0xFF80                                         # -Inf
        x[2][3 * S] = 0x7F80                                         # +Inf: Inf - Inf = NaN
        x[0][7] = 0x0001                                             # subnormals
        x[1][7] = 0x8003
        for mode in H.MODES:
            out = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
            dpr.dpr_reduce_scatter(_upload(x, dev, vec_offset), K, 1, N, out, mode=mode, scale=1.0)
            want, _ = ring.reduce_scatter(x, K, 1, mode, 1.0)
            for j in range(K):
                H.assert_f32_equal(out[j].cpu().numpy(), want[j], f"mode {mode} shard {j}")


def test_empty_calls_launch_nothing():
    dev = H.device()
    t = torch.zeros(4, device=dev)
    dpr.dpr_reduce_scatter([], 4, 1, 0, [])
    dpr.dpr_allgather([], 4, 0, [])
    dpr.dpr_allreduce([], 4, 0, [])
    torch.cuda.synchronize()
    assert t.sum().item() == 0


AR_CASES = [(2, 8), (3, 24), (4, 1024), (5, 13), (8, 1000), (8, 8008), (16, 72), (64, 16)]


@pytest.mark.parametrize("K,S", AR_CASES)
@pytest.mark.parametrize("mode", H.MODES)
@pytest.mark.parametrize("in_place", [False, True])
def test_allreduce_parity(K, S, mode, in_place):
    dev = H.device()
    N = K * S
    x = _inputs(K, 1, N, 500 + K + S + mode, "spread")
    xin = _upload(x, dev)
    out = xin if in_place else [torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    dpr.dpr_allreduce(xin, K, N, out, mode=mode, scale=1.0 / K)
    want, _ = ring.allreduce(x, K, mode, 1.0 / K)
    for r in range(K):
        H.assert_bf16_equal(H.bits(out[r]), want[r], f"replica {r}")


AG_CASES = [(2, 8), (3, 21), (4, 1024), (7, 8), (8, 8008), (16, 5), (64, 40)]


@pytest.mark.parametrize("K,S", AG_CASES)
@pytest.mark.parametrize("layout", ["separate", "in_place", "unaligned"])
def test_allgather_parity(K, S, layout):
    dev = H.device()
    N = K * S
    rng = np.random.default_rng(K * 100 + S)
    shards = [rng.integers(0, 65536, S, dtype=np.uint16) for _ in range(K)]
    if layout == "in_place":
        out = [torch.zeros(N, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        src = []
        for j in range(K):
            out[j][j * S:(j + 1) * S].copy_(syn.bits_to_bf16(shards[j]).to(dev))
            src.append(out[j][j * S:(j + 1) * S])
    else:
        off = 1 if layout == "unaligned" else 0
        src = _upload(shards, dev, off)
        bases = [torch.zeros(N + 8, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        out = [b[off:off + N] for b in bases]
    dpr.dpr_allgather(src, K, N, out)
    want, _ = ring.allgather(shards, K)
    for r in range(K):
        H.assert_bf16_equal(H.bits(out[r]), want[r], f"replica {r}")


def test_allreduce_identity_with_reduce_scatter():
    """AllReduce = ReduceScatter + AllGather on the device: the all-reduce
    replicas equal bf16(reduce-scatter shards) gathered."""
    dev = H.device()
    K, S = 8, 4096
    N = K * S
    x = _upload(_inputs(K, 1, N, 42, "gauss"), dev)
    for mode in H.MODES:
        sh = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
        dpr.dpr_reduce_scatter(x, K, 1, N, sh, mode=mode)
        sh16 = [s.to(torch.bfloat16) for s in sh]
        ag = [torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        dpr.dpr_allgather(sh16, K, N, ag)
        ar = [torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        dpr.dpr_allreduce(x, K, N, ar, mode=mode)
        for r in range(K):
            assert torch.equal(ar[r].view(torch.int16), ag[r].view(torch.int16))


def test_non_default_stream_and_repeatability():
    dev = H.device()
    K, S = 8, 8008
    N = K * S
    x = _upload(_inputs(K, 2, N, 3, "gauss"), dev)
    s = torch.cuda.Stream()
    outs = []
    for _ in range(2):
        o = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
        with torch.cuda.stream(s):
            dpr.dpr_reduce_scatter(x, K, 2, N, o, mode=ring.HOP_BF16)
        s.synchronize()
        outs.append(o)
    for j in range(K):
        assert torch.equal(outs[0][j], outs[1][j])


def test_binding_rejects_short_tensors():
    dev = H.device()
    x = [torch.empty(64, dtype=torch.bfloat16, device=dev) for _ in range(4)]
    out = [torch.empty(8, dtype=torch.float32, device=dev) for _ in range(4)]   # need 16
    with pytest.raises(ValueError):
        dpr.dpr_reduce_scatter(x, 4, 1, 64, out)
    with pytest.raises(dpr.DprError):
        dpr.dpr_reduce_scatter(x, 4, 1, 64, [x[0].float()[:16]] * 4)   # outputs alias
