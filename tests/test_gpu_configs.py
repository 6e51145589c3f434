"""The five workload configurations at their full sizes, through the C ABI.

Results are compared with the oracle on sampled positions of every chunk (the
first, last and random positions; the oracle runs the same ring on those
positions of every rank); the reduce-scatters of configurations 2 and 3 (56
tensors), and of every sweep point with at most 2 GiB of inputs, also at every
element, against the oracle's C ring simulation on the inputs copied back from
the device.  Every element is also checked with
properties that hold at any size: the reduce-scatter's error bound against the exact
fp64 sum, all-gather replicas identical to the concatenated shards, flat
buckets identical to the concatenated gradients.  Inputs are generated on the
GPU by the seeded generator; the tests also check that the device-generated
bytes equal the host-generated ones at the sampled positions."""
import gc

import numpy as np
import pytest
import torch

import gradient_reduction_gb300 as dpr
from oracle import flatten as ofl
from oracle import ring
from tests import gpu_helpers as H
from workloads import configs as C

pytestmark = pytest.mark.gpu


def _free_gib():
    free, _ = torch.cuda.mem_get_info()
    return free / 2 ** 30


def _release():
    gc.collect()
    torch.cuda.empty_cache()


def _check_device_inputs(x, at_fn, K, M, S, T):
    """Device-generated inputs equal host-generated ones at c*S + T."""
    idx = H.chunk_positions(K, S, T)
    didx = torch.from_numpy(idx).to(x[0].device)
    for m in range(M):
        for r in (0, K - 1):
            dev_bits = H.bits(x[m * K + r].index_select(0, didx))
            host = H.bits(at_fn(r, m, idx))
            assert np.array_equal(dev_bits, host), f"generator mismatch rank {r} micro {m}"


def _check_rs_sampled(out, at_fn, K, M, S, mode, scale, seed, w=64, x=None):
    T = H.sample_positions(S, w, seed)
    want = H.oracle_rs_sampled(at_fn, K, M, S, T, mode, scale, x=x)
    idx = torch.from_numpy(T).to(out[0].device)
    for j in range(K):
        got = out[j].index_select(0, idx).cpu().numpy()
        H.assert_f32_equal(got, want[j], f"shard {j}")
    return T


def _rs_error_bound(x, out, K, M, S, mode):
    """|K*out - exact| <= gamma_{K-1} * sum|x| element-wise (M == 1; scale 1/K
    a power of two, so K*out is the landed sum exactly)."""
    u = 2.0 ** -24 if mode == ring.RING_FP32 else 2.0 ** -8
    gamma = (K - 1) * u / (1 - (K - 1) * u)
    for j in range(K):
        sl = slice(j * S, (j + 1) * S)
        xs = torch.stack([x[r][sl].double() for r in range(K)])
        exact = xs.sum(0)
        bound = gamma * xs.abs().sum(0)
        err = (out[j].double() * K - exact).abs()
        assert bool((err <= bound).all()), f"error bound violated in chunk {j}"
        del xs, exact, bound, err


# ---- config 2: K=8, one 25,000,000-element bucket, 1% outliers ----------------------

@pytest.mark.parametrize("mode", H.MODES)
def test_cfg2_reduce_scatter(mode):
    dev = H.device()
    cfg = C.CFG2
    K, N = cfg.K, cfg.N
    S = N // K
    x = [cfg.buffer(r, 0, device=dev) for r in range(K)]
    out = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
    dpr.dpr_reduce_scatter(x, K, 1, N, out, mode=mode, scale=1.0 / K)
    torch.cuda.synchronize()
    T = _check_rs_sampled(out, cfg.at, K, 1, S, mode, 1.0 / K, seed=2 + mode)
    _check_device_inputs(x, cfg.at, K, 1, S, T)
    _rs_error_bound(x, out, K, 1, S, mode)
    # every element, against the C ring simulation on the same 400 MB of inputs
    H.assert_rs_every_element(x, out, K, 1, mode, 1.0 / K, "cfg2")


# ---- config 3: fragmented transformer gradients, flatten + reduce-scatter -----------

def _bucket_at_fn(cfg, bk):
    """at(rank, micro, idx) over a bucket's element indices: the generator's
    value of the gradient stored there, zero in the padding."""
    numels = [cfg.arrival_order()[p][2] for p in bk.params]

    def at(rank, _m, idx):
        idx = np.asarray(idx, dtype=np.int64)
        out = torch.zeros(len(idx), dtype=torch.bfloat16)
        for p, o, n in zip(bk.params, bk.offsets, numels):
            sel = np.flatnonzero((idx >= o) & (idx < o + n))
            if len(sel):
                out[torch.from_numpy(sel)] = cfg.grad_at(rank, p, idx[sel] - o)
        return out
    return at


def _run_cfg3(cfg, mode, check_buckets, every_element=False):
    dev = H.device()
    K = cfg.K
    arr = cfg.arrival_order()
    numel = [n for *_, n in arr]
    total = sum(numel)
    need = (total * 2 * K + total * 4) / 2 ** 30 + 2
    if _free_gib() < need:
        pytest.skip(f"needs {need:.0f} GiB free on the device")
    buckets = ofl.assign_buckets(numel, cfg.bucket_cap, pad_to=8 * K)
    grads = [[cfg.grad(r, p, device=dev) for p in range(len(arr))] for r in range(K)]
    part_len = sum(b.numel for b in buckets) // K
    partition = [torch.empty(part_len, dtype=torch.float32, device=dev) for _ in range(K)]
    ipg = [torch.zeros(max(b.numel for b in buckets), dtype=torch.bfloat16, device=dev)
           for _ in range(K)]
    plans = [dpr.dpr_flatten_plan_create([[grads[r][p] for p in b.params] for r in range(K)],
                                         [numel[p] for p in b.params], b.offsets, b.numel)
             for b in buckets]
    shard_off = 0
    for bi, (b, plan) in enumerate(zip(buckets, plans)):
        S = b.numel // K
        views = [t[:b.numel] for t in ipg]
        dpr.dpr_flatten_bucket(plan, views)
        # the flat bucket is the gradients laid end to end (every element)
        for r in range(K):
            for p, o in zip(b.params, b.offsets):
                assert torch.equal(views[r][o:o + numel[p]], grads[r][p].view(-1))
        out = [partition[j][shard_off:shard_off + S] for j in range(K)]
        dpr.dpr_reduce_scatter(views, K, 1, b.numel, out, mode=mode, scale=1.0 / K)
        if bi in check_buckets:
            torch.cuda.synchronize()
            _check_rs_sampled(out, _bucket_at_fn(cfg, b), K, 1, S, mode, 1.0 / K,
                              seed=bi, w=32)
        if every_element:
            # the whole bucket, against the C ring simulation on the gathered
            # bucket (equal to the gradients laid end to end, checked above)
            H.assert_rs_every_element(views, out, K, 1, mode, 1.0 / K, f"bucket {bi}")
        shard_off += S
    torch.cuda.synchronize()
    for p in plans:
        p.close()
    del grads, partition, ipg
    _release()


@pytest.mark.parametrize("mode", H.MODES)
def test_cfg3_flatten_reduce_scatter_56_tensors(mode):
    _run_cfg3(C.CFG3, mode, check_buckets={0, 1, 2, 5, 20, 41}, every_element=True)


def test_cfg3_flatten_reduce_scatter_224_tensors():
    _run_cfg3(C.CFG3_224, ring.RING_FP32, check_buckets={0, 3, 100, 167})


# ---- config 4: parameter all-gather of one hidden-8192 layer ------------------------

def test_cfg4_allgather():
    dev = H.device()
    K, N = C.CFG4.K, C.CFG4.N
    S = N // K
    shards = [C.cfg4_shard(j, device=dev) for j in range(K)]
    out = [torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(K)]
    dpr.dpr_allgather(shards, K, N, out)
    torch.cuda.synchronize()
    full = torch.cat(shards)
    for r in range(K):
        assert torch.equal(out[r].view(torch.int16), full.view(torch.int16)), f"replica {r}"
    del full
    T = H.sample_positions(S, 128, 4)
    shard_bits = [H.bits(C.cfg4_at(j * S + T)) for j in range(K)]
    want, _ = ring.allgather(shard_bits, K)
    idx = torch.from_numpy(np.concatenate([c * S + T for c in range(K)])).to(dev)
    for r in range(K):
        H.assert_bf16_equal(H.bits(out[r].index_select(0, idx)), want[r], f"replica {r}")
    del shards, out
    _release()


# ---- config 5: the sweep ------------------------------------------------------------

def _sweep_point(K, nbytes, dev, check_ag_ar):
    cfg = C.cfg5(K, nbytes)
    N, M = cfg.N, cfg.M
    S = N // K
    need = (M * K * N * 2 + N * 4 + (K * N * 4 if check_ag_ar else 0)) / 2 ** 30 + 1
    if _free_gib() < need:
        return f"skipped K={K} {nbytes} B: needs {need:.0f} GiB"
    x = [cfg.buffer(r, m, device=dev) for m in range(M) for r in range(K)]
    out = [torch.empty(S, dtype=torch.float32, device=dev) for _ in range(K)]
    T = H.sample_positions(S, 16, K + nbytes)
    xh = H.gather_inputs(cfg.at, K, M, S, T)
    every = M * K * nbytes <= (2 << 30)      # inputs the host oracle takes whole
    for mode in H.MODES:
        dpr.dpr_reduce_scatter(x, K, M, N, out, mode=mode, scale=1.0 / K)
        torch.cuda.synchronize()
        _check_rs_sampled(out, cfg.at, K, M, S, mode, 1.0 / K, seed=K + nbytes, w=16, x=xh)
        if every:
            H.assert_rs_every_element(x, out, K, M, mode, 1.0 / K, f"K={K} {nbytes} B")
    _check_device_inputs(x, cfg.at, K, M, S, T)
    if check_ag_ar:
        ar = [torch.empty(N, dtype=torch.bfloat16, device=dev) for _ in range(K)]
        for mode in H.MODES:
            dpr.dpr_allreduce(x[:K], K, N, ar, mode=mode, scale=1.0 / K)
            torch.cuda.synchronize()
            want = H.oracle_ar_sampled(cfg.at, K, S, T, mode, 1.0 / K, x=xh)
            idx = torch.from_numpy(np.concatenate([c * S + T for c in range(K)])).to(dev)
            for r in (0, K // 2, K - 1):
                H.assert_bf16_equal(H.bits(ar[r].index_select(0, idx)), want[r], f"AR {r}")
            for r in range(1, K):
                assert torch.equal(ar[r].view(torch.int16), ar[0].view(torch.int16))
        sh = [x[j][:S] for j in range(K)]
        dpr.dpr_allgather(sh, K, N, ar)
        torch.cuda.synchronize()
        full = torch.cat(sh)
        for r in range(K):
            assert torch.equal(ar[r].view(torch.int16), full.view(torch.int16))
        del ar, full
    del x, out
    _release()
    return None


@pytest.mark.parametrize("K", [2, 4, 8, 16, 64])
def test_cfg5_sweep(K):
    dev = H.device()
    skipped = []
    for k, nbytes in C.cfg5_points():
        if k != K:
            continue
        msg = _sweep_point(K, nbytes, dev, check_ag_ar=nbytes <= (1 << 28))
        if msg:
            skipped.append(msg)
    if skipped:
        print("\n".join(skipped))
    assert len(skipped) <= 1
