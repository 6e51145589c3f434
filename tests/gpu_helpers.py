"""Shared pieces of the GPU parity tests: device buffers from the seeded
generator, the oracle evaluated on sampled element positions, and every
element of a reduce-scatter against the oracle's C ring simulation.

A reduce-scatter's result at position t of chunk j depends only on the K (x M)
inputs at element j*S + t and on j (which fixes the ring order).  So the
oracle can be run on a sub-problem made of the same positions T of every
chunk (N' = K*|T| per rank): its shard j is the full problem's shard j at T.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from oracle import ring
from oracle import ring_c
from workloads import synthetic as syn

MODES = (ring.RING_FP32, ring.HOP_BF16)


def device():
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from gradient_reduction_gb300 import build
    build.build()
    return torch.device("cuda", 0)


def bits(t: torch.Tensor) -> np.ndarray:
    return syn.bf16_bits(t)


def f32_bits(t) -> np.ndarray:
    a = t.detach().cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def assert_f32_equal(got, want, what=""):
    """Bit equality, except that any NaN matches any NaN (payloads differ
    between the GPU's and the oracle's canonical NaN)."""
    g, w = np.asarray(got, np.float32), np.asarray(want, np.float32)
    assert g.shape == w.shape, what
    nan = np.isnan(w)
    assert np.array_equal(np.isnan(g), nan), f"{what}: NaN positions differ"
    ok = f32_bits(g)[~nan] == f32_bits(w)[~nan]
    if not ok.all():
        i = int(np.flatnonzero(~ok)[0])
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} differ; first at "
                             f"{i}: got {g[~nan][i]!r} want {w[~nan][i]!r}")


def assert_bf16_equal(got_bits, want_bits, what=""):
    g, w = np.asarray(got_bits, np.uint16), np.asarray(want_bits, np.uint16)
    assert g.shape == w.shape, what
    gn = (g & 0x7FFF) > 0x7F80
    wn = (w & 0x7FFF) > 0x7F80
    assert np.array_equal(gn, wn), f"{what}: NaN positions differ"
    ok = g[~wn] == w[~wn]
    if not ok.all():
        i = int(np.flatnonzero(~ok)[0])
        raise AssertionError(f"{what}: {int((~ok).sum())} of {ok.size} differ; first at "
                             f"{i}: got {hex(g[~wn][i])} want {hex(w[~wn][i])}")


def sample_positions(S: int, w: int, seed: int) -> np.ndarray:
    """Positions inside a chunk: the first and last w, and w random ones."""
    rng = np.random.default_rng(seed)
    w = min(w, S)
    pos = set(range(w)) | set(range(S - w, S))
    pos |= set(int(x) for x in rng.integers(0, S, w))
    return np.array(sorted(pos), dtype=np.int64)


def chunk_positions(K: int, S: int, T: np.ndarray) -> np.ndarray:
    """Element indices c*S + T for every chunk c, chunk by chunk."""
    return np.concatenate([c * S + T for c in range(K)]).astype(np.int64)


def gather_inputs(at_fn, K: int, M: int, S: int, T: np.ndarray) -> list:
    """Host inputs of the sampled sub-problem: x[m*K + r] = rank r's micro m
    buffer at c*S + T for every chunk c.  at_fn(rank, micro, idx) -> bf16
    tensor of the generator's values at those element indices."""
    idx = chunk_positions(K, S, T)
    return [bits(at_fn(r, m, idx)) for m in range(M) for r in range(K)]


def oracle_rs_sampled(at_fn, K: int, M: int, S: int, T: np.ndarray, mode: int, scale: float,
                      out_init=None, x=None):
    """Oracle reduce-scatter on positions T of every chunk.  Returns K float32
    arrays of |T|."""
    if x is None:
        x = gather_inputs(at_fn, K, M, S, T)
    shards, _ = ring.reduce_scatter(x, K, M, mode, scale, out_init=out_init)
    return shards


def oracle_ar_sampled(at_fn, K: int, S: int, T: np.ndarray, mode: int, scale: float, x=None):
    if x is None:
        x = gather_inputs(at_fn, K, 1, S, T)
    outs, _ = ring.allreduce(x[:K], K, mode, scale)
    return outs           # each: K chunks of |T|, chunk by chunk


# ---- guard bytes ------------------------------------------------------------------

PAT = 0xA5
GAP = 768


class Arena:
    """Buffers carved out of one uint8 device allocation filled with PAT."""

    def __init__(self):
        self.specs = []       # (byte offset, element count, dtype)
        self.size = GAP

    def add(self, n: int, dtype, shift: int = 0) -> int:
        off = (self.size + GAP + 255) // 256 * 256 + shift
        self.specs.append((off, n, dtype))
        self.size = off + n * torch.tensor([], dtype=dtype).element_size()
        return len(self.specs) - 1

    def build(self, dev):
        self.buf = torch.full((self.size + GAP,), PAT, dtype=torch.uint8, device=dev)
        self.views = [self.buf[off:off + n * torch.tensor([], dtype=dt).element_size()].view(dt)
                      for off, n, dt in self.specs]
        return self.views

    def snapshot(self):
        torch.cuda.synchronize()
        self.before = self.buf.cpu().numpy().copy()

    def check_untouched(self, written):
        """written: list of (buffer index, first element, element count)."""
        torch.cuda.synchronize()
        after = self.buf.cpu().numpy()
        free = np.ones(after.size, bool)
        for i, e0, n in written:
            off, _, dt = self.specs[i]
            es = torch.tensor([], dtype=dt).element_size()
            free[off + e0 * es: off + (e0 + n) * es] = False
        bad = np.flatnonzero(free & (after != self.before))
        assert bad.size == 0, f"{bad.size} bytes outside the written regions changed, first at {bad[0]}"


def assert_rs_every_element(x, out, K: int, M: int, mode: int, scale: float, what=""):
    """Every element of a reduce-scatter's K fp32 shards against the oracle's C
    ring simulation run on the same inputs, copied from the device (x[m*K + r]
    bf16 of N, out[j] fp32 of N/K)."""
    torch.cuda.synchronize()
    host_x = [bits(t) for t in x]
    want, _ = ring_c.reduce_scatter(host_x, K, M, mode, scale)
    for j in range(K):
        assert_f32_equal(out[j].cpu().numpy(), want[j], f"{what} shard {j}")
