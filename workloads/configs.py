"""The workloads the tests and the bench run: shapes, sizes and value recipes.

Five configurations of the ZeRO gradient-bucket reduction, all with K
simulated data-parallel ranks held as K buffers in one GPU's memory:

  1  K=4, 4096 bf16 elements per rank ~ N(0, sigma=1e-2); plus the 4x4
     integer-valued ring worked example.
  2  K=8, one contiguous 25,000,000-element bucket per rank (50 MB),
     ~ N(0, 1e-3) with 1% of the entries multiplied by 100.
  3  K=8, fragmented per-parameter gradients of a 7-layer, hidden-4096
     transformer (q/k/v/o 4096x4096, MLP 4096x11008 and 11008x4096, two
     4096 norm vectors per layer = 56 tensors); a 28-layer variant has 224.
  4  K=8, all-gather of one hidden-8192 layer's parameters, U(-0.02, 0.02).
  5  sweep over K in {2,4,8,16,64} and per-rank buckets of 1 KiB .. 1 GiB in
     steps of 4x, both summation modes, 2 micro-batches accumulated.

and the bench workload (K=8, a 1 GiB bucket per rank built from 32
fragmented 4096x4096 gradients).

sigma is read as a standard deviation.  Values come from workloads.synthetic.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

from . import synthetic as syn

BASE_SEED = 0x5EED0000


@dataclass(frozen=True)
class Dist:
    kind: str                 # "gauss" | "uniform"
    scale: float              # sigma for gauss, amplitude for uniform
    outlier_frac: float = 0.0
    outlier_mult: float = 100.0

    def fill(self, start: int, count: int, key: int, device="cpu", out=None) -> torch.Tensor:
        if self.kind == "gauss":
            return syn.gauss_bf16(start, count, key, self.scale, self.outlier_frac,
                                  self.outlier_mult, device=device, out=out)
        if self.kind == "uniform":
            return syn.uniform_bf16(start, count, key, self.scale, device=device, out=out)
        raise ValueError(self.kind)

    def at(self, idx, key: int) -> torch.Tensor:
        """Host values at arbitrary element indices of the stream `key`."""
        if self.kind == "gauss":
            return syn.gauss_bf16_at(idx, key, self.scale, self.outlier_frac, self.outlier_mult)
        if self.kind == "uniform":
            return syn.uniform_bf16_at(idx, key, self.scale)
        raise ValueError(self.kind)


@dataclass(frozen=True)
class Flat:
    """K contiguous rank buckets of N bf16 elements each, M micro-batches."""
    name: str
    cid: int
    K: int
    N: int
    dist: Dist
    M: int = 1

    @property
    def seed(self) -> int:
        return BASE_SEED + self.cid

    def key(self, rank: int, micro: int = 0) -> int:
        return syn.stream_key(self.seed, rank, micro, tag=self.N & 0xFFFFFFFF)

    def slab(self, rank: int, micro: int, start: int, count: int, device="cpu", out=None):
        """Elements [start, start+count) of rank `rank`'s micro-batch `micro` buffer."""
        return self.dist.fill(start, count, self.key(rank, micro), device=device, out=out)

    def at(self, rank: int, micro: int, idx) -> torch.Tensor:
        """Host values of rank `rank`'s micro-batch `micro` buffer at indices idx."""
        return self.dist.at(idx, self.key(rank, micro))

    def buffer(self, rank: int, micro: int = 0, device="cpu", out=None):
        return self.slab(rank, micro, 0, self.N, device=device, out=out)


CFG1 = Flat("cfg1_k4_4096", 1, K=4, N=4096, dist=Dist("gauss", 1e-2))
CFG2 = Flat("cfg2_k8_25M", 2, K=8, N=25_000_000, dist=Dist("gauss", 1e-3, 0.01, 100.0))


def cfg5_points():
    """(K, bytes per rank) of the sweep: K in {2,4,8,16,64}, 1 KiB .. 1 GiB by 4x."""
    pts = []
    for K in (2, 4, 8, 16, 64):
        for i in range(11):
            pts.append((K, 1024 * 4 ** i))
    return pts


def cfg5(K: int, nbytes: int) -> Flat:
    return Flat(f"cfg5_k{K}_{nbytes}B", 5, K=K, N=nbytes // 2, dist=Dist("gauss", 1e-3), M=2)


# --- config 3: fragmented transformer gradients ---------------------------------

def transformer_layer(hidden: int = 4096, ffn: int = 11008):
    """One layer's parameter tensors in forward order (name, shape)."""
    return [("norm1", (hidden,)),
            ("q", (hidden, hidden)), ("k", (hidden, hidden)),
            ("v", (hidden, hidden)), ("o", (hidden, hidden)),
            ("norm2", (hidden,)),
            ("fc1", (hidden, ffn)), ("fc2", (ffn, hidden))]


@dataclass(frozen=True)
class Fragmented:
    """K ranks, each holding P separately allocated bf16 gradients."""
    name: str
    cid: int
    K: int
    layers: int
    dist: Dist
    bucket_cap: int = 25_000_000
    hidden: int = 4096
    ffn: int = 11008

    @property
    def seed(self) -> int:
        return BASE_SEED + self.cid

    def params_forward(self):
        out = []
        for layer in range(self.layers):
            for nm, shp in transformer_layer(self.hidden, self.ffn):
                n = 1
                for d in shp:
                    n *= d
                out.append((f"layer{layer}.{nm}", shp, n))
        return out

    def arrival_order(self):
        """Parameters in gradient-arrival order: backward visits the last layer
        first, so arrival is the reverse of forward order."""
        return list(reversed(self.params_forward()))

    def key(self, rank: int, p: int) -> int:
        return syn.stream_key(self.seed, rank, 0, tag=p)

    def grad(self, rank: int, p: int, device="cpu", out=None):
        """Gradient of parameter p (index in arrival order) on rank `rank`."""
        n = self.arrival_order()[p][2]
        return self.dist.fill(0, n, self.key(rank, p), device=device, out=out)

    def grad_slab(self, rank: int, p: int, start: int, count: int, device="cpu"):
        return self.dist.fill(start, count, self.key(rank, p), device=device)

    def grad_at(self, rank: int, p: int, idx) -> torch.Tensor:
        return self.dist.at(idx, self.key(rank, p))


CFG3 = Fragmented("cfg3_7layer_h4096", 3, K=8, layers=7, dist=Dist("gauss", 1e-3))
CFG3_224 = Fragmented("cfg3_28layer_h4096_224t", 3, K=8, layers=28, dist=Dist("gauss", 1e-3))


# --- config 4: parameter all-gather of one hidden-8192 layer --------------------

CFG4_SHAPES = [("qkv", (8192, 24576)), ("out", (8192, 8192)),
               ("mlp_a", (8192, 28672)), ("mlp_b", (8192, 28672)), ("mlp_c", (28672, 8192))]
CFG4_N = sum(a * b for _, (a, b) in CFG4_SHAPES)          # 973,078,528
CFG4 = Flat("cfg4_k8_h8192_layer", 4, K=8, N=CFG4_N, dist=Dist("uniform", 0.02))


def cfg4_shard(j: int, device="cpu", out=None):
    """Shard j (of K=8) of the concatenated layer parameters: elements
    [j*S, (j+1)*S) of one flat stream, S = N/8."""
    S = CFG4.N // CFG4.K
    return CFG4.dist.fill(j * S, S, syn.stream_key(CFG4.seed, 0, 0, 0), device=device, out=out)


def cfg4_slab(start: int, count: int, device="cpu"):
    return CFG4.dist.fill(start, count, syn.stream_key(CFG4.seed, 0, 0, 0), device=device)


def cfg4_at(idx) -> torch.Tensor:
    return CFG4.dist.at(idx, syn.stream_key(CFG4.seed, 0, 0, 0))


# --- bench workload -------------------------------------------------------------

@dataclass(frozen=True)
class BenchWorkload:
    """K=8 ranks, one 1 GiB bf16 bucket per rank (N = 2**29), filled from 32
    fragmented 4096x4096 gradients per rank; a second, already-flat micro-batch
    bucket; fp32 partition shards; bf16 parameter shards for the all-gather."""
    name: str = "zero_bucket_k8_1GiB"
    K: int = 8
    N: int = 1 << 29
    frag_shape: tuple = (4096, 4096)
    n_frag: int = 32
    dist: Dist = field(default_factory=lambda: Dist("gauss", 1e-3))
    param_dist: Dist = field(default_factory=lambda: Dist("uniform", 0.02))
    seed: int = BASE_SEED + 6

    @property
    def frag_numel(self) -> int:
        return self.frag_shape[0] * self.frag_shape[1]

    def frag_key(self, rank: int, p: int) -> int:
        return syn.stream_key(self.seed, rank, 1, tag=p)

    def micro0_key(self, rank: int) -> int:
        return syn.stream_key(self.seed, rank, 0, tag=0xB0)

    def param_key(self) -> int:
        return syn.stream_key(self.seed, 0, 0, tag=0xA6)

    def prev_grad_key(self, j: int) -> int:
        return syn.stream_key(self.seed, j, 2, tag=0xF3)


BENCH = BenchWorkload()
