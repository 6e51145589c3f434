"""Seeded, counter-based synthetic gradients and parameters.

This module is shared by the CPU oracle side and the CUDA side of the tests and
the bench, so it holds none of the reduction's arithmetic: it only turns
(seed, stream, element index) into bf16 values.

Every value is a pure function of its element index and a 32-bit stream key,
so any element range of any rank buffer can be regenerated on its own
("slab-addressable"), and a slab generated on the host is bit-identical to the
same slab generated on a GPU.  Bit-identity holds because the recipe uses only
  * 64-bit integer arithmetic whose intermediates never exceed 2**63
    (32-bit multiplies are split into 16-bit halves),
  * one exact int -> fp32 conversion (|z| < 2**24),
  * one or two IEEE fp32 multiplies (correctly rounded on every device), and
  * PyTorch's fp32 -> bf16 conversion, round-to-nearest-even on CPU and CUDA.

Distributions
  gauss:   centred Irwin-Hall sum of four 16-bit uniforms, scaled to standard
           deviation sigma (a bounded, bell-shaped stand-in for N(0, sigma));
           optionally a fraction of the entries multiplied by an outlier factor.
  uniform: 24-bit uniform integer scaled onto [-amp, amp).
  integer: small integer-valued buffers for worked examples.

The hash is MurmurHash3's 32-bit finaliser (fmix32), applied to the element
index and a per-stream key.
"""
from __future__ import annotations

import math

import numpy as np
import torch

M32 = 0xFFFFFFFF
_CHUNK_CPU = 1 << 16     # keeps the int64 temporaries cache-resident on a host
_CHUNK_GPU = 1 << 26


def _chunk(device) -> int:
    return _CHUNK_CPU if torch.device(device).type == "cpu" else _CHUNK_GPU


# fixed odd constants that separate the three words drawn per element
_W0, _W1, _W2 = 0x68E31DA4, 0xB5297A4D, 0x1B56C4E9


def fmix32_int(h: int) -> int:
    """MurmurHash3 fmix32 on a Python int (used to derive stream keys)."""
    h &= M32
    h ^= h >> 16
    h = (h * 0x85EBCA6B) & M32
    h ^= h >> 13
    h = (h * 0xC2B2AE35) & M32
    h ^= h >> 16
    return h


def _mul32(a: torch.Tensor, c: int) -> torch.Tensor:
    """(a * c) mod 2**32 for int64 tensors holding values in [0, 2**32).

    The multiply is split into 16-bit halves so that no int64 product exceeds
    2**48 (no signed overflow on any backend)."""
    lo = a & 0xFFFF
    hi = a >> 16
    return (lo * c + (((hi * c) & 0xFFFF) << 16)) & M32


def _fmix32(h: torch.Tensor) -> torch.Tensor:
    h = h ^ (h >> 16)
    h = _mul32(h, 0x85EBCA6B)
    h = h ^ (h >> 13)
    h = _mul32(h, 0xC2B2AE35)
    h = h ^ (h >> 16)
    return h


def stream_key(seed: int, rank: int, micro: int = 0, tag: int = 0) -> int:
    """32-bit key of one rank buffer (one rank, one micro-batch, one tensor)."""
    k = fmix32_int(seed & M32)
    k = fmix32_int(k ^ ((rank * 0x9E3779B1) & M32))
    k = fmix32_int(k ^ ((micro * 0x85EBCA77) & M32))
    k = fmix32_int(k ^ ((tag * 0xC2B2AE3D) & M32))
    return k


def _words(start: int, count: int, key: int, device) -> tuple:
    return _words_at(torch.arange(start, start + count, dtype=torch.int64, device=device), key)


def _words_at(idx: torch.Tensor, key: int) -> tuple:
    lo = idx & M32
    hi = idx >> 32
    base = _fmix32(_fmix32(lo ^ key) ^ _mul32(hi, 0x27D4EB2F) ^ fmix32_int(key ^ 0x5BD1E995))
    return _fmix32(base ^ _W0), _fmix32(base ^ _W1), _fmix32(base ^ _W2)


# standard deviation of the sum of four independent uniforms on {0..65535}
_IRWIN_HALL4_STD = math.sqrt(4.0 * (65536.0 ** 2 - 1.0) / 12.0)
_IRWIN_HALL4_MEAN = 2 * 65535


def gauss_bf16(start: int, count: int, key: int, sigma: float,
               outlier_frac: float = 0.0, outlier_mult: float = 100.0,
               device="cpu", out: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 values of elements [start, start+count) of the stream `key`."""
    if out is None:
        out = torch.empty(count, dtype=torch.bfloat16, device=device)
    step = _chunk(device)
    for s in range(0, count, step):
        n = min(step, count - s)
        w0, w1, w2 = _words(start + s, n, key, device)
        out[s:s + n] = _gauss_from_words(w0, w1, w2, sigma, outlier_frac, outlier_mult, device)
    return out


def _gauss_from_words(w0, w1, w2, sigma, outlier_frac, outlier_mult, device):
    scale = torch.tensor(float(np.float32(sigma / _IRWIN_HALL4_STD)), dtype=torch.float32,
                         device=device)
    z = (w0 & 0xFFFF) + (w0 >> 16) + (w1 & 0xFFFF) + (w1 >> 16) - _IRWIN_HALL4_MEAN
    x = z.to(torch.float32) * scale
    thresh = int(outlier_frac * 4294967296.0)
    if thresh > 0:
        mult = torch.tensor(float(np.float32(outlier_mult)), dtype=torch.float32, device=device)
        x = torch.where(w2 < thresh, x * mult, x)
    return x.to(torch.bfloat16)


def gauss_bf16_at(idx, key: int, sigma: float, outlier_frac: float = 0.0,
                  outlier_mult: float = 100.0) -> torch.Tensor:
    """gauss_bf16 evaluated at arbitrary element indices (host)."""
    idx = torch.as_tensor(np.asarray(idx, dtype=np.int64))
    w0, w1, w2 = _words_at(idx, key)
    return _gauss_from_words(w0, w1, w2, sigma, outlier_frac, outlier_mult, "cpu")


def _uniform_from_word(w0, amp, device):
    scale = torch.tensor(float(np.float32(amp)) * 2.0 ** -23, dtype=torch.float32, device=device)
    return (((w0 >> 8) - (1 << 23)).to(torch.float32) * scale).to(torch.bfloat16)


def uniform_bf16_at(idx, key: int, amp: float) -> torch.Tensor:
    """uniform_bf16 evaluated at arbitrary element indices (host)."""
    idx = torch.as_tensor(np.asarray(idx, dtype=np.int64))
    w0, _, _ = _words_at(idx, key)
    return _uniform_from_word(w0, amp, "cpu")


def uniform_bf16(start: int, count: int, key: int, amp: float, device="cpu",
                 out: torch.Tensor | None = None) -> torch.Tensor:
    """bf16 values on [-amp, amp) of elements [start, start+count) of stream `key`."""
    if out is None:
        out = torch.empty(count, dtype=torch.bfloat16, device=device)
    step = _chunk(device)
    for s in range(0, count, step):
        n = min(step, count - s)
        w0, _, _ = _words(start + s, n, key, device)
        out[s:s + n] = _uniform_from_word(w0, amp, device)
    return out


def integer_example(K: int, N: int, device="cpu") -> list:
    """Integer-valued rank buffers x_r[c*S + t] = (c + 1) * 2**r for the ring
    worked examples: every partial sum (c + 1) * (sum of 2**r over the ranks
    that contributed) is exact in bf16 and fp32 while (c + 1) * (2**K - 1) < 256,
    and the contributor set can be read back from the value."""
    S = N // K
    bufs = []
    for r in range(K):
        c = torch.arange(N, device=device) // S
        bufs.append(((c + 1) * (2 ** r)).to(torch.bfloat16))
    return bufs


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Host copy of a bf16 tensor as a numpy uint16 array of its bit patterns."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits_to_bf16(a: np.ndarray) -> torch.Tensor:
    """Inverse of bf16_bits (a CPU bf16 tensor sharing no memory with `a`)."""
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16).copy()).view(torch.bfloat16)
