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
  * exact integer -> float conversions and exact bit manipulations,
  * IEEE double and fp32 additions, multiplications, tensor-by-tensor
    divisions and square roots, each a separate, correctly rounded operation
    on every device (no fused multiply-add, no library transcendental), and
  * PyTorch's fp64 -> fp32 and fp32 -> bf16 conversions, round-to-nearest-even
    on CPU and CUDA.

Distributions
  gauss:   N(0, sigma) by the Box-Muller transform (Box and Muller, 1958) in
           IEEE double precision: two 32-bit hash words give u1 in (0, 1] and
           u2 in [0, 1), and z = sqrt(-2 ln u1) cos(2 pi u2).  ln and cos are
           evaluated here by series (ln m = 2 atanh((m-1)/(m+1)) after an
           exact split u1 = m 2^e; cos by octant reduction done exactly on the
           integer word and Taylor polynomials on [0, pi/4]) using only
           additions, multiplications, one tensor-by-tensor division and one
           square root, each correctly rounded on every device, so a host slab
           and a GPU slab are bit-identical.  |z| <= sqrt(64 ln 2) = 6.66, so
           the tails beyond 6.66 sigma (probability 3e-11) are cut.  x = sigma z
           is rounded to fp32, optionally a fraction of the entries is
           multiplied by an outlier factor in fp32, and the result is rounded
           to bf16.
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


_LN2 = math.log(2.0)
_PI_4 = math.pi / 4.0
_SQRT2 = math.sqrt(2.0)
# ln m = 2 (z + z^3/3 + z^5/5 + ...), z = (m-1)/(m+1), |z| <= 0.1716 on
# [1/sqrt2, sqrt2]: 12 terms leave a truncation below 2^-60
_ATANH_C = [1.0 / (2 * k + 1) for k in range(12)]
# Taylor coefficients of sin(x)/x and cos(x) in x^2, to x^18 / x^20: on
# [0, pi/4] the first omitted term is below 2^-65
_SIN_C = [(-1.0) ** k / math.factorial(2 * k + 1) for k in range(10)]
_COS_C = [(-1.0) ** k / math.factorial(2 * k) for k in range(11)]


def _horner(c, x2):
    """sum_k c[k] x2^k by Horner's rule: one multiply and one add per step."""
    acc = torch.full_like(x2, c[-1])
    for ck in reversed(c[:-1]):
        acc = acc * x2 + ck
    return acc


def _ln_u1(w0: torch.Tensor) -> torch.Tensor:
    """ln(u1) in double, u1 = (w0 + 1) 2^-32 in (0, 1], for int64 words w0 in
    [0, 2^32).  n = w0 + 1 is split exactly as n = m 2^e with m in
    [1/sqrt2, sqrt2) (from its double's exponent and mantissa bits), and
    ln u1 = (e - 32) ln 2 + 2 atanh((m-1)/(m+1))."""
    d = (w0 + 1).to(torch.float64)                    # exact: n <= 2^32
    b = d.view(torch.int64)
    e = (b >> 52) - 1023
    m = ((b & ((1 << 52) - 1)) | (1023 << 52)).view(torch.float64)   # [1, 2)
    big = m > _SQRT2
    m = torch.where(big, m * 0.5, m)                  # exact
    e = e + big.to(torch.int64)
    z = (m - 1.0) / (m + 1.0)
    z2 = z * z
    ln_m = (z * _horner(_ATANH_C, z2)) * 2.0
    return (e - 32).to(torch.float64) * _LN2 + ln_m


def _cos_2pi_u2(w1: torch.Tensor) -> torch.Tensor:
    """cos(2 pi u2) in double, u2 = w1 2^-32 in [0, 1), for int64 words w1 in
    [0, 2^32).  The octant o = w1 >> 29 and the fraction f in [0, 1) inside it
    are exact; theta = k pi/2 + s psi with psi in [0, pi/4]:
      even o: k = o/2,       s = +1, psi = f pi/4;
      odd o:  k = (o+1)/2,   s = -1, psi = (1 - f) pi/4;
    cos(k pi/2 + s psi) is cos psi, -s sin psi, -cos psi, s sin psi for
    k mod 4 = 0, 1, 2, 3."""
    o = w1 >> 29
    f = (w1 & ((1 << 29) - 1)).to(torch.float64) * (2.0 ** -29)     # exact
    odd = (o & 1) == 1
    psi = torch.where(odd, 1.0 - f, f) * _PI_4
    x2 = psi * psi
    sin_p = psi * _horner(_SIN_C, x2)
    cos_p = _horner(_COS_C, x2)
    k = ((o + 1) >> 1) & 3
    s = torch.where(odd, -1.0, 1.0).to(torch.float64)
    val = torch.where((k & 1) == 1, sin_p, cos_p)
    sign = torch.where(k == 0, 1.0, torch.where(k == 2, -1.0, torch.where(k == 1, -s, s)))
    return val * sign


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
    r = torch.sqrt(_ln_u1(w0) * -2.0)
    x = ((r * _cos_2pi_u2(w1)) * float(sigma)).to(torch.float32)
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
