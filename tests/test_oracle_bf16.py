"""Pins of the oracle's bf16 conversions against PyTorch's CPU bf16 conversion
(a library routine) and against exact rational rounding."""
import random

import numpy as np
import torch

from oracle import bf16 as obf
from tests import exact_fp as X


def _torch_bits(f32: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(f32.copy()).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def test_from_f32_every_upper_half_and_every_rounding_case():
    """All 65536 upper halves (sign, exponent, kept fraction bits) times the
    lower halves that decide the rounding: zero, just above zero, just below,
    at and just above the halfway point, the maximum, plus random ones."""
    rng = np.random.default_rng(0)
    lows = np.array([0x0000, 0x0001, 0x3FFF, 0x7FFE, 0x7FFF, 0x8000, 0x8001, 0xBFFF,
                     0xFFFE, 0xFFFF] + list(rng.integers(0, 65536, 6)), dtype=np.uint32)
    upper = np.arange(65536, dtype=np.uint32)
    bits = (upper[:, None] << 16 | lows[None, :]).reshape(-1)
    f = bits.view(np.float32)
    mine, ref = obf.from_f32(f), _torch_bits(f)
    nan = np.isnan(f)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.all(np.isnan(obf.to_f32(mine[nan])))
    assert np.all(mine[nan] == 0x7FC0)


def test_from_f32_random_sample():
    rng = np.random.default_rng(1)
    bits = rng.integers(0, 2 ** 32, 1 << 22, dtype=np.uint64).astype(np.uint32)
    f = bits.view(np.float32)
    nan = np.isnan(f)
    assert np.array_equal(obf.from_f32(f)[~nan], _torch_bits(f)[~nan])


def test_to_f32_is_exact_widening():
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(b.view(np.int16).copy()).view(torch.bfloat16).float().numpy()
    got = obf.to_f32(b)
    nan = np.isnan(ref)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))
    assert np.all(np.isnan(got[nan]))


def test_from_f32_special_values():
    f = np.array([0.0, -0.0, np.inf, -np.inf, 3.4028235e38, 1e-45, -1e-45], np.float32)
    got = obf.from_f32(f)
    assert list(got[:4]) == [0x0000, 0x8000, 0x7F80, 0xFF80]
    assert got[4] == 0x7F80                # rounds past the largest bf16: +Inf
    assert list(got[5:]) == [0x0000, 0x8000]   # smallest subnormal rounds to +-0


def test_bf16_add_is_correctly_rounded_sum():
    """bf16(f32(a) + f32(b)) equals the exact sum of a and b rounded once to
    bf16, including operands whose exponents differ widely (double rounding
    through fp32 never changes the result)."""
    rng = random.Random(3)
    n = 20000
    a = np.empty(n, np.uint16)
    b = np.empty(n, np.uint16)
    for i in range(n):
        ea = rng.randint(1, 254)
        eb = max(1, min(254, ea - rng.choice([0, 1, 7, 8, 9, 15, 16, 17, 24, 25, 40, 100])))
        a[i] = rng.getrandbits(1) << 15 | ea << 7 | rng.getrandbits(7)
        b[i] = rng.getrandbits(1) << 15 | eb << 7 | rng.getrandbits(7)
    got = obf.add(a, b)
    for i in range(n):
        want = X.bf16(X.of_bf16_bits(a[i]) + X.of_bf16_bits(b[i]))
        assert X.same(X.of_bf16_bits(got[i]), want), (hex(a[i]), hex(b[i]))
