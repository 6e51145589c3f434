"""Pins of the oracle's bf16 conversions against PyTorch's CPU bf16 conversion
(a library routine) and against exact rational rounding."""
import os
import random

import numpy as np
import pytest
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


def _build_exhaustive(tmp_path, *defines):
    """Compiles tests/bf16_add_exhaustive.c with the host C compiler (OpenMP
    when available); skips where there is none."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = os.path.join(os.path.dirname(__file__), "bf16_add_exhaustive.c")
    exe = str(tmp_path / ("bf16x" + "".join(d.lower() for d in defines)))
    base = [cc, "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", *defines,
            src, "-o", exe]
    if subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True).returncode:
        subprocess.run(base, check=True, capture_output=True)
    return exe


def _run(exe, *args):
    import subprocess
    out = subprocess.run([exe, *map(str, args)], capture_output=True, text=True, timeout=600,
                         check=True).stdout
    kv = dict(f.split("=") for f in out.split())
    return int(kv["pairs"]), int(kv["mismatches"])


def test_bf16_add_rule_exhaustive_over_all_pairs(tmp_path):
    """Every one of the 2**32 (a, b) bf16 pairs: rounding the binary32 sum to
    bf16 gives the exactly rounded bf16 sum (the per-hop rounding rule),
    including zeros, subnormals, infinities and NaN.  The same checker built
    with truncation in place of rounding must find mismatches."""
    pairs, bad = _run(_build_exhaustive(tmp_path))
    assert pairs == 1 << 32 and bad == 0
    pairs, bad = _run(_build_exhaustive(tmp_path, "-DROUTE1_TRUNCATES"), 0x3F80, 0x3FC0)
    assert pairs == 64 << 16 and bad > 0


def test_oracle_add_equals_exact_rounding_for_every_b(tmp_path):
    """The oracle's bf16 add against the checker's exact integer route, for
    every b and first operands spread over signs, binades, subnormals and the
    largest finite values."""
    import subprocess
    exe = _build_exhaustive(tmp_path)
    a_list = [0x0000, 0x0001, 0x007F, 0x0080, 0x0081, 0x0100, 0x1234, 0x3F80, 0x3F81,
              0x3FFF, 0x4000, 0x42C8, 0x5F00, 0x7F00, 0x7F7E, 0x7F7F, 0x7F80,
              0x8000, 0x8001, 0x80FF, 0xBF80, 0xC000, 0xC2C8, 0xFF7F, 0xFF80]
    raw = subprocess.run([exe, "--dump", *map(str, a_list)], capture_output=True, timeout=300,
                         check=True).stdout
    want = np.frombuffer(raw, dtype="<u2").reshape(len(a_list), 65536)
    b = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    for i, a in enumerate(a_list):
        with np.errstate(invalid="ignore"):         # inf + -inf
            got = obf.add(np.full(65536, a, np.uint16), b)
        assert np.array_equal(got, want[i]), hex(a)
