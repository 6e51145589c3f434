"""bf16 <-> fp32 conversions on bit patterns (oracle; test infrastructure).

bf16 is the upper half of an IEEE binary32: 1 sign, 8 exponent, 7 fraction
bits.  Widening is exact (append 16 zero bits).  Narrowing rounds to nearest,
ties to even, over the 16 dropped bits; NaN maps to the quiet NaN 0x7FC0 and
overflow rounds to +-Inf, as IEEE round-to-nearest prescribes.  No flush of
subnormals.

The bf16 gradients of the pages' systems ("param.grad (BF16)" in DeepSpeed
ZeRO-3 source walkthrough, section 1; "bf16 communication" in DeepSpeed issue
8364) are stored here as numpy uint16 arrays of their bit patterns.
"""
import numpy as np


def to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32)


def from_f32(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    rounded = ((u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)).astype(np.uint16)
    is_nan = (u & np.uint64(0x7FFFFFFF)) > np.uint64(0x7F800000)
    return np.where(is_nan, np.uint16(0x7FC0), rounded).astype(np.uint16)


def add(a_bits: np.ndarray, b_bits: np.ndarray) -> np.ndarray:
    """bf16 + bf16 -> bf16: the fp32 sum of the widened operands, then rounded
    to bf16 (the fp32 sum of two bf16 values is exact unless their exponents
    differ by more than 15, and then the smaller one is too small to move the
    bf16 rounding, so this is the correctly rounded bf16 sum)."""
    with np.errstate(over="ignore", invalid="ignore"):     # inf + -inf is NaN, as in IEEE
        return from_f32(to_f32(a_bits) + to_f32(b_bits))
