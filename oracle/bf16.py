"""bf16 / fp32 storage rounding for the oracle (test infrastructure only).

bf16 is the 16-bit format with 8 exponent bits and 8 significant bits.  The
oracle rounds a double to it directly (no intermediate float32), to nearest,
ties to even.  fp32 rounding is numpy's float64 -> float32 cast (IEEE round to
nearest even).
"""
import numpy as np


def bf16_round(x):
    """Round float64 values to the nearest bf16 value (ties to even), as float64.

    Written from the definition: keep 8 significant bits of the binary
    significand, rounding half to even (np.rint).  Valid for the normal range
    of bf16 (all values this path produces).
    """
    x = np.asarray(x, dtype=np.float64)
    m, e = np.frexp(x)                      # x = m * 2**e, |m| in [0.5, 1)
    return np.ldexp(np.rint(np.ldexp(m, 8)), e - 8)


def bf16_from_bits(bits):
    """uint16 bf16 bit patterns -> float64 values (exact)."""
    b = np.asarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def bf16_to_bits(x):
    """float64 values that are exactly bf16-representable -> uint16 bit patterns."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    if not np.array_equal(f.astype(np.float64), x) or np.any(f.view(np.uint32) & np.uint32(0xFFFF)):
        raise ValueError("bf16_to_bits: value is not bf16-representable")
    return (f.view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def fp32_round(x):
    """Round float64 values to float32 (nearest even), returned as float64."""
    return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)
