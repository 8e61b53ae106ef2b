"""bf16 rounding used by the oracle's bf16 model: round-to-nearest-even onto the
8-bit-mantissa bfloat16 grid, stated on the IEEE-754 bit patterns."""
from __future__ import annotations

import numpy as np


def f32_to_bf16_bits(x) -> np.ndarray:
    """float32 -> bf16 bit patterns (uint16), round to nearest, ties to even:
    add 0x7FFF plus the lowest kept bit, then drop the low 16 bits. The sum can
    wrap in 32 bits only for NaN patterns, which are handled apart (NaN stays
    NaN, quiet); infinities stay infinite."""
    u = np.ascontiguousarray(np.asarray(x, dtype=np.float32)).view(np.uint32)
    lsb = (u >> np.uint32(16)) & np.uint32(1)
    r = ((u + np.uint32(0x7FFF) + lsb) >> np.uint32(16)).astype(np.uint16)
    nan = (u & np.uint32(0x7FFFFFFF)) > np.uint32(0x7F800000)
    if nan.any():
        r[nan] = ((u[nan] >> np.uint32(16)) | np.uint32(0x40)).astype(np.uint16)
    return r


def bf16_bits_to_f64(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32).astype(np.float64)


def round_f32_to_bf16(x) -> np.ndarray:
    """float32 values -> float64 values on the bf16 grid (RNE)."""
    return bf16_bits_to_f64(f32_to_bf16_bits(x))


def _f64_to_f32_round_to_odd(x: np.ndarray) -> np.ndarray:
    """Round float64 to float32 with round-to-odd: truncate toward zero, then
    set the last bit when the truncation was inexact. Rounding that result to
    a format with at most 22 fewer bits is the correctly rounded result."""
    x = np.asarray(x, dtype=np.float64)
    f = x.astype(np.float32)
    over = np.abs(f.astype(np.float64)) > np.abs(x)
    f = np.where(over, np.nextafter(f, np.float32(0)), f).astype(np.float32)
    inexact = f.astype(np.float64) != x
    bits = f.view(np.uint32) | np.where(inexact, np.uint32(1), np.uint32(0))
    return bits.astype(np.uint32).view(np.float32)


def round_to_bf16(x) -> np.ndarray:
    """float64 values -> float64 values on the bf16 grid, correctly rounded
    (nearest, ties to even) from the exact float64 value."""
    return round_f32_to_bf16(_f64_to_f32_round_to_odd(x))
