"""Philox4x64-10 counter-based generator and the Box-Muller weight stream.

Philox4x64-10 is restated from its published definition (J. Salmon, M. Moraes,
R. Dror, D. Shaw, "Parallel random numbers: as easy as 1, 2, 3", SC'11): ten
rounds of two 64x64->128 multiplies with the Weyl key schedule. The
normal variates use the Box-Muller transform (Box & Muller, 1958).

Weight stream of the random-init model (a reading: the pages give no weights;
the configurations ask for N(0, 0.02^2) entries):
  element i of tensor t  ->  block n = i // 4, lane j = i % 4,
  words (w0, w1, w2, w3) = Philox4x64-10(counter = (n, t, 0, 0), key = (seed, 0)),
  lanes 0/1 come from (w0, w1), lanes 2/3 from (w2, w3):
     u1 = ((w_a >> 11) + 1) * 2^-53   in (0, 1]
     u2 =  (w_b >> 11)      * 2^-53   in [0, 1)
     r = sqrt(-2 ln u1),  theta = u2 * 6.283185307179586
     lane 0/2 -> r cos(theta),  lane 1/3 -> r sin(theta)
  value = float32(sigma * z) (double product, one rounding), then bf16 (RNE)
  for bf16 models.
"""
from __future__ import annotations

import numpy as np

_M0 = np.uint64(0xD2E7470EE14C6C93)
_M1 = np.uint64(0xCA5A826395121157)
_W0 = np.uint64(0x9E3779B97F4A7C15)
_W1 = np.uint64(0xBB67AE8584CAA73B)
_LO32 = np.uint64(0xFFFFFFFF)
_S32 = np.uint64(32)


def _mulhilo(a: np.uint64, b: np.ndarray):
    """(hi, lo) of the 128-bit product a*b, elementwise, from 32-bit halves."""
    a0, a1 = a & _LO32, a >> _S32
    b0, b1 = b & _LO32, b >> _S32
    p00 = a0 * b0
    p01 = a0 * b1
    p10 = a1 * b0
    p11 = a1 * b1
    mid = (p00 >> _S32) + (p01 & _LO32) + (p10 & _LO32)
    hi = p11 + (p01 >> _S32) + (p10 >> _S32) + (mid >> _S32)
    lo = a * b  # wraps mod 2^64
    return hi, lo


def philox4x64_10(c0, c1, c2, c3, k0, k1):
    """Vectorised Philox4x64-10. Counter words and key words are uint64 arrays
    or scalars (broadcast). Returns four uint64 arrays."""
    with np.errstate(over="ignore"):
        x0, x1, x2, x3 = (np.asarray(c, dtype=np.uint64) for c in (c0, c1, c2, c3))
        k0 = np.asarray(k0, dtype=np.uint64)
        k1 = np.asarray(k1, dtype=np.uint64)
        for rnd in range(10):
            if rnd:
                k0 = k0 + _W0
                k1 = k1 + _W1
            hi0, lo0 = _mulhilo(_M0, x0)
            hi1, lo1 = _mulhilo(_M1, x2)
            x0, x1, x2, x3 = hi1 ^ x1 ^ k0, lo1, hi0 ^ x3 ^ k1, lo0
        return x0, x1, x2, x3


def box_muller(wa: np.ndarray, wb: np.ndarray):
    """Two standard normals (cos branch, sin branch) from two uint64 words."""
    u1 = ((wa >> np.uint64(11)).astype(np.float64) + 1.0) * 2.0 ** -53
    u2 = (wb >> np.uint64(11)).astype(np.float64) * 2.0 ** -53
    r = np.sqrt(-2.0 * np.log(u1))
    theta = u2 * 6.283185307179586
    return r * np.cos(theta), r * np.sin(theta)


def normal_stream(seed: int, tensor_id: int, start: int, count: int) -> np.ndarray:
    """Standard normals z for flat elements [start, start+count) of a tensor (float64)."""
    if count <= 0:
        return np.zeros(0, dtype=np.float64)
    n0 = start // 4
    n1 = (start + count + 3) // 4
    n = np.arange(n0, n1, dtype=np.uint64)
    w0, w1, w2, w3 = philox4x64_10(n, np.uint64(tensor_id), np.uint64(0), np.uint64(0),
                                   np.uint64(seed), np.uint64(0))
    za, zb = box_muller(w0, w1)
    zc, zd = box_muller(w2, w3)
    z = np.stack([za, zb, zc, zd], axis=1).reshape(-1)
    off = start - n0 * 4
    return z[off: off + count]


def weight_values(seed: int, tensor_id: int, start: int, count: int, sigma: float = 0.02):
    """float32 weight values sigma*z (one rounding from the double product)."""
    return (sigma * normal_stream(seed, tensor_id, start, count)).astype(np.float32)
