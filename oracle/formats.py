"""E2M1, E4M3 and bfloat16 as exact float64 arithmetic (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

The main KV cache stores E2M1 values with one E4M3 scale per 16 channels
([FP4] in the package docstring). The bit layouts below are the OCP
microscaling / NVFP4 element formats the page names:

E2M1: sign(1) exponent(2, bias 1) mantissa(1). Magnitudes, by code 0..7:
      0, 0.5, 1, 1.5, 2, 3, 4, 6. No Inf, no NaN.
E4M3 ("fn"): sign(1) exponent(4, bias 7) mantissa(3). Normal values
      (1 + m/8) * 2^(e-7) for e in 1..15; subnormals m * 2^-9; S.1111.111
      is NaN; no Inf; largest finite 448.

Rounding is round-to-nearest, ties to the even mantissa, saturating to the
largest finite magnitude ("satfinite"). Inputs must be finite.
"""
from __future__ import annotations

import numpy as np

E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)
E4M3_MAX = 448.0


def bf16_bits_to_f64(bits) -> np.ndarray:
    """bfloat16 bit patterns (uint16) -> exact float64 values."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    with np.errstate(invalid="ignore"):
        return b.view(np.float32).astype(np.float64)


def e4m3_decode(b) -> np.ndarray:
    """E4M3 bytes -> float64 (NaN for the two NaN codes)."""
    b = np.asarray(b, dtype=np.uint8).astype(np.int64)
    s = (b >> 7) & 1
    e = (b >> 3) & 0xF
    m = b & 7
    mag = np.where(e == 0, m * 2.0 ** -9, (1.0 + m / 8.0) * np.exp2((e - 7).astype(np.float64)))
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return np.where(s == 1, -mag, mag)


def _binade(v: np.ndarray) -> np.ndarray:
    """floor(log2(v)) for v > 0, computed exactly with frexp (v = f*2^x, f in [0.5,1))."""
    _, x = np.frexp(v)
    return x.astype(np.int64) - 1


def e4m3_encode(x) -> np.ndarray:
    """float64 -> E4M3 byte, round to nearest even, saturating at +-448."""
    x = np.asarray(x, dtype=np.float64)
    sign = np.signbit(x).astype(np.int64)
    v = np.abs(x)
    e = np.maximum(_binade(np.where(v > 0, v, 1.0)), -6)       # subnormals share binade -6
    q = np.exp2((e - 3).astype(np.float64))                    # 3 mantissa bits in the binade
    r = np.rint(v / q) * q                                     # np.rint rounds half to even
    r = np.where(v >= E4M3_MAX, E4M3_MAX, np.minimum(r, E4M3_MAX))
    # encode the representable magnitude r
    er = _binade(np.where(r > 0, r, 1.0))
    normal = r >= 2.0 ** -6
    mant_n = np.rint((r / np.exp2(er.astype(np.float64)) - 1.0) * 8.0).astype(np.int64)
    bits_n = ((er + 7) << 3) | mant_n
    bits_s = np.rint(r / 2.0 ** -9).astype(np.int64)
    bits = np.where(normal, bits_n, bits_s)
    return ((sign << 7) | bits).astype(np.uint8)


def e2m1_encode_mag(v) -> np.ndarray:
    """Non-negative float64 magnitude -> E2M1 magnitude code 0..7 (RNE, saturating at 6)."""
    v = np.asarray(v, dtype=np.float64)
    e = np.maximum(_binade(np.where(v > 0, v, 1.0)), 0)         # the subnormal 0.5 shares binade 0
    q = np.exp2((e - 1).astype(np.float64))                    # 1 mantissa bit in the binade
    r = np.minimum(np.rint(v / q) * q, 6.0)
    return np.searchsorted(E2M1_GRID, r).astype(np.uint8)
