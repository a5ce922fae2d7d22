"""Pins for the oracle's E4M3 / E2M1 / bf16 codecs (CPU only).

Pinned against: the torch float8_e4m3fn cast and decode (library routine),
brute-force nearest-representable enumeration in exact rational arithmetic,
and hand-derived points in tests/golden/.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from tests._golden import rows


def _e4m3_all_values():
    """(code, exact Fraction) for every non-negative finite E4M3 code, from the bit fields."""
    out = []
    for c in range(0x7F):  # 0x7F is NaN
        e, m = (c >> 3) & 0xF, c & 7
        v = Fraction(m, 2 ** 9) if e == 0 else (1 + Fraction(m, 8)) * Fraction(2) ** (e - 7)
        out.append((c, v))
    return out


E4M3_VALUES = _e4m3_all_values()
E2M1_VALUES = [(c, Fraction(v).limit_denominator(4)) for c, v in enumerate([0, 0.5, 1, 1.5, 2, 3, 4, 6])]


def _nearest_even(v: Fraction, table, vmax):
    """Brute force: nearest representable magnitude; ties to the code with mantissa LSB 0."""
    if v >= vmax:
        return max(c for c, x in table if x == vmax)
    best = None
    for c, x in table:
        d = abs(v - x)
        if best is None or d < best[0] or (d == best[0] and (c & 1) == 0):
            best = (d, c)
    return best[1]


@pytest.mark.parametrize("code", range(256))
def test_e4m3_decode_matches_torch(code):
    ref = torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).item()
    got = oracle.e4m3_decode(np.array([code], dtype=np.uint8))[0]
    if np.isnan(ref):
        assert np.isnan(got)
    else:
        assert got == ref


def test_e4m3_encode_matches_torch_cast_in_range():
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0,
        rng.uniform(-447.9, 447.9, 5000),
        rng.standard_normal(5000) * 1e-3,
        np.array([0.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -11, 2.0 ** -9, 2.0 ** -6, 447.0, -447.0]),
    ]).astype(np.float32).astype(np.float64)
    ref = torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    got = oracle.e4m3_encode(x)
    np.testing.assert_array_equal(got, ref)


def test_e4m3_encode_brute_force():
    rng = np.random.default_rng(2)
    xs = list(rng.standard_normal(400) * 30) + list(rng.uniform(0, 500, 200)) + list(rng.uniform(0, 2e-3, 200))
    # every midpoint between consecutive values is a tie case
    vals = sorted(v for _, v in E4M3_VALUES)
    xs += [float((a + b) / 2) for a, b in zip(vals[:-1], vals[1:])]
    got = oracle.e4m3_encode(np.array(xs, dtype=np.float64))
    for x, g in zip(xs, got):
        f = Fraction(abs(x))
        c = _nearest_even(f, E4M3_VALUES, Fraction(448))
        if x < 0 or (x == 0 and np.signbit(x)):
            c |= 0x80
        assert g == c, (x, hex(g), hex(c))


def test_e2m1_brute_force_and_ties():
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    rng = np.random.default_rng(3)
    xs = mids + list(rng.uniform(0, 7, 2000)) + [0.0, 6.0, 6.5, 1e9]
    got = oracle.e2m1_encode_mag(np.array(xs))
    for x, g in zip(xs, got):
        assert g == _nearest_even(Fraction(x), E2M1_VALUES, Fraction(6)), x


def test_golden_e4m3_points():
    for v, b in rows("e4m3_points.txt"):
        got = oracle.e4m3_encode(np.array([float(v)]))[0]
        assert got == int(b, 16), (v, hex(got), b)


def test_golden_e2m1_points():
    for v, c in rows("e2m1_points.txt"):
        assert oracle.e2m1_encode_mag(np.array([float(v)]))[0] == int(c), v


def test_bf16_decode_matches_torch():
    bits = np.arange(65536, dtype=np.uint16)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = oracle.bf16_bits_to_f64(bits)
    np.testing.assert_array_equal(np.isnan(got), np.isnan(ref))
    ok = ~np.isnan(ref)
    np.testing.assert_array_equal(got[ok], ref[ok])
