"""Pins for the oracle's FP4 quantiser (E2M1 codes + one E4M3 scale per 16 channels).

Pinned against: hand-derived examples in tests/golden/, an exact
threshold classifier (|x| compared against scale * E2M1 midpoints, all
products exact in float64), exhaustive bf16 coverage, and invariants
(grid round trip, sign symmetry, power-of-two scaling).
"""
import numpy as np
import pytest

import oracle
from tests._golden import rows

E2M1_MIDS = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])


def f64_to_bf16_bits(x):
    """float64 values that are exactly representable in bf16 -> bit patterns."""
    f = np.asarray(x, dtype=np.float32)
    assert np.all(f.astype(np.float64) == np.asarray(x, dtype=np.float64))
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "input is not bf16-exact"
    return (b >> 16).astype(np.uint16)


def unpack(codes):
    return np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(codes.shape[:-1] + (-1,))


def test_golden_groups():
    for name, xs, scale, codes in rows("fp4_quant_examples.txt"):
        x = np.array([float(v) for v in xs.split()])
        assert x.size == 16
        c, s = oracle.quantize_fp4(f64_to_bf16_bits(x))
        assert s[0] == int(scale, 16), (name, hex(s[0]))
        assert list(c) == [int(b, 16) for b in codes.split()], (name, [hex(v) for v in c])


def _threshold_classify(x, s):
    """E2M1 code of x at scale s by exact comparisons with s*midpoints (ties -> even code)."""
    a = np.abs(x)[..., None]
    t = np.broadcast_to(s[:, None], x.shape)[..., None] * E2M1_MIDS   # exact: <=4 sig. bits x <=3
    above = (a > t).sum(-1)
    tie = (a == t)
    # at a tie between code c and c+1 (mid index c) the even code wins
    tie_idx = np.argmax(tie, axis=-1)
    even_up = (tie_idx + 1) % 2 == 0
    code = np.where(tie.any(-1), np.where(even_up, tie_idx + 1, tie_idx), above)
    return code


def _scale_classify(amax):
    """E4M3 scale byte of amax/6 by exact comparison of amax with 6 * (E4M3 midpoints)."""
    vals = oracle.e4m3_decode(np.arange(0x7F, dtype=np.uint8))   # 0 .. 448 ascending
    mids = (vals[:-1] + vals[1:]) / 2.0
    a = amax[..., None]
    t = 6.0 * mids                                   # exact in float64
    above = (a > t).sum(-1)
    tie = (a == t)
    tie_idx = np.argmax(tie, axis=-1)
    even_up = (tie_idx + 1) % 2 == 0
    return np.where(tie.any(-1), np.where(even_up, tie_idx + 1, tie_idx), above).astype(np.uint8)


def _random_bf16_groups(rng, g, lo_exp=-20, hi_exp=12):
    sign = rng.integers(0, 2, (g, 16)) << 15
    exp = rng.integers(127 + lo_exp, 127 + hi_exp, (g, 16)) << 7
    man = rng.integers(0, 128, (g, 16))
    bits = (sign | exp | man).astype(np.uint16)
    # sprinkle zeros and -0
    z = rng.random((g, 16)) < 0.05
    bits[z] = np.where(rng.random(z.sum()) < 0.5, 0x0000, 0x8000)
    return bits


def test_threshold_classifier_agrees_random():
    rng = np.random.default_rng(7)
    bits = _random_bf16_groups(rng, 20000)
    codes, scales = oracle.quantize_fp4(bits)
    x = oracle.bf16_bits_to_f64(bits)
    amax = np.abs(x).max(-1)
    np.testing.assert_array_equal(scales[:, 0], _scale_classify(amax))
    s = oracle.e4m3_decode(scales[:, 0])
    mag = _threshold_classify(x, s)
    sign = np.signbit(x).astype(np.int64)
    exp_code = np.where((s > 0)[:, None], mag | (sign << 3), 0)
    np.testing.assert_array_equal(unpack(codes), exp_code)


@pytest.mark.parametrize("amax_bits", [0x3F80, 0x4040, 0x3E2A, 0x4380, 0x3B80, 0x4500, 0x3C00, 0x3A00])
def test_exhaustive_bf16_member(amax_bits):
    """Every finite bf16 value with |x| <= amax as one member of a group whose amax is fixed."""
    all_bits = np.arange(65536, dtype=np.uint16)
    x_all = oracle.bf16_bits_to_f64(all_bits)
    amax = oracle.bf16_bits_to_f64(np.array([amax_bits], dtype=np.uint16))[0]
    ok = np.isfinite(x_all) & (np.abs(x_all) <= amax)
    members = all_bits[ok]
    g = np.zeros((members.size, 16), dtype=np.uint16)
    g[:, 0] = amax_bits
    g[:, 1] = members
    codes, scales = oracle.quantize_fp4(g)
    x = oracle.bf16_bits_to_f64(g)
    np.testing.assert_array_equal(scales[:, 0], _scale_classify(np.abs(x).max(-1)))
    s = oracle.e4m3_decode(scales[:, 0])
    mag = _threshold_classify(x, s)
    sign = np.signbit(x).astype(np.int64)
    exp_code = np.where((s > 0)[:, None], mag | (sign << 3), 0)
    np.testing.assert_array_equal(unpack(codes), exp_code)


def test_grid_round_trip():
    """A group holding +-grid*s with amax = 6s reproduces s and the codes exactly."""
    grid = oracle.E2M1_GRID
    for sc in [0x38, 0x23, 0x01, 0x7E, 0x30, 0x49, 0x08]:
        s = oracle.e4m3_decode(np.array([sc], dtype=np.uint8))[0]
        vals = np.concatenate([grid, -grid])          # 16 values, includes +-6
        x = vals * s
        try:
            bits = f64_to_bf16_bits(x)
        except AssertionError:
            continue
        codes, scales = oracle.quantize_fp4(bits)
        assert scales[0] == sc
        deq = oracle.dequant_fp4(codes, scales)
        np.testing.assert_array_equal(deq, x)


def test_sign_symmetry_and_pow2_scaling():
    rng = np.random.default_rng(11)
    bits = _random_bf16_groups(rng, 3072, lo_exp=-3, hi_exp=3).reshape(-1, 512)
    c1, s1 = oracle.quantize_fp4(bits)
    c2, s2 = oracle.quantize_fp4(bits ^ np.uint16(0x8000))
    np.testing.assert_array_equal(s1, s2)
    u1, u2 = unpack(c1), unpack(c2)
    live = np.repeat(oracle.e4m3_decode(s1) > 0, 16, axis=-1)
    np.testing.assert_array_equal(np.where(live, u1 ^ 8, 0), u2)
    # x * 2^3: exponent field + 3 (no overflow in this range) -> scale * 8, same codes
    x = oracle.bf16_bits_to_f64(bits)
    nz = x != 0
    bits8 = np.where(nz, bits + np.uint16(3 << 7), bits).astype(np.uint16)
    c3, s3 = oracle.quantize_fp4(bits8)
    np.testing.assert_array_equal(c3, c1)
    d1, d3 = oracle.e4m3_decode(s1), oracle.e4m3_decode(s3)
    norm = d1 >= 2.0 ** -6 * 8  # both scales normal -> exact factor 8
    np.testing.assert_array_equal(d3[norm], d1[norm] * 8)


def test_dequant_reconstruction_error_bound():
    """|x - dequant| <= scale * (half the local E2M1 spacing) unless saturated."""
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 512)).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)
    codes, scales = oracle.quantize_fp4(bits)
    xd = oracle.bf16_bits_to_f64(bits)
    xh = oracle.dequant_fp4(codes, scales)
    s = np.repeat(oracle.e4m3_decode(scales), 16, axis=-1)
    err = np.abs(xd - xh)
    assert np.all(err <= s * 1.0 + np.abs(xd) * 0.13)
    assert np.all(np.abs(xh) <= 6 * s + 0)
