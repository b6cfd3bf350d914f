"""Pins of the oracle's E5M6 cache (page P1, paragraph 3: the activations that
are re-tiled from 1x128 to 128x1 tiles are kept in a custom E5M6 format).

The E5M6 value set is pinned against numpy's IEEE half precision (the same
exponent field; E5M6 keeps the top 6 of half's 10 mantissa bits), rounding
against a float64 closed form, the bit packing against hand-worked bytes,
and the quantizers against definitions already pinned elsewhere."""
import os
from fractions import Fraction

import numpy as np
import pytest

import synth


def _half_from_e5m6_bits(c):
    """The half-precision value whose bits are the E5M6 code with 4 zero
    mantissa bits appended."""
    h = ((c & 0x800) << 4) | ((c & 0x7FF) << 4)
    return np.array([h], np.uint16).view(np.float16)[0]


def test_decode_matches_half_precision_subset(oracle_mod):
    for c in range(4096):
        v = oracle_mod.e5m6_decode(c)
        h = float(_half_from_e5m6_bits(c))
        if np.isnan(h):
            assert np.isnan(v), c
        else:
            assert v == h, (hex(c), v, h)
    assert oracle_mod.e5m6_decode(0x7BF) == 65024.0
    assert oracle_mod.e5m6_decode(0x001) == 2.0 ** -20
    assert oracle_mod.e5m6_decode(0x040) == 2.0 ** -14
    assert oracle_mod.e5m6_decode(0x3C0) == 1.0
    assert np.isinf(oracle_mod.e5m6_decode(0x7C0)) and np.isnan(oracle_mod.e5m6_decode(0x7FF))


def test_encode_round_trip_and_specials(oracle_mod):
    for c in list(range(0x000, 0x7C0)) + list(range(0x800, 0xFC0)):
        assert oracle_mod.e5m6_encode(oracle_mod.e5m6_decode(c)) == c, hex(c)
    assert oracle_mod.e5m6_encode(float("nan")) == 0x7FF
    assert oracle_mod.e5m6_encode(float("inf")) == 0x7BF
    assert oracle_mod.e5m6_encode(float("-inf")) == 0xFBF
    assert oracle_mod.e5m6_encode(70000.0) == 0x7BF
    assert oracle_mod.e5m6_encode(-0.0) == 0x800


def _closed_form(y):
    """Nearest value with 7 significant bits and E5M6's exponent range, ties
    to even (numpy's rint), saturating at 65024."""
    a = abs(float(y))
    if a == 0.0:
        return 0.0
    e = max(int(np.floor(np.log2(a))), -14)
    q = 2.0 ** (e - 6)
    v = float(np.rint(a / q)) * q
    return float(np.copysign(min(v, 65024.0), y))


def test_encode_matches_closed_form(oracle_mod):
    rng = np.random.default_rng(7)
    ys = (rng.standard_normal(4000) * 2.0 ** rng.uniform(-24, 17, 4000)).astype(np.float32)
    for y in ys:
        got = oracle_mod.e5m6_decode(oracle_mod.e5m6_encode(float(y)))
        assert got == _closed_form(y), (float(y), got, _closed_form(y))


def test_midpoints_round_to_even(oracle_mod):
    for c in (0x000, 0x001, 0x03F, 0x040, 0x2A5, 0x3C0, 0x7BE):
        lo, hi = oracle_mod.e5m6_decode(c), oracle_mod.e5m6_decode(c + 1)
        mid = np.float32((lo + hi) / 2)
        assert float(mid) == (lo + hi) / 2  # exactly representable
        want = c if c % 2 == 0 else c + 1
        assert oracle_mod.e5m6_encode(float(mid)) == want, hex(c)
        assert oracle_mod.e5m6_encode(float(np.nextafter(mid, np.float32(np.inf)))) == c + 1
        assert oracle_mod.e5m6_encode(float(np.nextafter(mid, np.float32(-np.inf)))) == c


def test_pack_layout(oracle_mod):
    # element i occupies bits 12i .. 12i+11 of a little-endian byte stream
    assert oracle_mod.e5m6_pack(np.array([0xABC, 0x123])).tolist() == [0xBC, 0x3A, 0x12]
    assert oracle_mod.e5m6_pack(np.array([0x001, 0x800, 0xFFF, 0x000])).tolist() == \
        [0x01, 0x00, 0x80, 0xFF, 0x0F, 0x00]
    rng = np.random.default_rng(8)
    c = rng.integers(0, 4096, (5, 256)).astype(np.uint16)
    assert np.array_equal(oracle_mod.e5m6_unpack(oracle_mod.e5m6_pack(c)), c)


def _codes(oracle_mod, packed):
    return oracle_mod.e5m6_unpack(packed)


def test_quant_e5m6_unit_scale_is_plain_encoding(oracle_mod):
    """A tile whose max-abs is 65024 has scale 1: codes are the plain
    encoding of the values."""
    rng = np.random.default_rng(9)
    x = (rng.standard_normal((4, 256)) * 3000.0).astype(np.float32)
    x[:, 5] = 65024.0
    x[:, 130] = -65024.0
    bits = synth.f32_to_bf16_bits(x)
    packed, s = oracle_mod.quant_act_e5m6_1x128(bits)
    assert np.all(s == 1.0)
    vals = synth.bf16_bits_to_f32(bits)
    codes = _codes(oracle_mod, packed)
    want = np.array([[oracle_mod.e5m6_encode(float(v)) for v in row] for row in vals])
    assert np.array_equal(codes, want)


def test_quant_e5m6_invariants_and_specials(oracle_mod):
    rng = np.random.default_rng(10)
    bits, _ = synth.normal_with_outlier_columns(rng, (16, 384), 3, 100.0)
    packed, s = oracle_mod.quant_act_e5m6_1x128(bits)
    x = synth.bf16_bits_to_f32(bits).astype(np.float64)
    dec = oracle_mod.e5m6_decode_array(_codes(oracle_mod, packed))
    for kb in range(3):
        sc = s[kb].astype(np.float64)[:, None]
        xs, d = x[:, kb * 128:(kb + 1) * 128], dec[:, kb * 128:(kb + 1) * 128]
        assert np.all(np.abs(d).max(axis=1) == 65024.0)
        y = np.abs(xs / sc)
        e = np.floor(np.log2(np.maximum(y, 2.0 ** -14)))
        half = 0.5 * 2.0 ** (e - 6)
        assert np.all(np.abs(xs - d * sc) <= (half + 2.0 ** -24 * y) * sc)
    # zeros, NaN and Inf
    z = np.zeros((2, 128), np.float32)
    z[1, 3] = -0.0
    z[0, 9] = np.nan
    packed, s = oracle_mod.quant_act_e5m6_1x128(synth.f32_to_bf16_bits(z))
    c = _codes(oracle_mod, packed)
    assert np.all(s == 0.0) and c[0, 9] == 0x7FF and c[1, 3] == 0x800
    assert np.all(np.delete(c.ravel(), [9, 128 + 3]) == 0)
    w = np.ones((1, 128), np.float32)
    w[0, 0] = np.inf
    packed, s = oracle_mod.quant_act_e5m6_1x128(synth.f32_to_bf16_bits(w))
    c = _codes(oracle_mod, packed)
    assert np.isinf(s[0, 0]) and c[0, 0] == 0x7FF and np.all(c[0, 1:] == 0)


def test_requant_e5m6_reduces_to_128x1_quantizer(oracle_mod):
    """With power-of-two scales every decoded value is exactly a bf16 value,
    so the re-tiling equals the 128x1 quantizer applied to those values."""
    rng = np.random.default_rng(11)
    M, K = 256, 384
    codes = rng.integers(0, 0x7C0, (M, K)).astype(np.uint16) | \
        (rng.integers(0, 2, (M, K)).astype(np.uint16) << 11)
    s = (2.0 ** rng.integers(-30, -10, (K // 128, M))).astype(np.float32)
    packed = oracle_mod.e5m6_pack(codes)
    qT, sT = oracle_mod.requant_e5m6_to_128x1(packed, s)
    xh = oracle_mod.e5m6_decode_array(codes) * np.repeat(s.T.astype(np.float64), 128, axis=1)
    xh_bits = synth.f32_to_bf16_bits(xh.astype(np.float32))
    assert np.array_equal(synth.bf16_bits_to_f32(xh_bits).astype(np.float64), xh)
    q_ref, s_ref = oracle_mod.quant_act_128x1(xh_bits)
    assert np.array_equal(qT, q_ref) and np.array_equal(sT.view(np.uint32), s_ref.view(np.uint32))


def test_requant_e5m6_general_scales_half_ulp(oracle_mod):
    rng = np.random.default_rng(12)
    bits, _ = synth.normal_with_outlier_columns(rng, (128, 256), 2, 100.0)
    packed, s = oracle_mod.quant_act_e5m6_1x128(bits)
    qT, sT = oracle_mod.requant_e5m6_to_128x1(packed, s)
    xh = oracle_mod.e5m6_decode_array(_codes(oracle_mod, packed)).astype(np.float32) * \
        np.repeat(s.T, 128, axis=1)
    d = oracle_mod.e4m3_decode_array(qT).T * sT[0][None, :].astype(np.float64)
    y = np.abs(xh.astype(np.float64) / sT[0][None, :])
    e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
    half = 0.5 * np.where(y < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))
    assert np.all(np.abs(xh - d) <= (half + 2.0 ** -24 * y) * sT[0][None, :])
    assert np.all(np.abs(oracle_mod.e4m3_decode_array(qT)).max(axis=1) == 448.0)


def test_hand_worked_golden_values(oracle_mod):
    """Codes worked out by hand from the format definition
    (tests/golden/e5m6_hand_values.txt)."""
    path = os.path.join(os.path.dirname(__file__), "golden", "e5m6_hand_values.txt")
    n = 0
    for line in open(path):
        line = line.split("#")[0].strip()
        if not line:
            continue
        value, code = line.split()
        v = np.float32(float(Fraction(value)) if value != "-0.0" else -0.0)
        assert float(v) == float(Fraction(value)), value  # the value is exact in FP32
        assert oracle_mod.e5m6_encode(float(v)) == int(code, 16), (value, code)
        n += 1
    assert n == 14
