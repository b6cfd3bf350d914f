"""Pins of the oracle's quantizers (1x128 activation tiles, 128x128 weight
blocks, the 128x1 backward-pass tiles) to hand-worked values, invariants and
layout identities.  Page 1, paragraph 3 defines the granularity and the
online max-abs scaling; the E4M3 format and scale = amax/448 are readings.
"""
import math
import os

import numpy as np
import pytest

import synth
from synth import f32_to_bf16_bits, bf16_bits_to_f32, normal, normal_with_outlier_columns

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e4m3_hand_tiles.txt")


def _golden_rows():
    rows = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if not line:
            continue
        amax, x, code = line.split()
        rows.append((float(amax), float(x), int(code, 16)))
    return rows


@pytest.mark.parametrize("amax,x,code", _golden_rows())
def test_hand_worked_tiles(oracle_mod, amax, x, code):
    tile = np.zeros((1, 128), np.float32)
    tile[0, 0] = amax
    tile[0, 1] = x
    bits = f32_to_bf16_bits(tile)
    assert bf16_bits_to_f32(bits)[0, 1] == np.float32(x) or x == 0.0  # bf16-exact fixture
    q, s = oracle_mod.quant_act_1x128(bits)
    assert s[0, 0] == np.float32(amax) / np.float32(448.0)
    assert q[0, 1] == code, (amax, x, hex(q[0, 1]))
    assert (q[0, 0] & 0x7F) == 0x7E


def _ulp_e4m3(y):
    a = np.abs(y)
    e = np.floor(np.log2(np.where(a > 0, a, 1.0)))
    return np.where(a < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))


def _check_invariants(oracle_mod, x_vals, q, s_per_elem):
    """|x - dec(q) s| <= (ulp(y)/2 + 2^-24 |y|) s with y = x/s (bound of the
    two roundings), and every group reaches +-448 unless it is all zero."""
    dec = oracle_mod.e4m3_decode_array(q)
    s = s_per_elem.astype(np.float64)
    x = x_vals.astype(np.float64)
    nz = s > 0
    y = np.where(nz, x / np.where(nz, s, 1.0), 0.0)
    bound = (0.5 * _ulp_e4m3(y) + 2.0 ** -24 * np.abs(y)) * s
    err = np.abs(x - dec * s)
    assert np.all(err[nz] <= bound[nz] * (1 + 1e-12))
    assert np.all(dec[~nz] == 0)


def test_act_1x128_invariants_tiny(oracle_mod):
    rng = np.random.default_rng(0)
    x, _ = normal_with_outlier_columns(rng, (96, 512), 4, 50.0)
    q, s = oracle_mod.quant_act_1x128(x)
    xf = bf16_bits_to_f32(x)
    M, K = x.shape
    s_elem = np.repeat(s.T, 128, axis=1)  # [M, K]
    _check_invariants(oracle_mod, xf, q, s_elem)
    # scale = amax/448 with amax computed independently by numpy
    amax = np.abs(xf.reshape(M, K // 128, 128)).max(axis=2)  # [M, KB]
    assert np.array_equal(s, (amax / np.float32(448.0)).astype(np.float32).T)
    # each group holds an element coded +-448
    grp = (q.reshape(M, K // 128, 128) & 0x7F) == 0x7E
    assert grp.any(axis=2).all()


def test_act_1x128_scale_layout(oracle_mod):
    """Group (m, kb) gets amax 2^(m + 3 kb): the scale array must be [KB][M]."""
    M, K = 5, 384
    x = np.zeros((M, K), np.float32)
    for m in range(M):
        for kb in range(3):
            x[m, kb * 128 + (m * 7 + kb) % 128] = -(2.0 ** (m + 3 * kb))
    q, s = oracle_mod.quant_act_1x128(f32_to_bf16_bits(x))
    for m in range(M):
        for kb in range(3):
            assert s[kb, m] == np.float32(2.0 ** (m + 3 * kb)) / np.float32(448)
            assert q[m, kb * 128 + (m * 7 + kb) % 128] == 0xFE


def test_all_zero_and_signed_zero_tile(oracle_mod):
    x = np.zeros((2, 128), np.float32)
    x[0, 3] = -0.0
    x[1, :] = -0.0
    q, s = oracle_mod.quant_act_1x128(f32_to_bf16_bits(x))
    assert np.all(s == 0)
    assert q[0, 3] == 0x80 and q[0, 4] == 0x00
    assert np.all(q[1] == 0x80)


def test_nonfinite_reading(oracle_mod):
    """Reading R5: NaN ignored by amax and coded 0x7F; Inf makes s = Inf."""
    x = np.zeros((2, 128), np.float32)
    x[0, :] = 1.0
    x[0, 5] = np.nan
    x[0, 6] = 448.0
    x[1, :] = -3.0
    x[1, 9] = np.inf
    q, s = oracle_mod.quant_act_1x128(f32_to_bf16_bits(x))
    assert s[0, 0] == 1.0
    assert q[0, 5] == 0x7F and q[0, 6] == 0x7E and q[0, 0] == 0x38
    assert math.isinf(s[0, 1])
    assert q[1, 9] == 0x7F and q[1, 0] == 0x80


def test_subnormal_range_tile(oracle_mod):
    """Tiny amax keeps a nonzero (subnormal FP32) scale; codes stay in range."""
    x = np.zeros((1, 128), np.float32)
    x[0, 0] = np.float32(2.0 ** -133)  # smallest bf16 subnormal
    x[0, 1] = -np.float32(2.0 ** -130)
    q, s = oracle_mod.quant_act_1x128(f32_to_bf16_bits(x))
    assert s[0, 0] > 0 and s[0, 0] < np.float32(2.0 ** -126)
    assert q[0, 1] == 0xFE
    _check_invariants(oracle_mod, bf16_bits_to_f32(f32_to_bf16_bits(x)), q,
                      np.full((1, 128), s[0, 0]))


def test_act_128x1_is_transpose_of_1x128(oracle_mod):
    rng = np.random.default_rng(1)
    x, _ = normal_with_outlier_columns(rng, (256, 200), 3, 100.0)
    qT, sT = oracle_mod.quant_act_128x1(x)
    q2, s2 = oracle_mod.quant_act_1x128(np.ascontiguousarray(x.T))
    assert np.array_equal(qT, q2) and np.array_equal(sT, s2)
    assert qT.shape == (200, 256) and sT.shape == (2, 200)


def test_weight_blocks(oracle_mod):
    rng = np.random.default_rng(2)
    N, K = 384, 256
    w = rng.standard_normal((N, K)).astype(np.float32) * 0.02
    # block (nb, kb) gets a distinct power-of-two max-abs element
    for nb in range(3):
        for kb in range(2):
            w[nb * 128 + 5 * kb + nb, kb * 128 + 11 * nb + kb] = 2.0 ** (nb + 3 * kb)
    bits = f32_to_bf16_bits(w)
    q, s, qT, sT = oracle_mod.quant_weight_128x128(bits, transposed=True)
    for nb in range(3):
        for kb in range(2):
            assert s[nb, kb] == np.float32(2.0 ** (nb + 3 * kb)) / np.float32(448)
            assert q[nb * 128 + 5 * kb + nb, kb * 128 + 11 * nb + kb] == 0x7E
    assert np.array_equal(qT, q.T) and np.array_equal(sT, s.T)
    s_elem = np.repeat(np.repeat(s, 128, axis=0), 128, axis=1)
    _check_invariants(oracle_mod, bf16_bits_to_f32(bits), q, s_elem)
    q_only, s_only = oracle_mod.quant_weight_128x128(bits)
    assert np.array_equal(q_only, q) and np.array_equal(s_only, s)


def test_requant_identity_when_columns_reach_448(oracle_mod):
    """Codes with s = 1 whose every 128x1 group contains +-448: re-tiling
    reproduces the transposed codes and unit scales exactly."""
    rng = np.random.default_rng(3)
    M, K = 256, 256
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    q = rng.choice(finite, size=(M, K)).astype(np.uint8)
    for mb in range(M // 128):
        q[mb * 128 + (np.arange(K) % 128), np.arange(K)] = 0x7E
    s = np.ones((K // 128, M), np.float32)
    qT, sT = oracle_mod.requant_1x128_to_128x1(q, s)
    assert np.all(sT == 1.0)
    assert np.array_equal(qT, q.T)


def test_requant_matches_128x1_quant_of_dequantized(oracle_mod):
    """When x_hat = dec(q) * s is bf16-exact (power-of-two scales), the
    re-tiling equals the 128x1 quantizer applied to x_hat."""
    rng = np.random.default_rng(4)
    M, K = 256, 384
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    q = rng.choice(finite, size=(M, K)).astype(np.uint8)
    s = (2.0 ** rng.integers(-8, 8, size=(K // 128, M))).astype(np.float32)
    xhat = oracle_mod.e4m3_decode_array(q) * np.repeat(s.T, 128, axis=1)
    xbits = f32_to_bf16_bits(xhat.astype(np.float32))
    assert np.array_equal(bf16_bits_to_f32(xbits).astype(np.float64), xhat)
    qT, sT = oracle_mod.requant_1x128_to_128x1(q, s)
    qT2, sT2 = oracle_mod.quant_act_128x1(xbits)
    assert np.array_equal(qT, qT2) and np.array_equal(sT, sT2)


def test_requant_general_invariants(oracle_mod):
    rng = np.random.default_rng(6)
    x, _ = normal_with_outlier_columns(rng, (256, 256), 2, 100.0)
    q, s = oracle_mod.quant_act_1x128(x)
    qT, sT = oracle_mod.requant_1x128_to_128x1(q, s)
    xhat = (oracle_mod.e4m3_decode_array(q).astype(np.float32)
            * np.repeat(s.T, 128, axis=1))  # float32 multiply, as defined
    s_elem = np.repeat(sT.T, 128, axis=1)  # [K, M]
    _check_invariants(oracle_mod, xhat.T.astype(np.float32), qT, s_elem)


def test_rowwise(oracle_mod):
    rng = np.random.default_rng(8)
    x = normal(rng, (8, 512))
    q, s = oracle_mod.quant_rowwise(x)
    xf = bf16_bits_to_f32(x)
    amax = np.abs(xf).max(axis=1)
    for kb in range(4):
        assert np.array_equal(s[kb], (amax / np.float32(448)).astype(np.float32))
    _check_invariants(oracle_mod, xf, q, np.repeat(s[:1].T, 512, axis=1))


def test_f32_1x128_equals_bf16_rule_on_bf16_values(oracle_mod):
    """On values that are exactly bf16 the FP32-input quantizer is the bf16
    one (same rule, same arithmetic)."""
    rng = np.random.default_rng(31)
    bits, _ = synth.normal_with_outlier_columns(rng, (64, 512), 3, 100.0)
    q16, s16 = oracle_mod.quant_act_1x128(bits)
    q32, s32 = oracle_mod.quant_f32_1x128(synth.bf16_bits_to_f32(bits))
    assert np.array_equal(q16, q32) and np.array_equal(s16.view(np.uint32), s32.view(np.uint32))


def test_f32_1x128_invariants(oracle_mod):
    """Full-precision FP32 inputs: every element within half an E4M3 step
    (plus the FP32 quotient's rounding) of its dequantized code, and the
    tile maximum maps to 448."""
    rng = np.random.default_rng(32)
    x = (rng.standard_normal((32, 256)) * 10.0 ** rng.uniform(-3, 3, (32, 1))).astype(np.float32)
    x[3, :128] = 0.0
    q, s = oracle_mod.quant_f32_1x128(x)
    dec = oracle_mod.e4m3_decode_array(q)
    for m in range(32):
        for kb in range(2):
            sc = float(s[kb, m])
            xs = x[m, kb * 128:(kb + 1) * 128].astype(np.float64)
            d = dec[m, kb * 128:(kb + 1) * 128]
            if sc == 0.0:
                assert np.all(d == 0.0)
                continue
            y = np.abs(xs / sc)
            e = np.floor(np.log2(np.maximum(y, 2.0 ** -6)))
            half_ulp = 0.5 * np.where(y < 2.0 ** -6, 2.0 ** -9, 2.0 ** (e - 3))
            assert np.all(np.abs(xs - d * sc) <= (half_ulp + 2.0 ** -24 * y) * sc + 1e-300)
            assert np.max(np.abs(d)) == 448.0


def _tiles_with_common_max(rng, rows, cols, peak):
    """bf16 bits whose every 1x128 tile holds +-peak exactly once, the rest
    N(0, 1) below it in magnitude."""
    x = np.clip(rng.standard_normal((rows, cols)), -0.9 * peak, 0.9 * peak).astype(np.float32)
    for kb in range(cols // 128):
        j = rng.integers(0, 128, rows)
        x[np.arange(rows), kb * 128 + j] = np.where(rng.random(rows) < 0.5, -peak, peak)
    return f32_to_bf16_bits(x)


def test_per_tensor_equals_1x128_when_every_tile_holds_the_max(oracle_mod):
    """One scale for the tensor is the 1x128 scale of every tile when every
    tile has the tensor's max-abs, so the codes must agree."""
    rng = np.random.default_rng(41)
    bits = _tiles_with_common_max(rng, 48, 384, 3.0)
    q_t, s_t = oracle_mod.quant_per_tensor(bits)
    q_g, s_g = oracle_mod.quant_act_1x128(bits)
    assert np.all(s_g == s_t) and np.array_equal(q_t, q_g)
    assert s_t == np.float32(3.0) / np.float32(448.0)


def test_per_tensor_unit_scale_is_plain_encoding(oracle_mod):
    """A tensor whose max-abs is 448 has scale 1, so each code is the plain
    E4M3 rounding of the value (x / 1 = x)."""
    rng = np.random.default_rng(42)
    x = (rng.standard_normal((16, 64)) * 40.0).astype(np.float32)
    x[3, 7] = -448.0
    bits = f32_to_bf16_bits(np.clip(x, -448.0, 448.0))
    q, s = oracle_mod.quant_per_tensor(bits)
    assert s == np.float32(1.0)
    vals = bf16_bits_to_f32(bits)
    assert all(q.flat[i] == oracle_mod.e4m3_encode(float(vals.flat[i])) for i in range(vals.size))


def test_per_tensor_specials_and_outlier(oracle_mod):
    """NaN is ignored by the max and encodes as 0x7F; an all-zero tensor has
    scale 0 and signed-zero codes; one outlier sets the scale of everything
    (the outlier sensitivity that motivates the 1x128 tiles)."""
    z = f32_to_bf16_bits(np.array([[0.0, -0.0] * 8], np.float32))
    q, s = oracle_mod.quant_per_tensor(z)
    assert s == 0.0 and np.array_equal(q[0], np.array([0x00, 0x80] * 8, np.uint8))
    x = np.full((2, 16), 1.0, np.float32)
    x[0, 0] = np.nan
    x[1, 5] = 2.0 ** 20
    q, s = oracle_mod.quant_per_tensor(f32_to_bf16_bits(x))
    assert s == np.float32(2.0 ** 20) / np.float32(448.0)
    assert q[0, 0] == 0x7F and q[1, 5] == 0x7E
    # 1.0 / s = 448 * 2^-20 < 2^-9 / 2 (half the smallest subnormal): code 0
    assert np.all(np.delete(q.ravel(), [0, 21]) == 0x00)
