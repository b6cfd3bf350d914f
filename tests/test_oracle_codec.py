"""Pins of the oracle's E4M3 codec to the OCP FP8 E4M3FN definition.

Independent evidence only: the format's published closed forms, brute force
over all 256 codes, exact midpoints, and PyTorch's own float8_e4m3fn
conversion (a separate library routine) on the in-range values.
"""
import math

import numpy as np
import pytest
import torch

pytestmark = []


def test_closed_forms(oracle_mod):
    o = oracle_mod
    # OCP FP8 E4M3: max normal S.1111.110 = 1.75*2^8, min normal S.0001.000 =
    # 2^-6, max subnormal S.0000.111 = 0.875*2^-6, min subnormal 2^-9.
    assert o.e4m3_decode(0x7E) == 448.0
    assert o.e4m3_decode(0x08) == 2.0 ** -6
    assert o.e4m3_decode(0x07) == 0.875 * 2.0 ** -6
    assert o.e4m3_decode(0x01) == 2.0 ** -9
    assert o.e4m3_decode(0x38) == 1.0
    assert o.e4m3_decode(0xFE) == -448.0
    assert math.isnan(o.e4m3_decode(0x7F)) and math.isnan(o.e4m3_decode(0xFF))
    z = o.e4m3_decode(0x80)
    assert z == 0.0 and math.copysign(1.0, z) < 0


def test_decode_matches_torch_all_codes(oracle_mod):
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    mine = np.array([oracle_mod.e4m3_decode(c) for c in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(mine), nan)
    assert np.array_equal(mine[~nan], ref[~nan])
    assert np.array_equal(np.signbit(mine[~nan]), np.signbit(ref[~nan]))
    assert nan.sum() == 2


def test_round_trip_every_finite_code(oracle_mod):
    o = oracle_mod
    for c in range(256):
        v = o.e4m3_decode(c)
        if math.isnan(v):
            assert o.e4m3_encode(v) == 0x7F
            continue
        assert o.e4m3_encode(v) == c, hex(c)


def _f32_next(x, direction):
    return float(np.nextafter(np.float32(x), np.float32(direction)))


def test_midpoints_ties_to_even(oracle_mod):
    o = oracle_mod
    for c in range(0x00, 0x7E):
        lo, hi = o.e4m3_decode(c), o.e4m3_decode(c + 1)
        mid = (lo + hi) / 2  # at most 5 significant bits: exact in float32
        assert float(np.float32(mid)) == mid
        even = c if c % 2 == 0 else c + 1
        assert o.e4m3_encode(mid) == even, hex(c)
        assert o.e4m3_encode(-mid) == 0x80 | even
        assert o.e4m3_encode(_f32_next(mid, -np.inf)) == c
        assert o.e4m3_encode(_f32_next(mid, np.inf)) == c + 1
        assert o.e4m3_encode(-_f32_next(mid, np.inf)) == 0x80 | (c + 1)


def test_saturation_and_specials(oracle_mod):
    o = oracle_mod
    for y in (448.0, 448.03125, 463.99997, 464.0, 464.00003, 480.0, 1e6, 3.0e38, math.inf):
        assert o.e4m3_encode(y) == 0x7E, y
        assert o.e4m3_encode(-y) == 0xFE, y
    assert o.e4m3_encode(math.nan) == 0x7F
    assert o.e4m3_encode(0.0) == 0x00
    assert o.e4m3_encode(-0.0) == 0x80
    # below half the smallest subnormal -> zero, sign kept
    assert o.e4m3_encode(2.0 ** -11) == 0x00
    assert o.e4m3_encode(-(2.0 ** -11)) == 0x80
    assert o.e4m3_encode(1e-45) == 0x00


def test_encode_matches_torch_in_range(oracle_mod):
    """torch's float -> float8_e4m3fn cast is RNE for |y| <= 464 (it returns
    NaN above, so the comparison stops there)."""
    rng = np.random.default_rng(123)
    ys = np.concatenate([
        rng.uniform(-464, 464, 4000),
        rng.standard_normal(4000) * 10.0 ** rng.uniform(-4, 2, 4000),
        (rng.uniform(-1, 1, 2000) * 2.0 ** -6),
    ]).astype(np.float32)
    ref = torch.from_numpy(ys).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    mine = np.array([oracle_mod.e4m3_encode(float(y)) for y in ys], dtype=np.uint8)
    assert np.array_equal(mine, ref)


def test_encode_is_nearest_by_brute_force(oracle_mod):
    """Against an exhaustive nearest search over all finite codes."""
    o = oracle_mod
    vals = [(c, o.e4m3_decode(c)) for c in range(256) if not math.isnan(o.e4m3_decode(c))]
    rng = np.random.default_rng(7)
    ys = (rng.standard_normal(1500) * 10.0 ** rng.uniform(-3, 2.6, 1500)).astype(np.float32)
    for y in ys:
        y = float(y)
        if abs(y) >= 448:
            continue
        best = min(abs(y - v) for _, v in vals)
        c = o.e4m3_encode(y)
        assert abs(y - o.e4m3_decode(c)) == best
        assert (c & 0x80) == (0x80 if y < 0 else 0)


def test_bf16_helpers_match_torch(oracle_mod):
    o = oracle_mod
    rng = np.random.default_rng(5)
    xs = (rng.standard_normal(3000) * 10.0 ** rng.uniform(-40, 38, 3000)).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    mine = o.double_to_bf16_array(xs.astype(np.float64))
    assert np.array_equal(mine, ref)
    for b in (0x0000, 0x8000, 0x3F80, 0x7F7F, 0x0001, 0xC2F7):
        t = torch.tensor([b], dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float().item()
        assert o.bf16_to_float(b) == t or (math.isnan(t) and math.isnan(o.bf16_to_float(b)))
