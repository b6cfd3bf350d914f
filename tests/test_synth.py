"""The seeded input generators follow the stated workload recipes: shapes,
seed determinism, outlier channels and their factors, and the value
distributions (normal widths, Student-t nu=4, log-uniform row magnitudes),
plus the bf16 rounding they apply."""
import numpy as np
import pytest

import synth
from synth import bf16_bits_to_f32, f32_to_bf16_bits


def _f(bits):
    return bf16_bits_to_f32(bits).astype(np.float64)


def test_bf16_rounding():
    x = np.array([1.0, 1.0 + 2.0 ** -8, 1.0 + 3 * 2.0 ** -8, -2.5, 3.0e38, np.inf, np.nan],
                 np.float32)
    b = f32_to_bf16_bits(x)
    # halfway cases round to the even neighbour: 1 + 2^-8 -> 1.0,
    # 1 + 3 * 2^-8 -> 1 + 2^-6
    assert list(_f(b[:4])) == [1.0, 1.0, 1.0 + 2.0 ** -6, -2.5]
    assert b[5] == 0x7F80 and b[6] == 0x7FC0
    assert np.isfinite(_f(b[4:5])).all()


@pytest.mark.parametrize("name", ["tiny", "dense", "moe", "bwd", "stress"])
def test_shapes_and_determinism(name):
    w = synth.WORKLOADS[name]
    rows = min(w.M, 256)
    a1 = synth.make_inputs(name, scale_rows=rows)
    a2 = synth.make_inputs(name, scale_rows=rows)
    other = synth.make_inputs(name, scale_rows=rows, seed=w.seed + 100)
    if name == "bwd":
        assert a1["X"].shape == (rows, w.K) and a1["W"].shape == (w.N, w.K)
        assert a1["dY"].shape == (rows, w.N)
    else:
        assert a1["A"].shape == (rows, w.K) and a1["B"].shape == (w.N, w.K)
    for k in a1:
        assert a1[k].dtype == np.uint16
        assert np.array_equal(a1[k], a2[k])
        assert not np.array_equal(a1[k], other[k])


def _outlier_columns(bits, factor):
    std = _f(bits).std(axis=0)
    typical = np.median(std)
    big = np.flatnonzero(std > typical * factor / 3)
    return big, std[big] / typical


@pytest.mark.parametrize("name,key,count,factor", [
    ("tiny", "A", 4, 50.0), ("dense", "A", 7, 100.0), ("bwd", "X", 2, 100.0)])
def test_outlier_channels(name, key, count, factor):
    bits = synth.make_inputs(name, scale_rows=512)[key]
    cols, ratio = _outlier_columns(bits, factor)
    assert len(cols) == count
    assert np.all(np.abs(ratio / factor - 1.0) < 0.25)


def test_widths_and_distributions():
    tiny = synth.make_inputs("tiny")
    assert abs(_f(tiny["B"]).std() / 0.02 - 1.0) < 0.02
    bwd = synth.make_inputs("bwd", scale_rows=256)
    assert abs(_f(bwd["W"]).std() / 0.02 - 1.0) < 0.01
    assert abs(_f(bwd["dY"]).std() / 1e-3 - 1.0) < 0.01
    # Student-t, nu = 4: variance nu / (nu - 2) = 2, heavy tails
    t = _f(synth.make_inputs("moe", scale_rows=512)["A"]).ravel()
    assert abs(t.var() / 2.0 - 1.0) < 0.1
    assert np.mean(np.abs(t) > 4.604) == pytest.approx(0.01, abs=0.002)  # t_4 two-sided 1%
    # stress rows: U(-1, 1) times 10^U(-2, 2) per row
    s = _f(synth.make_inputs("stress", scale_rows=2048)["A"])
    row_max = np.abs(s).max(axis=1)
    lg = np.log10(row_max)
    assert lg.min() > -2.01 and lg.max() < 2.01
    assert np.histogram(lg, bins=4, range=(-2, 2))[0].min() > 0.2 * len(lg)
    # within a row: uniform on (-row magnitude, +row magnitude)
    ratio = np.abs(s) / row_max[:, None]
    assert abs(ratio.mean() - 0.5) < 0.01
