"""Pins of the oracle GEMM: C = sum over k of dequantized products, with each
128-wide K-group carrying its own scale pair (page 1, paragraph 2; page 4,
paragraph 4).  Independent evidence: exact rational arithmetic on tiny
inputs, one-hot probes of every scale index, and an exact integer case.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

BLOCK, TILE = 0, 1


def _torch_decode(codes):
    return torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8)).view(
        torch.float8_e4m3fn).to(torch.float64).numpy()


def _finite_codes(rng, shape):
    finite = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    return rng.choice(finite, size=shape).astype(np.uint8)


@pytest.mark.parametrize("bkind", [BLOCK, TILE])
def test_exact_rational_tiny(oracle_mod, bkind):
    rng = np.random.default_rng(11)
    M, N, K = 3, 130, 256  # N spans two 128-row blocks of B
    a = _finite_codes(rng, (M, K))
    b = _finite_codes(rng, (N, K))
    sa = rng.uniform(0.01, 3.0, (K // 128, M)).astype(np.float32)
    if bkind == BLOCK:
        sb = rng.uniform(0.01, 3.0, (2, K // 128)).astype(np.float32)
    else:
        sb = rng.uniform(0.01, 3.0, (K // 128, N)).astype(np.float32)
    c = oracle_mod.gemm(a, sa, b, sb, bkind)
    da, db = _torch_decode(a), _torch_decode(b)
    for m in range(M):
        for n in (0, 1, 127, 128, 129):
            exact = Fraction(0)
            for k in range(K):
                ska = Fraction(float(sa[k // 128, m]))
                skb = Fraction(float(sb[n // 128, k // 128] if bkind == BLOCK else sb[k // 128, n]))
                exact += Fraction(da[m, k]) * ska * Fraction(db[n, k]) * skb
            err = abs(Fraction(c[m, n]) - exact)
            scale = sum(abs(Fraction(da[m, k]) * Fraction(db[n, k])) for k in range(K)) * 9
            assert err <= scale * Fraction(1, 2 ** 50), (m, n)


@pytest.mark.parametrize("bkind", [BLOCK, TILE])
def test_one_hot_scale_indices(oracle_mod, bkind):
    """A one at (m, k) and at (n, k): C[m][n] = sa(m, k) * sb(n, k) exactly,
    with every scale a distinct power of two, so a transposed or shifted
    index shows up."""
    M, N, K = 5, 256, 384
    KB = K // 128
    sa = (2.0 ** (np.arange(KB * M).reshape(KB, M) - 7)).astype(np.float32)
    if bkind == BLOCK:
        sb = (2.0 ** (-np.arange(2 * KB).reshape(2, KB) - 20)).astype(np.float32)
    else:
        sb = (2.0 ** (-(np.arange(KB * N) % 60).reshape(KB, N) - 20)).astype(np.float32)
    for (m, n, k) in [(0, 0, 0), (4, 255, 383), (2, 130, 200), (3, 127, 128), (1, 128, 255)]:
        a = np.zeros((M, K), np.uint8)
        b = np.zeros((N, K), np.uint8)
        a[m, k] = 0x38  # 1.0
        b[n, k] = 0xC0  # -2.0
        c = oracle_mod.gemm(a, sa, b, sb, bkind)
        sbv = sb[n // 128, k // 128] if bkind == BLOCK else sb[k // 128, n]
        expect = -2.0 * float(sa[k // 128, m]) * float(sbv)
        assert c[m, n] == expect
        mask = np.ones_like(c, bool)
        mask[m, n] = False
        assert np.all(c[mask] == 0)


def test_integer_case_exact(oracle_mod):
    """Unit scales and small-integer codes: C is an exact integer matmul."""
    rng = np.random.default_rng(12)
    ints = {v: c for c in range(256) for v in [float(_torch_decode(np.array([c]))[0])]
            if v == v and v == int(v) and abs(v) <= 16}
    vals = np.array(sorted(ints))
    M, N, K = 7, 128, 512
    ai = rng.choice(vals, size=(M, K)).astype(np.int64)
    bi = rng.choice(vals, size=(N, K)).astype(np.int64)
    a = np.vectorize(lambda v: ints[float(v)])(ai).astype(np.uint8)
    b = np.vectorize(lambda v: ints[float(v)])(bi).astype(np.uint8)
    sa = np.ones((K // 128, M), np.float32)
    sb = np.ones((1, K // 128), np.float32)
    c = oracle_mod.gemm(a, sa, b, sb, BLOCK)
    assert np.array_equal(c, (ai @ bi.T).astype(np.float64))


def test_sampled_equals_full(oracle_mod):
    rng = np.random.default_rng(13)
    M, N, K = 9, 256, 256
    a = _finite_codes(rng, (M, K)); b = _finite_codes(rng, (N, K))
    sa = rng.uniform(0.1, 1, (2, M)).astype(np.float32)
    sb = rng.uniform(0.1, 1, (2, 2)).astype(np.float32)
    full = oracle_mod.gemm(a, sa, b, sb, BLOCK)
    ms = rng.integers(0, M, 50); ns = rng.integers(0, N, 50)
    samp = oracle_mod.gemm_sampled(a, sa, b, sb, BLOCK, ms, ns)
    assert np.array_equal(samp, full[ms, ns])


def test_limited_acc_special_cases(oracle_mod):
    """Parity of the accumulator model itself is unpinned; its two limits
    are not: with 53 kept bits it is the exact sum, and products that are
    small integers never lose a bit at 14."""
    rng = np.random.default_rng(14)
    M, N, K = 4, 128, 512
    a = _finite_codes(rng, (M, K)); b = _finite_codes(rng, (N, K))
    sa = np.ones((K // 128, M), np.float32); sb = np.ones((1, K // 128), np.float32)
    ms = np.repeat(np.arange(M), 8); ns = np.tile(np.arange(0, 128, 16), M)
    exact = oracle_mod.gemm_sampled(a, sa, b, sb, BLOCK, ms, ns)
    wide = oracle_mod.gemm_limited_acc(a, sa, b, sb, BLOCK, ms, ns, bits=53, group=32,
                                       promote_every=0)
    # 53 kept bits: only the truncation back to FP32 after each of the K/32
    # groups loses anything, at most one FP32 ulp of a partial sum each
    da, db = _torch_decode(a), _torch_decode(b)
    abs_sum = np.abs(da[ms] * db[ns]).sum(axis=1)
    assert np.all(np.abs(wide - exact) <= (K // 32) * 2.0 ** -23 * abs_sum)
    one = np.full((M, K), 0x38, np.uint8)  # 1.0
    two = np.full((N, K), 0x40, np.uint8)  # 2.0
    r = oracle_mod.gemm_limited_acc(one, sa, two, sb, BLOCK, ms, ns, bits=14, group=32,
                                    promote_every=128)
    assert np.all(r == 2.0 * K)
    # and the model does lose accuracy at K = 4096 with wide-range magnitudes
    K2 = 4096
    a2 = _finite_codes(rng, (2, K2)); b2 = _finite_codes(rng, (128, K2))
    sa2 = np.ones((K2 // 128, 2), np.float32); sb2 = np.ones((1, K2 // 128), np.float32)
    ms2 = np.zeros(16, np.int64); ns2 = np.arange(16)
    ex2 = oracle_mod.gemm_sampled(a2, sa2, b2, sb2, BLOCK, ms2, ns2)
    lim = oracle_mod.gemm_limited_acc(a2, sa2, b2, sb2, BLOCK, ms2, ns2, bits=14, group=32,
                                      promote_every=0)
    assert not np.array_equal(lim, ex2)


def _one_row(codes_a, codes_b):
    """A 1x128 times 128x128-block operand pair with unit scales."""
    a = np.array([codes_a], np.uint8)
    b = np.zeros((128, 128), np.uint8)
    b[0] = codes_b
    return a, np.ones((1, 1), np.float32), b, np.ones((1, 1), np.float32)


def test_limited_acc_hand_worked(oracle_mod):
    """The accumulator model against its own stated steps, worked by hand:
    per group of 32 products, align everything to the largest exponent E,
    keep 14 bits below it (units of 2^(E-13)) by flooring each term
    (sign-fill right shift), add exactly, truncate to FP32."""
    one, tiny, neg_tiny = 0x38, 0x01, 0x81  # 1.0, 2^-9, -2^-9
    # 1.0 * 1.0 then 31 products of 2^-9 * 2^-9 = 2^-18: with E = 0 the unit
    # is 2^-13 and floor(2^-18 / 2^-13) = 0, so every tiny term is lost.
    codes_a = np.array([one] + [tiny] * 31 + [0] * 96, np.uint8)
    codes_b = np.array([one] + [tiny] * 31 + [0] * 96, np.uint8)
    a, sa, b, sb = _one_row(codes_a, codes_b)
    got = oracle_mod.gemm_limited_acc(a, sa, b, sb, BLOCK, [0], [0], bits=14, group=32)
    assert got[0] == 1.0
    assert oracle_mod.gemm(a, sa, b, sb, BLOCK)[0, 0] == 1.0 + 31 * 2.0 ** -18
    # negative tiny products: floor(-2^-5) = -1 unit each, so the group sums
    # to (2^13 - 31) units = 1 - 31 * 2^-13
    codes_b2 = np.array([one] + [neg_tiny] * 31 + [0] * 96, np.uint8)
    a, sa, b, sb = _one_row(codes_a, codes_b2)
    got = oracle_mod.gemm_limited_acc(a, sa, b, sb, BLOCK, [0], [0], bits=14, group=32)
    assert got[0] == 1.0 - 31 * 2.0 ** -13
    # the same tiny terms in a group of their own, with nothing larger: E is
    # their own exponent (-18), so they are kept exactly (31 * 2^-18)
    codes_a3 = np.array([tiny] * 31 + [0] * 97, np.uint8)
    a, sa, b, sb = _one_row(codes_a3, codes_a3)
    got = oracle_mod.gemm_limited_acc(a, sa, b, sb, BLOCK, [0], [0], bits=14, group=32)
    assert got[0] == 31 * 2.0 ** -18
