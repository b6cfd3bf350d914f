"""E5M6 cache of the re-tiled activations (page P1, paragraph 3): GPU parity
with the oracle, bit for bit, for the cache itself (packed codes and
scales), for the E4M3 codes the same launch writes, and for the re-tiling of
the cache into 128x1 E4M3 tiles for the weight gradient.  Plus the reason for
the format, measured: re-tiling from E5M6 adds less error than re-tiling
from the E4M3 1x128 codes."""
import numpy as np
import pytest
import torch

import synth
from tests._helpers import assert_codes_equal, assert_scales_equal, dev, dev_bf16, host

pytestmark = pytest.mark.gpu


def _check_quant(fp8bs, oracle_mod, bits, what, with_e4m3=True):
    packed, s5, q, s = fp8bs.quant_act_e5m6(dev_bf16(bits), with_e4m3=with_e4m3)
    p_ref, s5_ref = oracle_mod.quant_act_e5m6_1x128(bits)
    assert_codes_equal(packed, p_ref, what + " packed E5M6")
    assert_scales_equal(s5, s5_ref, what + " E5M6 scales")
    if with_e4m3:
        q_ref, s_ref = oracle_mod.quant_act_1x128(bits)
        assert_codes_equal(q, q_ref, what + " E4M3 codes")
        assert_scales_equal(s, s_ref, what + " E4M3 scales")
    return packed, s5


@pytest.mark.parametrize("M,K", [(1, 128), (37, 256), (300, 1024), (128, 7168)])
def test_quant_e5m6_bit_exact(fp8bs, oracle_mod, M, K):
    rng = np.random.default_rng(M + K)
    bits, _ = synth.normal_with_outlier_columns(rng, (M, K), 3, 100.0)
    _check_quant(fp8bs, oracle_mod, bits, f"{M}x{K}")
    _check_quant(fp8bs, oracle_mod, bits, f"{M}x{K} cache only", with_e4m3=False)


def test_quant_e5m6_special_values(fp8bs, oracle_mod):
    rng = np.random.default_rng(2)
    x = rng.standard_normal((8, 512)).astype(np.float32)
    x[0, :128] = 0.0
    x[0, 7] = -0.0
    x[1, 3] = np.nan
    x[2, 130] = np.inf
    x[2, 131] = -np.inf
    x[3, 256:384] = (rng.integers(-127, 128, 128) * 2.0 ** -133).astype(np.float32)  # bf16 subnormals
    x[4, 384:] *= 1e30
    x[5, :128] *= 2.0 ** -60  # small groups
    x[6, 128:256] = rng.uniform(-1, 1, 128) * 2.0 ** -20  # quotients near the E5M6 subnormals
    x[6, 130] = 1.0
    _check_quant(fp8bs, oracle_mod, synth.f32_to_bf16_bits(x), "specials")


def test_quant_e5m6_full_size(fp8bs, oracle_mod):
    """The backward workload's cached activation X (4096 x 2048)."""
    _check_quant(fp8bs, oracle_mod, synth.make_inputs("bwd")["X"], "bwd X")


def _check_requant(fp8bs, oracle_mod, packed, s5, what):
    qT, sT = fp8bs.requant_e5m6_to_128x1(dev(packed), dev(s5))
    q_ref, s_ref = oracle_mod.requant_e5m6_to_128x1(packed, s5)
    assert_codes_equal(qT, q_ref, what + " codes")
    assert_scales_equal(sT, s_ref, what + " scales")


@pytest.mark.parametrize("M,K", [(128, 128), (256, 384), (1024, 1024)])
def test_requant_e5m6_bit_exact(fp8bs, oracle_mod, M, K):
    """Input written by the oracle (random finite codes, random scales), so
    the re-tiling is checked on its own."""
    rng = np.random.default_rng(M * 3 + K)
    codes = rng.integers(0, 0x7C0, (M, K)).astype(np.uint16) | \
        (rng.integers(0, 2, (M, K)).astype(np.uint16) << 11)
    s5 = (rng.uniform(0.5, 2.0, (K // 128, M)) * 10.0 ** rng.uniform(-8, 2, (K // 128, M))) \
        .astype(np.float32)
    _check_requant(fp8bs, oracle_mod, oracle_mod.e5m6_pack(codes), s5, f"{M}x{K}")


def test_requant_e5m6_special_codes(fp8bs, oracle_mod):
    rng = np.random.default_rng(4)
    M, K = 256, 256
    codes = rng.integers(0, 0x7C0, (M, K)).astype(np.uint16)
    codes[5, 9] = 0x7FF     # NaN
    codes[9, 130] = 0x7C0   # Inf
    codes[:128, 200] = 0     # an all-zero column group
    codes[130, :] = 0x800    # negative zeros
    s5 = rng.uniform(0.5, 2.0, (K // 128, M)).astype(np.float32)
    s5[0, 17] = 0.0
    _check_requant(fp8bs, oracle_mod, oracle_mod.e5m6_pack(codes), s5, "special codes")


def test_e5m6_chain_full_size(fp8bs, oracle_mod):
    """Quantize X to the cache and re-tile it, all on the GPU, against the
    oracle's chain."""
    bits = synth.make_inputs("bwd")["X"]
    packed, s5, _, _ = fp8bs.quant_act_e5m6(dev_bf16(bits), with_e4m3=False)
    qT, sT = fp8bs.requant_e5m6_to_128x1(packed, s5)
    p_ref, s5_ref = oracle_mod.quant_act_e5m6_1x128(bits)
    q_ref, s_ref = oracle_mod.requant_e5m6_to_128x1(p_ref, s5_ref)
    assert_codes_equal(qT, q_ref, "chain codes")
    assert_scales_equal(sT, s_ref, "chain scales")


def test_e5m6_cache_reduces_retiling_error(fp8bs, oracle_mod):
    """Relative error of the 128x1 E4M3 operand against X itself, for three
    routes: quantizing X directly (no cache), re-tiling the E4M3 1x128 cache,
    and re-tiling the E5M6 cache."""
    bits = synth.make_inputs("bwd")["X"]
    x = synth.bf16_bits_to_f32(bits).astype(np.float64)
    xd = dev_bf16(bits)

    def err(qT, sT):
        d = oracle_mod.e4m3_decode_array(host(qT)).T * np.repeat(host(sT), 128, axis=0)
        return float(np.linalg.norm(d - x) / np.linalg.norm(x))

    e_direct = err(*fp8bs.quant_act_1x128(xd, transpose_out=True))
    q8, s8 = fp8bs.quant_act_1x128(xd)
    e_e4m3 = err(*fp8bs.requant_1x128_to_128x1(q8, s8))
    packed, s5, _, _ = fp8bs.quant_act_e5m6(xd, with_e4m3=False)
    e_e5m6 = err(*fp8bs.requant_e5m6_to_128x1(packed, s5))
    print(f"\n128x1 operand vs X: direct {e_direct:.4e}  via E4M3 cache {e_e4m3:.4e}  "
          f"via E5M6 cache {e_e5m6:.4e}")
    assert e_e5m6 < e_e4m3
    assert e_e5m6 <= 1.01 * e_direct
