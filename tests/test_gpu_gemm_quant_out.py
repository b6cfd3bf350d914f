"""GEMM with the next layer's 1x128 quantization fused into its epilogue
(page P2, paragraph 1: the BF16 GEMM output otherwise goes through HBM
once more to be quantized; page P1, paragraph 3: the 1x128 rule).

The fused kernel computes the same FP32 sums as the FP32-output GEMM of the
same tile shape (the 256 x 256 CTA pair), so its codes and scales must equal,
bit for bit, the oracle's 1x128 quantizer applied to that kernel's own FP32
output.  Separately, the dequantized result is compared with the oracle's
double-precision GEMM: each element within half an E4M3 step of it (plus the
GEMM tolerance)."""
import numpy as np
import pytest
import torch

import synth
from tests._helpers import assert_codes_equal, assert_scales_equal, dev, host

pytestmark = pytest.mark.gpu

BLOCK, TILE = 0, 1
TILE_256x256_PAIR = 6


def _inputs(oracle_mod, M, N, K, seed, bkind):
    rng = np.random.default_rng(seed)
    a_bits, _ = synth.normal_with_outlier_columns(rng, (M, K), 3, 50.0)
    a, sa = oracle_mod.quant_act_1x128(a_bits)
    if bkind == BLOCK:
        b, sb = oracle_mod.quant_weight_128x128(synth.normal(rng, (N, K), 0.02))
    else:
        b, sb = oracle_mod.quant_act_1x128(synth.normal(rng, (N, K), 1e-3))
    return a, sa, b, sb


def _check(fp8bs, oracle_mod, a, sa, b, sb, bkind, what, ref=None):
    da, dsa, db, dsb = dev(a), dev(sa), dev(b), dev(sb)
    M, N = a.shape[0], b.shape[0]
    # sentinels: every code and scale must be written
    c = torch.full((M, N), 0xAA, dtype=torch.uint8, device="cuda")
    cs = torch.full((N // 128, M), float("nan"), dtype=torch.float32, device="cuda")
    fp8bs.gemm_quant_out(da, dsa, db, dsb, bkind, out=c, out_scales=cs)
    c32 = host(fp8bs.gemm(da, dsa, db, dsb, bkind, out_dtype=torch.float32,
                          tile=TILE_256x256_PAIR))
    torch.cuda.synchronize()
    q_ref, s_ref = oracle_mod.quant_f32_1x128(c32)
    assert_codes_equal(c, q_ref, what + " codes")
    assert_scales_equal(cs, s_ref, what + " scales")
    if ref is not None:
        # half an E4M3 step: 2^-4 relative for normal codes, s * 2^-10 for
        # subnormal ones; plus the GEMM's own tolerance on the FP32 sums
        deq = oracle_mod.e4m3_decode_array(host(c)) * np.repeat(
            host(cs).T.astype(np.float64), 128, axis=1)
        s_el = np.repeat(host(cs).T.astype(np.float64), 128, axis=1)
        bound = 2.0 ** -4 * np.abs(ref) + s_el * 2.0 ** -10 + 5e-3 * np.abs(ref).max()
        assert np.all(np.abs(deq - ref) <= bound), what


@pytest.mark.parametrize("bkind", [BLOCK, TILE])
@pytest.mark.parametrize("M,N,K", [(1, 128, 128), (128, 256, 256), (300, 640, 640),
                                   (513, 384, 1152)])
def test_fused_quant_bit_exact(fp8bs, oracle_mod, bkind, M, N, K):
    a, sa, b, sb = _inputs(oracle_mod, M, N, K, 7 + M + N + K, bkind)
    ref = oracle_mod.gemm(a, sa, b, sb, bkind)
    _check(fp8bs, oracle_mod, a, sa, b, sb, bkind, f"{M}x{N}x{K}", ref)


def test_fused_quant_special_values(fp8bs, oracle_mod):
    """A NaN code in a B row makes that output column NaN (code 0x7F, the
    group's scale from its other elements); an all-zero A row gives scale 0
    and zero codes, except the NaN column."""
    M, N, K = 256, 512, 256
    a, sa, b, sb = _inputs(oracle_mod, M, N, K, 99, BLOCK)
    a = a.copy()
    b = b.copy()
    b[5, 17] = 0x7F
    a[3, :] = 0
    _check(fp8bs, oracle_mod, a, sa, b, sb, BLOCK, "special")
    c, cs = fp8bs.gemm_quant_out(dev(a), dev(sa), dev(b), dev(sb), BLOCK)
    c, cs = host(c), host(cs)
    assert np.all(c[:, 5] == 0x7F)
    assert np.all(np.delete(c[3], 5) == 0) and np.all(cs[:, 3] == 0)


def test_fused_quant_rejects_ragged_n(fp8bs):
    a = torch.zeros((128, 128), dtype=torch.uint8, device="cuda")
    sa = torch.ones((1, 128), dtype=torch.float32, device="cuda")
    b = torch.zeros((144, 128), dtype=torch.uint8, device="cuda")
    sb = torch.ones((2, 1), dtype=torch.float32, device="cuda")
    with pytest.raises(fp8bs.Fp8bsError):
        fp8bs.gemm_quant_out(a, sa, b, sb, BLOCK,
                             out_scales=torch.empty((2, 128), dtype=torch.float32,
                                                    device="cuda"))


def test_fused_quant_dense_full_size(fp8bs, oracle_mod):
    """The dense projection workload (M=4096, K=N=7168), every code and scale."""
    inp = synth.make_inputs("dense")
    a, sa = oracle_mod.quant_act_1x128(inp["A"])
    b, sb = oracle_mod.quant_weight_128x128(inp["B"])
    _check(fp8bs, oracle_mod, a, sa, b, sb, BLOCK, "dense")
