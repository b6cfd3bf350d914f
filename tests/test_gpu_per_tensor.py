"""Per-tensor FP8 scaling, the baseline the fine-grained tiles replace (page
P1, paragraph 4; page P3, paragraph 4: one scale per tensor, its max-abs
mapped to the FP8 maximum, which makes training sensitive to activation
outliers).

Parity: codes and the scale bit-identical to the oracle; the GEMM on
per-tensor codes within the GEMM tolerance of the oracle on the same codes.

Accuracy study (run with -s for the table): the error of the FP8 GEMM against
the exact product of the bf16 inputs, with 1x128 / 128x128 scales and with
per-tensor scales.  The pages' claim, checked here: 1x128 tiles confine an
outlier to its own tile, so rows without outliers keep their accuracy however
large the outlier is, while one scale per tensor pushes them towards the
bottom of E4M3's range (normal values span only 448 / 2^-6 = 28672)."""
import numpy as np
import pytest
import torch

import synth
from tests._helpers import (assert_codes_equal, assert_gemm_f32, assert_scales_equal, dev,
                            dev_bf16, host)

pytestmark = pytest.mark.gpu

BLOCK = 0


def _check_per_tensor(fp8bs, oracle_mod, bits, what, n_bcast=5):
    q, s, bc = fp8bs.quant_per_tensor(dev_bf16(bits), bcast_shape=(n_bcast,))
    q_ref, s_ref = oracle_mod.quant_per_tensor(bits)
    assert_codes_equal(q, q_ref, what + " codes")
    assert_scales_equal(s, np.array([s_ref], np.float32), what + " scale")
    assert_scales_equal(bc, np.full(n_bcast, s_ref, np.float32), what + " broadcast")
    return q, s


@pytest.mark.parametrize("rows,cols", [(1, 16), (37, 144), (256, 1024), (1000, 4096)])
def test_per_tensor_bit_exact(fp8bs, oracle_mod, rows, cols):
    rng = np.random.default_rng(rows * 7 + cols)
    bits, _ = synth.normal_with_outlier_columns(rng, (rows, cols), 3, 50.0)
    _check_per_tensor(fp8bs, oracle_mod, bits, f"{rows}x{cols}")


def _bits(vals):
    return synth.f32_to_bf16_bits(np.asarray(vals, np.float32))


def test_per_tensor_special_values(fp8bs, oracle_mod):
    rng = np.random.default_rng(3)
    base = rng.standard_normal((8, 64)).astype(np.float32)
    # all zeros, both signs: scale 0, signed-zero codes
    z = np.zeros((4, 32), np.float32)
    z[1, ::3] = -0.0
    _check_per_tensor(fp8bs, oracle_mod, _bits(z), "zeros")
    # NaN elements: ignored by the max, encoded 0x7F
    x = base.copy()
    x[2, 5] = np.nan
    x[7, 63] = -np.nan
    _check_per_tensor(fp8bs, oracle_mod, _bits(x), "nan")
    # an infinity: scale Inf, finite values to signed zero, Inf to NaN
    x = base.copy()
    x[0, 1] = np.inf
    x[4, 9] = np.nan
    _check_per_tensor(fp8bs, oracle_mod, _bits(x), "inf")
    # bf16 subnormals only: a scale below the fast path's range
    tiny = (rng.integers(-127, 128, (4, 48)) * 2.0 ** -133).astype(np.float32)
    _check_per_tensor(fp8bs, oracle_mod, _bits(tiny), "subnormal")
    # values near the bf16 maximum
    big = (rng.uniform(-1, 1, (4, 48)) * 3.0e38).astype(np.float32)
    _check_per_tensor(fp8bs, oracle_mod, _bits(big), "huge")


def test_per_tensor_full_size(fp8bs, oracle_mod):
    """The dense projection workload's activation and weight."""
    inp = synth.make_inputs("dense")
    _check_per_tensor(fp8bs, oracle_mod, inp["A"], "dense A")
    _check_per_tensor(fp8bs, oracle_mod, inp["B"], "dense W")


def _gemm_per_tensor(fp8bs, a_bits, w_bits):
    """GPU: both operands quantized per tensor, scales broadcast to the
    GEMM's layouts (A: [K/128][M], B blocks: [N/128][K/128])."""
    M, K = a_bits.shape
    N = w_bits.shape[0]
    qa, _, sa = fp8bs.quant_per_tensor(dev_bf16(a_bits), bcast_shape=(K // 128, M))
    qb, _, sb = fp8bs.quant_per_tensor(dev_bf16(w_bits), bcast_shape=((N + 127) // 128, K // 128))
    return qa, sa, qb, sb


def _gemm_fine(fp8bs, a_bits, w_bits):
    qa, sa = fp8bs.quant_act_1x128(dev_bf16(a_bits))
    qb, sb = fp8bs.quant_weight_128x128(dev_bf16(w_bits))
    return qa, sa, qb, sb


def test_per_tensor_gemm_parity(fp8bs, oracle_mod):
    rng = np.random.default_rng(11)
    a_bits, _ = synth.normal_with_outlier_columns(rng, (300, 1024), 3, 50.0)
    w_bits = synth.normal(rng, (384, 1024), 0.02)
    qa, sa, qb, sb = _gemm_per_tensor(fp8bs, a_bits, w_bits)
    c = host(fp8bs.gemm(qa, sa, qb, sb, BLOCK, out_dtype=torch.float32))
    ref = oracle_mod.gemm(host(qa), host(sa), host(qb), host(sb), BLOCK)
    assert_gemm_f32(c, ref, "per-tensor GEMM")


def _exact(a_bits, w_bits, rows):
    a = synth.bf16_bits_to_f32(a_bits[rows]).astype(np.float64)
    w = synth.bf16_bits_to_f32(w_bits).astype(np.float64)
    return a @ w.T


def _rel(c, ref):
    return float(np.linalg.norm(c - ref) / np.linalg.norm(ref))


def test_outlier_sweep_fine_grained_vs_per_tensor(fp8bs):
    """Four outlier elements of magnitude F in an N(0, 1) activation; the
    error is measured on the rows that hold no outlier."""
    rng = np.random.default_rng(5)
    M, N, K = 256, 256, 2048
    base = rng.standard_normal((M, K)).astype(np.float32)
    w_bits = synth.normal(rng, (N, K), 0.02)
    out_rows = np.array([3, 77, 150, 201])
    out_cols = rng.integers(0, K, 4)
    clean = np.setdiff1d(np.arange(M), out_rows)
    errs = {}
    for F in (1e2, 1e4, 1e5, 1e6):
        x = base.copy()
        x[out_rows, out_cols] = F
        a_bits = synth.f32_to_bf16_bits(x)
        ref = _exact(a_bits, w_bits, clean)
        fine = host(fp8bs.gemm(*_gemm_fine(fp8bs, a_bits, w_bits), BLOCK,
                               out_dtype=torch.float32))[clean]
        pt = host(fp8bs.gemm(*_gemm_per_tensor(fp8bs, a_bits, w_bits), BLOCK,
                             out_dtype=torch.float32))[clean]
        errs[F] = (_rel(fine, ref), _rel(pt, ref))
        print(f"\noutlier {F:7.0e}: clean-row rel_fro 1x128/128x128 {errs[F][0]:.3e}  "
              f"per-tensor {errs[F][1]:.3e}")
    fine_errs = [e[0] for e in errs.values()]
    assert max(fine_errs) <= 1.01 * min(fine_errs) and max(fine_errs) < 0.05
    assert errs[1e5][1] >= 2.5 * errs[1e5][0]
    assert errs[1e6][1] >= 10.0 * errs[1e6][0]


@pytest.mark.parametrize("name", ["dense", "moe"])
def test_workload_fine_grained_beats_per_tensor(fp8bs, name):
    """Full-size workloads (dense: 0.1% channels x100; MoE: Student-t),
    error on 256 sampled rows of the full GEMM."""
    inp = synth.make_inputs(name)
    a_bits, w_bits = inp["A"], inp["B"]
    rows = np.sort(np.random.default_rng(1).choice(a_bits.shape[0], 256, replace=False))
    ref = _exact(a_bits, w_bits, rows)
    fine = host(fp8bs.gemm(*_gemm_fine(fp8bs, a_bits, w_bits), BLOCK,
                           out_dtype=torch.float32))[rows]
    pt = host(fp8bs.gemm(*_gemm_per_tensor(fp8bs, a_bits, w_bits), BLOCK,
                         out_dtype=torch.float32))[rows]
    e_f, e_p = _rel(fine, ref), _rel(pt, ref)
    print(f"\n{name}: rel_fro vs exact bf16 product: 1x128/128x128 {e_f:.3e}  "
          f"per-tensor {e_p:.3e}")
    assert e_f < e_p and e_f < 0.05
