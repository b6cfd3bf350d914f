"""GPU parity of the quantizers (1x128 activation tiles, their 128x1
transposed form, 128x128 weight blocks, and the 1x128 -> 128x1 re-tiling of
the backward pass; page 1, paragraph 3): codes and scales must be
bit-identical to the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import synth
from tests._helpers import assert_codes_equal, assert_scales_equal, dev, dev_bf16

pytestmark = pytest.mark.gpu


def _special_rows(K=512):
    """Rows built to hit every rule: exact E4M3 midpoints at s = 1, signed
    zeros, all-zero groups, NaN/Inf groups, subnormal-range groups, groups
    whose scale falls below the fast-path threshold, huge values."""
    def put(row, idx, val):
        if idx < K:
            row[idx] = val
    rows = []
    e4m3 = np.array([torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item()
                     for c in range(0x7F)])
    mids = (e4m3[:-1] + e4m3[1:]) / 2
    r = np.zeros(K, np.float32)
    r[0] = 448.0
    r[1:1 + 126] = mids[:126]
    r[128] = 448.0
    r[129:129 + 126] = -mids[:126]
    rows.append(r)
    z = np.zeros(K, np.float32); z[5] = -0.0; z[130:256] = -0.0; z[7] = 1.0; rows.append(z)
    n = np.ones(K, np.float32)
    put(n, 3, np.nan); put(n, 200, np.inf); put(n, 201, -np.inf); put(n, 202, np.nan)
    n[K - 128:] = np.nan
    rows.append(n)
    t = np.full(K, 2.0 ** -133, np.float32); t[1::2] = -(2.0 ** -130); t[128:256] *= 2.0 ** 40
    t[256:384] = 2.0 ** -90; put(t, 300, 3.0 * 2.0 ** -91); t[2] = -0.0; rows.append(t)
    h = np.linspace(-3.0e38, 3.0e38, K).astype(np.float32); h[9] = -0.0; rows.append(h)
    f = np.linspace(-1, 1, K).astype(np.float32) * np.float32(448 * 2.0 ** -92); f[4] = -0.0
    rows.append(f)
    return synth.f32_to_bf16_bits(np.stack(rows))


@pytest.mark.parametrize("M,K,seed", [(1, 128, 0), (127, 256, 1), (129, 512, 2), (333, 384, 3),
                                      (64, 1024, 4), (1000, 640, 5)])
def test_act_1x128_ragged(fp8bs, oracle_mod, M, K, seed):
    rng = np.random.default_rng(seed)
    x, _ = synth.normal_with_outlier_columns(rng, (M, K), 2, 100.0)
    q, s = fp8bs.quant_act_1x128(dev_bf16(x))
    rq, rs = oracle_mod.quant_act_1x128(x)
    assert_codes_equal(q, rq, "codes")
    assert_scales_equal(s, rs, "scales")


def test_act_1x128_special_values(fp8bs, oracle_mod):
    x = _special_rows()
    q, s = fp8bs.quant_act_1x128(dev_bf16(x))
    rq, rs = oracle_mod.quant_act_1x128(x)
    assert_codes_equal(q, rq, "codes")
    assert_scales_equal(s, rs, "scales")


def test_act_1x128_heavy_tail_and_loguniform(fp8bs, oracle_mod):
    rng = np.random.default_rng(9)
    for x in (synth.student_t4(rng, (512, 1024)), synth.loguniform_rows(rng, (512, 1024))):
        q, s = fp8bs.quant_act_1x128(dev_bf16(x))
        rq, rs = oracle_mod.quant_act_1x128(x)
        assert_codes_equal(q, rq, "codes")
        assert_scales_equal(s, rs, "scales")


def test_zero_size_is_noop(fp8bs):
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    q, s = fp8bs.quant_act_1x128(x)
    assert q.shape == (0, 256) and s.shape == (2, 0)


@pytest.mark.parametrize("M,K,seed", [(128, 128, 0), (256, 384, 1), (512, 1024, 2)])
def test_act_128x1(fp8bs, oracle_mod, M, K, seed):
    rng = np.random.default_rng(seed)
    x, _ = synth.normal_with_outlier_columns(rng, (M, K), 3, 50.0)
    qT, sT = fp8bs.quant_act_1x128(dev_bf16(x), transpose_out=True)
    rq, rs = oracle_mod.quant_act_128x1(x)
    assert_codes_equal(qT, rq, "codes")
    assert_scales_equal(sT, rs, "scales")


def test_act_128x1_special_values(fp8bs, oracle_mod):
    x = np.ascontiguousarray(np.concatenate([_special_rows(256).T] * 1, axis=1))  # [256, 6]
    x = np.ascontiguousarray(np.tile(x, (1, 22))[:, :128])  # [256, 128]
    qT, sT = fp8bs.quant_act_1x128(dev_bf16(x), transpose_out=True)
    rq, rs = oracle_mod.quant_act_128x1(x)
    assert_codes_equal(qT, rq, "codes")
    assert_scales_equal(sT, rs, "scales")


@pytest.mark.parametrize("M,K,seed", [(128, 128, 0), (256, 384, 1), (512, 1024, 2), (384, 2048, 3)])
def test_act_dual(fp8bs, oracle_mod, M, K, seed):
    """One read, both tilings: bit-identical to the 1x128 and the 128x1 quantizer."""
    rng = np.random.default_rng(40 + seed)
    x, _ = synth.normal_with_outlier_columns(rng, (M, K), 3, 50.0)
    q, s, qT, sT = fp8bs.quant_act_dual(dev_bf16(x))
    rq, rs = oracle_mod.quant_act_1x128(x)
    rqT, rsT = oracle_mod.quant_act_128x1(x)
    assert_codes_equal(q, rq, "codes 1x128")
    assert_scales_equal(s, rs, "scales 1x128")
    assert_codes_equal(qT, rqT, "codes 128x1")
    assert_scales_equal(sT, rsT, "scales 128x1")


def test_act_dual_special_values(fp8bs, oracle_mod):
    rows = _special_rows(256)  # 6 rows x 256
    x = np.zeros((256, 256), np.uint16)
    for i in range(256):
        x[i] = rows[(i * 5) % 6]
    x[:, 7] = rows[2][:256]  # a column with NaN/Inf
    q, s, qT, sT = fp8bs.quant_act_dual(dev_bf16(x))
    rq, rs = oracle_mod.quant_act_1x128(x)
    rqT, rsT = oracle_mod.quant_act_128x1(x)
    assert_codes_equal(q, rq, "codes 1x128")
    assert_scales_equal(s, rs, "scales 1x128")
    assert_codes_equal(qT, rqT, "codes 128x1")
    assert_scales_equal(sT, rsT, "scales 128x1")


@pytest.mark.parametrize("N,K,seed", [(128, 128, 0), (256, 640, 1), (1024, 384, 2)])
def test_weight_128x128(fp8bs, oracle_mod, N, K, seed):
    rng = np.random.default_rng(seed)
    w = synth.normal(rng, (N, K), 0.02)
    q, s, qT, sT = fp8bs.quant_weight_128x128(dev_bf16(w), transposed=True)
    rq, rs, rqT, rsT = oracle_mod.quant_weight_128x128(w, transposed=True)
    assert_codes_equal(q, rq, "codes")
    assert_scales_equal(s, rs, "scales")
    assert_codes_equal(qT, rqT, "codesT")
    assert_scales_equal(sT, rsT, "scalesT")
    q2, s2 = fp8bs.quant_weight_128x128(dev_bf16(w))
    assert_codes_equal(q2, rq, "codes (no transposed copy)")


def test_weight_special_values(fp8bs, oracle_mod):
    rows = _special_rows(256)  # 6 rows
    w = np.zeros((256, 256), np.uint16)
    for i in range(256):
        w[i] = rows[i % 6]
    w[128:, 128:] = synth.f32_to_bf16_bits(np.zeros((128, 128), np.float32))  # all-zero block
    q, s, qT, sT = fp8bs.quant_weight_128x128(dev_bf16(w), transposed=True)
    rq, rs, rqT, rsT = oracle_mod.quant_weight_128x128(w, transposed=True)
    assert_codes_equal(q, rq, "codes")
    assert_scales_equal(s, rs, "scales")
    assert_codes_equal(qT, rqT, "codesT")


@pytest.mark.parametrize("M,K,seed", [(128, 128, 0), (256, 512, 1), (640, 256, 2)])
def test_requant(fp8bs, oracle_mod, M, K, seed):
    rng = np.random.default_rng(seed)
    x, _ = synth.normal_with_outlier_columns(rng, (M, K), 2, 100.0)
    rq, rs = oracle_mod.quant_act_1x128(x)
    qT, sT = fp8bs.requant_1x128_to_128x1(dev(rq), dev(rs))
    rqT, rsT = oracle_mod.requant_1x128_to_128x1(rq, rs)
    assert_codes_equal(qT, rqT, "codes")
    assert_scales_equal(sT, rsT, "scales")


def test_requant_special_values(fp8bs, oracle_mod):
    rows = _special_rows(256)
    x = np.zeros((256, 256), np.uint16)
    for i in range(256):
        x[i] = rows[(i * 7) % 6]
    rq, rs = oracle_mod.quant_act_1x128(x)
    qT, sT = fp8bs.requant_1x128_to_128x1(dev(rq), dev(rs))
    rqT, rsT = oracle_mod.requant_1x128_to_128x1(rq, rs)
    assert_codes_equal(qT, rqT, "codes")
    assert_scales_equal(sT, rsT, "scales")


# ---- full-size workloads (the bench's launch configuration) -------------

def test_dense_activation_and_weight_full(fp8bs, oracle_mod):
    inp = synth.make_inputs("dense")
    q, s = fp8bs.quant_act_1x128(dev_bf16(inp["A"]))
    rq, rs = oracle_mod.quant_act_1x128(inp["A"])
    assert_codes_equal(q, rq, "A codes")
    assert_scales_equal(s, rs, "A scales")
    q, s = fp8bs.quant_weight_128x128(dev_bf16(inp["B"]))
    rq, rs = oracle_mod.quant_weight_128x128(inp["B"])
    assert_codes_equal(q, rq, "W codes")
    assert_scales_equal(s, rs, "W scales")


def test_moe_activation_full(fp8bs, oracle_mod):
    inp = synth.make_inputs("moe")
    q, s = fp8bs.quant_act_1x128(dev_bf16(inp["A"]))
    rq, rs = oracle_mod.quant_act_1x128(inp["A"])
    assert_codes_equal(q, rq, "A codes")
    assert_scales_equal(s, rs, "A scales")


def test_backward_quantizers_full(fp8bs, oracle_mod):
    inp = synth.make_inputs("bwd")
    # grad_out 128x1 tiles (weight-gradient A operand)
    qT, sT = fp8bs.quant_act_1x128(dev_bf16(inp["dY"]), transpose_out=True)
    rqT, rsT = oracle_mod.quant_act_128x1(inp["dY"])
    assert_codes_equal(qT, rqT, "dY^T codes")
    assert_scales_equal(sT, rsT, "dY^T scales")
    # both tilings of grad_out from one read
    q2, s2, qT2, sT2 = fp8bs.quant_act_dual(dev_bf16(inp["dY"]))
    rq2, rs2 = oracle_mod.quant_act_1x128(inp["dY"])
    assert_codes_equal(q2, rq2, "dY codes (dual)")
    assert_scales_equal(s2, rs2, "dY scales (dual)")
    assert_codes_equal(qT2, rqT, "dY^T codes (dual)")
    assert_scales_equal(sT2, rsT, "dY^T scales (dual)")
    # cached activation X: 1x128 then re-tiled to 128x1
    qx, sx = fp8bs.quant_act_1x128(dev_bf16(inp["X"]))
    rqx, rsx = oracle_mod.quant_act_1x128(inp["X"])
    assert_codes_equal(qx, rqx, "X codes")
    qxT, sxT = fp8bs.requant_1x128_to_128x1(qx, sx)
    rqxT, rsxT = oracle_mod.requant_1x128_to_128x1(rqx, rsx)
    assert_codes_equal(qxT, rqxT, "X^T codes")
    assert_scales_equal(sxT, rsxT, "X^T scales")
    # weight with transposed copy (input-gradient B operand)
    q, s, qT2, sT2 = fp8bs.quant_weight_128x128(dev_bf16(inp["W"]), transposed=True)
    rq, rs, rqT2, rsT2 = oracle_mod.quant_weight_128x128(inp["W"], transposed=True)
    assert_codes_equal(q, rq, "W codes (transposed call)")
    assert_scales_equal(s, rs, "W scales (transposed call)")
    assert_codes_equal(qT2, rqT2, "W^T codes")
    assert_scales_equal(sT2, rsT2, "W^T scales")


def test_stress_activation_full(fp8bs, oracle_mod):
    """Q1 on the large-K stress operand A (8192 x 16384, rows U(-1, 1) x
    10^U(-2, 2)), the bench step's first quantizer launch: every code and
    scale."""
    inp = synth.make_inputs("stress")
    q, s = fp8bs.quant_act_1x128(dev_bf16(inp["A"]))
    rq, rs = oracle_mod.quant_act_1x128(inp["A"])
    assert_codes_equal(q, rq, "stress A codes")
    assert_scales_equal(s, rs, "stress A scales")


def test_hand_worked_tiles_on_gpu(fp8bs):
    """The hand-derived codes of tests/golden/e4m3_hand_tiles.txt, straight
    from the GPU quantizer (no oracle in between)."""
    from tests.test_oracle_quant import _golden_rows
    rows = _golden_rows()
    tiles = np.zeros((len(rows), 128), np.float32)
    for i, (amax, x, _) in enumerate(rows):
        tiles[i, 0] = amax
        tiles[i, 1] = x
    q, s = fp8bs.quant_act_1x128(dev_bf16(synth.f32_to_bf16_bits(tiles)))
    q = q.cpu().numpy()
    for i, (amax, x, code) in enumerate(rows):
        assert q[i, 1] == code, (amax, x, hex(q[i, 1]), hex(code))


@pytest.mark.parametrize("M,K,N,Kw", [(1, 128, 128, 128), (300, 1024, 384, 1024),
                                      (129, 256, 1024, 640), (4096, 7168, 7168, 7168)])
def test_act_and_weight_one_launch(fp8bs, oracle_mod, M, K, N, Kw):
    """Q1 and Q2 in one launch: every code and scale of both outputs equals
    the oracle's (the last case is the dense projection workload)."""
    if (M, K) == (4096, 7168):
        inp = synth.make_inputs("dense")
        a_bits, w_bits = inp["A"], inp["B"]
    else:
        rng = np.random.default_rng(M + N + K + Kw)
        a_bits, _ = synth.normal_with_outlier_columns(rng, (M, K), 3, 100.0)
        w_bits = synth.normal(rng, (N, Kw), 0.02)
        w_bits[5 % N, 7] = synth.f32_to_bf16_bits(np.array([np.nan], np.float32))[0]
    q, s, qw, sw = fp8bs.quant_act_and_weight(dev_bf16(a_bits), dev_bf16(w_bits))
    q_ref, s_ref = oracle_mod.quant_act_1x128(a_bits)
    qw_ref, sw_ref = oracle_mod.quant_weight_128x128(w_bits)
    assert_codes_equal(q, q_ref, "activation codes")
    assert_scales_equal(s, s_ref, "activation scales")
    assert_codes_equal(qw, qw_ref, "weight codes")
    assert_scales_equal(sw, sw_ref, "weight scales")
