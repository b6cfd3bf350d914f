"""GPU parity of the block-scaled FP8 GEMM (page 1, paragraphs 2-4; page 4,
paragraph 4) against the oracle's double-precision sum of dequantized
products, through the C ABI.  Small cases are compared element by element;
the full-size workloads (the bench's launch configuration) on seeded
samples of output positions the oracle computes one by one."""
import numpy as np
import pytest
import torch

import synth
from tests._helpers import (assert_gemm_bf16, assert_gemm_f32, dev, dev_bf16, gemm_errors, host)

pytestmark = pytest.mark.gpu

BLOCK, TILE = 0, 1
# every output-tile shape of the kernel (the automatic choice differs by shape)
TILES = list(range(11))


def _quantized_pair(oracle_mod, M, N, K, seed, bkind):
    rng = np.random.default_rng(seed)
    a_bits, _ = synth.normal_with_outlier_columns(rng, (M, K), 3, 50.0)
    a, sa = oracle_mod.quant_act_1x128(a_bits)
    if bkind == BLOCK:
        # block scales cover ceil(N / 128) row blocks: quantize the weight
        # padded with zero rows to whole blocks, keep its first N code rows
        nb = (N + 127) // 128
        w = np.zeros((nb * 128, K), np.uint16)
        w[:N] = synth.normal(rng, (N, K), 0.02)
        b, sb = oracle_mod.quant_weight_128x128(w)
        b = np.ascontiguousarray(b[:N])
    else:
        b, sb = oracle_mod.quant_act_1x128(synth.normal(rng, (N, K), 1e-3))
    return a, sa, b, sb


@pytest.mark.parametrize("bkind", [BLOCK, TILE])
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_tiny(fp8bs, oracle_mod, bkind, out):
    inp = synth.make_inputs("tiny")
    a, sa = oracle_mod.quant_act_1x128(inp["A"])
    if bkind == BLOCK:
        b, sb = oracle_mod.quant_weight_128x128(inp["B"])
    else:
        b, sb = oracle_mod.quant_act_1x128(inp["B"])
    ref = oracle_mod.gemm(a, sa, b, sb, bkind)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    c = host(fp8bs.gemm(dev(a), dev(sa), dev(b), dev(sb), bkind, out_dtype=dt))
    if out == "f32":
        assert_gemm_f32(c, ref, "tiny")
    else:
        assert_gemm_bf16(c, ref, "tiny")


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("M,N,K,bkind", [
    (1, 128, 128, BLOCK), (100, 256, 256, BLOCK), (129, 384, 512, BLOCK), (333, 128, 1024, BLOCK),
    (256, 640, 384, BLOCK), (200, 256, 256, TILE), (385, 512, 640, TILE), (128, 1024, 128, BLOCK),
    (64, 144, 256, TILE), (130, 208, 384, TILE), (640, 912, 256, BLOCK), (520, 464, 384, TILE)])
def test_ragged_shapes(fp8bs, oracle_mod, M, N, K, bkind, tile):
    a, sa, b, sb = _quantized_pair(oracle_mod, M, N, K, M + N + K, bkind)
    ref = oracle_mod.gemm(a, sa, b, sb, bkind)
    c = host(fp8bs.gemm(dev(a), dev(sa), dev(b), dev(sb), bkind, out_dtype=torch.float32,
                        tile=tile))
    assert_gemm_f32(c, ref, f"{M}x{N}x{K} tile {tile}")
    c16 = host(fp8bs.gemm(dev(a), dev(sa), dev(b), dev(sb), bkind, out_dtype=torch.bfloat16,
                          tile=tile))
    assert_gemm_bf16(c16, ref, f"{M}x{N}x{K} bf16 tile {tile}")


@pytest.mark.parametrize("tile", TILES)
def test_integer_case_bit_exact(fp8bs, oracle_mod, tile):
    """Unit scales and small-integer codes: every partial and the FP32
    accumulator are exact, so the output must equal the integer matmul."""
    rng = np.random.default_rng(21)
    vals = {}
    for c in range(256):
        v = torch.tensor([c], dtype=torch.uint8).view(torch.float8_e4m3fn).float().item()
        if v == v and v == int(v) and abs(v) <= 16:
            vals[v] = c
    keys = np.array(sorted(vals))
    M, N, K = 256, 256, 1024
    ai = rng.choice(keys, (M, K)); bi = rng.choice(keys, (N, K))
    a = np.vectorize(vals.get)(ai).astype(np.uint8)
    b = np.vectorize(vals.get)(bi).astype(np.uint8)
    sa = np.ones((K // 128, M), np.float32)
    sb = np.ones((N // 128, K // 128), np.float32)
    c = host(fp8bs.gemm(dev(a), dev(sa), dev(b), dev(sb), BLOCK, out_dtype=torch.float32,
                        tile=tile))
    assert np.array_equal(c.astype(np.int64), ai.astype(np.int64) @ bi.astype(np.int64).T)


@pytest.mark.parametrize("tile", TILES)
def test_scale_index_one_hot(fp8bs, oracle_mod, tile):
    """Distinct power-of-two scales per (K-group, row) and per B block: a
    misplaced scale index changes the exact result."""
    M, N, K = 256, 384, 512
    KB = K // 128
    rng = np.random.default_rng(22)
    a = np.zeros((M, K), np.uint8); b = np.zeros((N, K), np.uint8)
    for m in range(M):
        a[m, rng.integers(0, K, 4)] = 0x38
    for n in range(N):
        b[n, rng.integers(0, K, 4)] = 0xC0
    # exponents in [-5, 5]: every output is a sum of at most 8 terms whose
    # magnitudes span < 2^24, so the FP32 result is exact
    sa = (2.0 ** rng.integers(-5, 6, (KB, M))).astype(np.float32)
    for bkind in (BLOCK, TILE):
        sb = (2.0 ** rng.integers(-5, 6, (N // 128, KB) if bkind == BLOCK else (KB, N))).astype(np.float32)
        ref = oracle_mod.gemm(a, sa, b, sb, bkind)
        c = host(fp8bs.gemm(dev(a), dev(sa), dev(b), dev(sb), bkind, out_dtype=torch.float32,
                            tile=tile))
        assert np.array_equal(c.astype(np.float64), ref), (bkind, tile)


@pytest.mark.parametrize("tile", TILES)
def test_unpromoted_matches_on_rowwise_codes(fp8bs, oracle_mod, tile):
    """The un-promoted variant needs scales constant along K (row-wise
    codes); on such inputs it computes the same sum, with whatever precision
    the tensor core accumulates in.  Its error is measured, not assumed."""
    rng = np.random.default_rng(23)
    M, N, K = 256, 256, 4096
    a, sa = oracle_mod.quant_rowwise(synth.loguniform_rows(rng, (M, K)))
    b, sb_rows = oracle_mod.quant_rowwise(synth.normal(rng, (N, K), 0.02))
    ref = oracle_mod.gemm(a, sa, b, sb_rows, TILE)
    c_un = host(fp8bs.gemm(dev(a), dev(sa), dev(b), dev(sb_rows), TILE, out_dtype=torch.float32,
                           promote=False, tile=tile))
    c_pr = host(fp8bs.gemm(dev(a), dev(sa), dev(b), dev(sb_rows), TILE, out_dtype=torch.float32,
                           tile=tile))
    e_un = gemm_errors(c_un, ref)
    e_pr = gemm_errors(c_pr, ref)
    print(f"K={K}: promoted rel_fro={e_pr[0]:.3e} max_rel={e_pr[1]:.3e}; "
          f"un-promoted rel_fro={e_un[0]:.3e} max_rel={e_un[1]:.3e}")
    assert_gemm_f32(c_pr, ref, "promoted")
    assert e_un[0] < 5e-2  # same sum, whatever the accumulator precision


def test_chain_gpu_quant_then_gemm(fp8bs, oracle_mod):
    """End-to-end forward path on the GPU (quantize both operands, GEMM)."""
    rng = np.random.default_rng(24)
    x, _ = synth.normal_with_outlier_columns(rng, (300, 1024), 3, 100.0)
    w = synth.normal(rng, (512, 1024), 0.02)
    qa, sa = fp8bs.quant_act_1x128(dev_bf16(x))
    qb, sb = fp8bs.quant_weight_128x128(dev_bf16(w))
    c = host(fp8bs.gemm(qa, sa, qb, sb, BLOCK, out_dtype=torch.float32))
    ra, rsa = oracle_mod.quant_act_1x128(x)
    rb, rsb = oracle_mod.quant_weight_128x128(w)
    assert_gemm_f32(c, oracle_mod.gemm(ra, rsa, rb, rsb, BLOCK), "chain")


@pytest.mark.parametrize("tile", TILES)
@pytest.mark.parametrize("M,N", [(128, 128), (256, 512)])
def test_bounded_wait_reports_timeout(fp8bs, oracle_mod, M, N, tile):
    """A pipeline stage whose copy is never issued: the kernel's bounded
    wait expires, the kernel returns, the status reads TIMEOUT, and the
    context keeps working."""
    a, sa, b, sb = _quantized_pair(oracle_mod, M, N, 512, 5, BLOCK)
    assert fp8bs.get_device_error() == fp8bs.OK
    fp8bs.debug_gemm_stall(dev(a), dev(sa), dev(b), dev(sb), skip_iter=2, tile=tile)
    assert fp8bs.get_device_error() == fp8bs.ERR_TIMEOUT
    assert fp8bs.get_device_error() == fp8bs.OK  # cleared
    ref = oracle_mod.gemm(a, sa, b, sb, BLOCK)
    c = host(fp8bs.gemm(dev(a), dev(sa), dev(b), dev(sb), BLOCK, out_dtype=torch.float32,
                        tile=tile))
    assert_gemm_f32(c, ref, "after timeout")


# ---- full-size workloads, sampled outputs --------------------------------

def _sample_positions(M, N, count, seed):
    rng = np.random.default_rng(seed)
    ms = np.concatenate([rng.integers(0, M, count), [0, M - 1, M - 1, 0]])
    ns = np.concatenate([rng.integers(0, N, count), [0, N - 1, 0, N - 1]])
    return ms, ns


def _check_sampled(fp8bs, oracle_mod, a, sa, b, sb, bkind, what, samples=4000, bf16=True):
    M, N = a.shape[0], b.shape[0]
    ms, ns = _sample_positions(M, N, samples, M + N)
    ref = oracle_mod.gemm_sampled(a, sa, b, sb, bkind, ms, ns)
    da, dsa, db, dsb = dev(a), dev(sa), dev(b), dev(sb)
    c32 = fp8bs.gemm(da, dsa, db, dsb, bkind, out_dtype=torch.float32)
    v32 = host(c32[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()])
    errs = assert_gemm_f32(v32, ref, what + " f32")
    if bf16:
        c16 = fp8bs.gemm(da, dsa, db, dsb, bkind, out_dtype=torch.bfloat16)
        v16 = host(c16[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()])
        assert_gemm_bf16(v16, ref, what + " bf16")
    return errs


def test_dense_full_sampled(fp8bs, oracle_mod):
    inp = synth.make_inputs("dense")
    a, sa = oracle_mod.quant_act_1x128(inp["A"])
    b, sb = oracle_mod.quant_weight_128x128(inp["B"])
    _check_sampled(fp8bs, oracle_mod, a, sa, b, sb, BLOCK, "dense")


def test_moe_full_sampled(fp8bs, oracle_mod):
    inp = synth.make_inputs("moe")
    a, sa = oracle_mod.quant_act_1x128(inp["A"])
    b, sb = oracle_mod.quant_weight_128x128(inp["B"])
    _check_sampled(fp8bs, oracle_mod, a, sa, b, sb, BLOCK, "moe")


def test_backward_full_sampled(fp8bs, oracle_mod):
    inp = synth.make_inputs("bwd")
    # input gradient: dX[4096, 2048] = dY[4096, 7168] * W[7168, 2048]
    dy, sdy = oracle_mod.quant_act_1x128(inp["dY"])
    _, _, wT, swT = oracle_mod.quant_weight_128x128(inp["W"], transposed=True)
    _check_sampled(fp8bs, oracle_mod, dy, sdy, wT, swT, BLOCK, "dgrad")
    # weight gradient: dW[7168, 2048] = dY^T[7168, 4096] * X[4096, 2048]
    dyT, sdyT = oracle_mod.quant_act_128x1(inp["dY"])
    qx, sx = oracle_mod.quant_act_1x128(inp["X"])
    xT, sxT = oracle_mod.requant_1x128_to_128x1(qx, sx)
    _check_sampled(fp8bs, oracle_mod, dyT, sdyT, xT, sxT, TILE, "wgrad", bf16=False)


def test_stress_full_sampled(fp8bs, oracle_mod):
    inp = synth.make_inputs("stress")
    a, sa = oracle_mod.quant_act_1x128(inp["A"])
    b, sb = oracle_mod.quant_act_1x128(inp["B"])
    _check_sampled(fp8bs, oracle_mod, a, sa, b, sb, TILE, "stress", samples=1500, bf16=False)


def test_bench_stress_step_full_sampled(fp8bs, oracle_mod):
    """The benchmark's headline step as it launches it: A quantized in 1x128
    tiles and B in 128x128 blocks on the device (two launches), then the
    promoted GEMM with block B scales, the automatic tile and FP32 output at
    8192 x 8192 x 16384; the device codes and scales equal the oracle's, and
    sampled outputs match the oracle's double sums."""
    inp = synth.make_inputs("stress")
    qa, sa = fp8bs.quant_act_1x128(dev_bf16(inp["A"]))
    qb, sb = fp8bs.quant_weight_128x128(dev_bf16(inp["B"]))
    c = fp8bs.gemm(qa, sa, qb, sb, BLOCK, out_dtype=torch.float32)
    a_ref, sa_ref = oracle_mod.quant_act_1x128(inp["A"])
    b_ref, sb_ref = oracle_mod.quant_weight_128x128(inp["B"])
    assert np.array_equal(host(qa), a_ref) and np.array_equal(host(sa).view(np.uint32), sa_ref.view(np.uint32))
    assert np.array_equal(host(qb), b_ref) and np.array_equal(host(sb).view(np.uint32), sb_ref.view(np.uint32))
    M, N = a_ref.shape[0], b_ref.shape[0]
    ms, ns = _sample_positions(M, N, 1500, 11)
    ref = oracle_mod.gemm_sampled(a_ref, sa_ref, b_ref, sb_ref, BLOCK, ms, ns)
    v = host(c[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()])
    assert_gemm_f32(v, ref, "bench stress step")


def test_bench_step_full_sampled(fp8bs, oracle_mod):
    """The dense projection step exactly as the benchmark launches it: both
    operands quantized in one launch, then the GEMM with the automatic tile
    and BF16 output; sampled outputs against the oracle's chain."""
    inp = synth.make_inputs("dense")
    qa, sa, qb, sb = fp8bs.quant_act_and_weight(dev_bf16(inp["A"]), dev_bf16(inp["B"]))
    c = fp8bs.gemm(qa, sa, qb, sb, BLOCK, out_dtype=torch.bfloat16)
    a_ref, sa_ref = oracle_mod.quant_act_1x128(inp["A"])
    b_ref, sb_ref = oracle_mod.quant_weight_128x128(inp["B"])
    M, N = a_ref.shape[0], b_ref.shape[0]
    ms, ns = _sample_positions(M, N, 4000, 7)
    ref = oracle_mod.gemm_sampled(a_ref, sa_ref, b_ref, sb_ref, BLOCK, ms, ns)
    v = host(c[torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda()])
    assert_gemm_bf16(v, ref, "bench step")
