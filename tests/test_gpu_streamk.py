"""GPU parity of the stream-K GEMM (fp8bs_gemm_streamk): the promoted
block-scaled GEMM of page 1, paragraphs 2-3, with the K-groups of an uneven
last wave of tiles spread over every SM and the split tiles summed through
a caller workspace.  Compared with the oracle's double-precision sums, with
fp8bs_gemm on the same inputs, and with itself over repeated calls (the
shares are summed in K order, so the result does not depend on which SM
finishes a tile last)."""
import numpy as np
import pytest
import torch

import synth
from tests._helpers import assert_gemm_bf16, assert_gemm_f32, dev, host

pytestmark = pytest.mark.gpu

BLOCK, TILE = 0, 1
ERR_INVALID_ARG, ERR_MISALIGNED = 1, 3


def _pair(oracle_mod, M, N, K, seed, bkind):
    rng = np.random.default_rng(seed)
    a, sa = oracle_mod.quant_act_1x128(synth.normal_with_outlier_columns(rng, (M, K), 3, 50.0)[0])
    if bkind == BLOCK:
        nb = (N + 127) // 128
        w = np.zeros((nb * 128, K), np.uint16)
        w[:N] = synth.normal(rng, (N, K), 0.02)
        b, sb = oracle_mod.quant_weight_128x128(w)
        b = np.ascontiguousarray(b[:N])
    else:
        b, sb = oracle_mod.quant_act_1x128(synth.normal(rng, (N, K), 1e-3))
    return a, sa, b, sb


@pytest.mark.parametrize("M,N,K,bkind", [
    (256, 256, 5120, BLOCK),    # one tile: its 40 K-groups split 40 ways
    (1000, 512, 2048, TILE),    # ragged M, a few tiles split over every SM
    (512, 768, 7168, BLOCK),    # 6 tiles of 56 K-groups over every SM
    (300, 144, 1024, TILE)])    # ragged M and N
@pytest.mark.parametrize("out", ["f32", "bf16"])
def test_streamk_against_oracle(fp8bs, oracle_mod, M, N, K, bkind, out):
    a, sa, b, sb = _pair(oracle_mod, M, N, K, M + N + K, bkind)
    dt = torch.float32 if out == "f32" else torch.bfloat16
    need = fp8bs.gemm_streamk_workspace(M, N, K, bkind, dt)
    assert need > 0, "these shapes leave most SMs idle: stream-K should be planned"
    ref = oracle_mod.gemm(a, sa, b, sb, bkind)
    c = host(fp8bs.gemm_streamk(dev(a), dev(sa), dev(b), dev(sb), bkind, out_dtype=dt))
    if out == "f32":
        assert_gemm_f32(c, ref, f"stream-K {M}x{N}x{K}")
    else:
        assert_gemm_bf16(c, ref, f"stream-K {M}x{N}x{K}")


def test_streamk_repeatable_and_close_to_gemm(fp8bs, oracle_mod):
    """Three calls on one workspace give identical bits (counters reset by
    the call; shares summed in K order), and the result differs from
    fp8bs_gemm only by FP32 rounding of the split sums."""
    M, N, K = 512, 768, 7168
    a, sa, b, sb = _pair(oracle_mod, M, N, K, 11, BLOCK)
    da, dsa, db, dsb = dev(a), dev(sa), dev(b), dev(sb)
    need = fp8bs.gemm_streamk_workspace(M, N, K, BLOCK, torch.float32)
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    ws.fill_(0xA5)  # no initialisation is needed
    outs = [host(fp8bs.gemm_streamk(da, dsa, db, dsb, BLOCK, out_dtype=torch.float32,
                                    workspace=ws)) for _ in range(3)]
    assert np.array_equal(outs[0].view(np.uint32), outs[1].view(np.uint32))
    assert np.array_equal(outs[0].view(np.uint32), outs[2].view(np.uint32))
    base = host(fp8bs.gemm(da, dsa, db, dsb, BLOCK, out_dtype=torch.float32))
    scale = np.abs(base).max()
    assert np.abs(outs[0] - base).max() <= 1e-5 * scale


@pytest.mark.parametrize("bkind", [BLOCK, TILE])
def test_streamk_sampled(fp8bs, oracle_mod, bkind):
    """16 pair tiles of 64 K-groups (1024 x 1024 x 8192): every tile split
    over several SMs, on sampled outputs of the oracle."""
    M, N, K = 1024, 1024, 8192
    a, sa, b, sb = _pair(oracle_mod, M, N, K, 21 + bkind, bkind)
    assert fp8bs.gemm_streamk_workspace(M, N, K, bkind, torch.float32) > 0
    rng = np.random.default_rng(5)
    ms = np.concatenate([rng.integers(0, M, 4000), [0, M - 1]])
    ns = np.concatenate([rng.integers(0, N, 4000), [N - 1, 0]])
    ref = oracle_mod.gemm_sampled(a, sa, b, sb, bkind, ms, ns)
    idx = (torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda())
    c = fp8bs.gemm_streamk(dev(a), dev(sa), dev(b), dev(sb), bkind, out_dtype=torch.float32)
    assert_gemm_f32(host(c[idx]), ref, "stream-K 1024x1024x8192")


def test_streamk_dgrad_runs_whole_tiles(fp8bs, oracle_mod):
    """The backward workload's input gradient (4096 x 2048 x 7168: 1.73
    waves of whole tiles) plans no stream-K -- its hand-off costs more than
    the partial wave -- and runs as fp8bs_gemm."""
    inp = synth.make_inputs("bwd")
    dy, sdy = oracle_mod.quant_act_1x128(inp["dY"])
    _, _, wT, swT = oracle_mod.quant_weight_128x128(inp["W"], transposed=True)
    M, N, K = dy.shape[0], wT.shape[0], dy.shape[1]
    assert fp8bs.gemm_streamk_workspace(M, N, K, BLOCK, torch.bfloat16) == 0
    da, dsa, db, dsb = dev(dy), dev(sdy), dev(wT), dev(swT)
    c1 = host(fp8bs.gemm_streamk(da, dsa, db, dsb, BLOCK, out_dtype=torch.bfloat16))
    c2 = host(fp8bs.gemm(da, dsa, db, dsb, BLOCK, out_dtype=torch.bfloat16))
    assert np.array_equal(c1.view(np.uint16), c2.view(np.uint16))


def _sampled_positions(M, N, count, seed):
    rng = np.random.default_rng(seed)
    ms = np.concatenate([rng.integers(0, M, count), [0, M - 1, M - 1, 0]])
    ns = np.concatenate([rng.integers(0, N, count), [0, N - 1, 0, N - 1]])
    return ms, ns


def test_streamk_uneven_last_wave_full_sampled(fp8bs, oracle_mod):
    """Large problems whose last wave of whole tiles is nearly empty get a
    stream-K plan over the last two waves: the weight gradient (7168 x 2048
    x 4096, per-column B scales: 3.03 waves of 128 x 256 tiles) and the
    dense projection (4096 x 7168 x 7168, block B scales: 6.05 waves);
    sampled outputs against the oracle's double sums."""
    inp = synth.make_inputs("bwd")
    dyT, sdyT = oracle_mod.quant_act_128x1(inp["dY"])
    qx, sx = oracle_mod.quant_act_1x128(inp["X"])
    xT, sxT = oracle_mod.requant_1x128_to_128x1(qx, sx)
    dense = synth.make_inputs("dense")
    a, sa = oracle_mod.quant_act_1x128(dense["A"])
    w, sw = oracle_mod.quant_weight_128x128(dense["B"])
    for (qa_, sa_, qb_, sb_, bkind, what) in ((dyT, sdyT, xT, sxT, TILE, "wgrad"),
                                              (a, sa, w, sw, BLOCK, "dense")):
        M, K = qa_.shape
        N = qb_.shape[0]
        need = fp8bs.gemm_streamk_workspace(M, N, K, bkind, torch.float32)
        assert need > 0, f"{what}: an uneven last wave should plan stream-K"
        ms, ns = _sampled_positions(M, N, 3000, M + N)
        ref = oracle_mod.gemm_sampled(qa_, sa_, qb_, sb_, bkind, ms, ns)
        c = fp8bs.gemm_streamk(dev(qa_), dev(sa_), dev(qb_), dev(sb_), bkind,
                               out_dtype=torch.float32)
        idx = (torch.from_numpy(ms).cuda(), torch.from_numpy(ns).cuda())
        assert_gemm_f32(host(c[idx]), ref, f"stream-K {what}")


def test_streamk_whole_waves_need_no_workspace(fp8bs, oracle_mod):
    """A problem whose tiles fill whole waves plans no stream-K: zero
    workspace, and the call is fp8bs_gemm bit for bit."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    M, N, K = 256 * (sms // 2), 256, 512  # one pair tile per pair
    a, sa, b, sb = _pair(oracle_mod, M, N, K, 3, BLOCK)
    assert fp8bs.gemm_streamk_workspace(M, N, K, BLOCK, torch.float32) == 0
    da, dsa, db, dsb = dev(a), dev(sa), dev(b), dev(sb)
    c1 = host(fp8bs.gemm_streamk(da, dsa, db, dsb, BLOCK, out_dtype=torch.float32))
    c2 = host(fp8bs.gemm(da, dsa, db, dsb, BLOCK, out_dtype=torch.float32))
    assert np.array_equal(c1.view(np.uint32), c2.view(np.uint32))


def test_streamk_workspace_errors(fp8bs, oracle_mod):
    M, N, K = 256, 256, 5120
    a, sa, b, sb = _pair(oracle_mod, M, N, K, 4, BLOCK)
    da, dsa, db, dsb = dev(a), dev(sa), dev(b), dev(sb)
    need = fp8bs.gemm_streamk_workspace(M, N, K, BLOCK, torch.float32)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(fp8bs.Fp8bsError) as e:
        fp8bs.gemm_streamk(da, dsa, db, dsb, BLOCK, out_dtype=torch.float32, workspace=small)
    assert e.value.status == ERR_INVALID_ARG
    big = torch.empty(need + 512, dtype=torch.uint8, device="cuda")
    with pytest.raises(fp8bs.Fp8bsError) as e:
        fp8bs.gemm_streamk(da, dsa, db, dsb, BLOCK, out_dtype=torch.float32,
                           workspace=big[16:])
    assert e.value.status == ERR_MISALIGNED
