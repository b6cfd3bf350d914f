"""fp8bs_gemm_streamk_noalloc, called through the C ABI: the stream-K GEMM
on the library's fixed scratch, for callers that cannot allocate.  Two
calls in a row must each match fp8bs_gemm_streamk (the same kernel on a
caller workspace) within the GEMM tolerance, and the oracle.  This file is
collected last so that it also runs after every other GPU test."""
import ctypes

import numpy as np
import pytest
import torch

import synth
from tests._helpers import assert_gemm_f32, dev, host

pytestmark = pytest.mark.gpu

TILE = 1
OUT_F32 = 1  # FP8BS_OUT_F32
ERR_UNSUPPORTED_SHAPE = 2
SCRATCH_BYTES = 48 << 20  # FP8BS_NOALLOC_SCRATCH_BYTES


def _entry(fp8bs):
    f = fp8bs.lib().fp8bs_gemm_streamk_noalloc
    P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
    f.argtypes = [P, P, P, P, I, I64, I64, I64, P, I, P]
    f.restype = I
    return f


def _call(f, a, sa, b, sb, bkind, c):
    M, K = a.shape
    N = b.shape[0]
    st = f(a.data_ptr(), sa.data_ptr(), b.data_ptr(), sb.data_ptr(), bkind, M, N, K,
           c.data_ptr(), OUT_F32, torch.cuda.current_stream().cuda_stream)
    return st


def test_noalloc_matches_streamk_two_calls(fp8bs, oracle_mod):
    M, N, K = 512, 512, 8192  # 4 pair tiles of 64 K-groups: every tile split
    rng = np.random.default_rng(17)
    a, sa = oracle_mod.quant_act_1x128(synth.normal(rng, (M, K), 1.0))
    b, sb = oracle_mod.quant_act_1x128(synth.normal(rng, (N, K), 1e-3))
    need = fp8bs.gemm_streamk_workspace(M, N, K, TILE, torch.float32)
    assert 0 < need <= SCRATCH_BYTES
    da, dsa, db, dsb = dev(a), dev(sa), dev(b), dev(sb)
    ref_api = host(fp8bs.gemm_streamk(da, dsa, db, dsb, TILE, out_dtype=torch.float32))
    ref = oracle_mod.gemm(a, sa, b, sb, TILE)
    f = _entry(fp8bs)
    scale = np.abs(ref_api).max()
    for call in range(2):
        c = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _call(f, da, dsa, db, dsb, TILE, c) == 0
        got = host(c)
        assert np.abs(got - ref_api).max() <= 1e-6 * scale, f"call {call}"
        assert_gemm_f32(got, ref, f"no-alloc stream-K call {call}")


def test_noalloc_scratch_covers_every_plan(fp8bs):
    """Every stream-K plan on this device, few-tile problems and uneven last
    waves of large ones alike, stays within the fixed scratch: the
    no-allocation call refuses none of them (the refusal is for devices with
    more SMs)."""
    worst = 0
    for M in (128, 256, 512, 1024, 2048, 4096, 7168, 8192):
        for N in (128, 256, 512, 1024, 2048, 4096, 7168, 8192):
            for bkind in (0, TILE):
                worst = max(worst, fp8bs.gemm_streamk_workspace(M, N, 8192, bkind, torch.float32))
    assert 0 < worst <= SCRATCH_BYTES


def test_noalloc_refuses_before_launch(fp8bs):
    """A refused call launches nothing (here: K not a multiple of 128)."""
    M, N, K = 256, 256, 1000
    a = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    sa = torch.ones((8, M), dtype=torch.float32, device="cuda")
    b = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    sb = torch.ones((8, N), dtype=torch.float32, device="cuda")
    c = torch.full((M, N), 7.0, dtype=torch.float32, device="cuda")
    assert _call(_entry(fp8bs), a, sa, b, sb, TILE, c) == ERR_UNSUPPORTED_SHAPE
    torch.cuda.synchronize()
    assert bool((c == 7.0).all())
