"""Accumulation precision study (page P1, paragraphs 3-4; page P2,
paragraph 3): FP32 promotion every 128 K against a deliberately un-promoted
GEMM that leaves the whole K inside the tensor core, on operands whose scales
are constant along K (row-wise codes, so both variants compute the same sum).
The stress workload's inputs: U(-1, 1) rows with magnitudes 10^U(-2, 2).

The promoted result must meet the stated tolerances at every K.  The
un-promoted error is measured and printed (B300's tensor-core accumulation
width is not documented, so no bound is asserted beyond sanity); beside it
the CPU model of a 14-bit accumulator (PARITY UNPINNED: a model of the
pages' H800 description, not a definition) shows the degradation the pages
report, on a sample of the same outputs.

Run with `-s` to see the table."""
import numpy as np
import pytest
import torch

import synth
from tests._helpers import assert_gemm_f32, dev, gemm_errors, host

pytestmark = pytest.mark.gpu

TILE = 1


@pytest.mark.parametrize("K", [1024, 4096, 16384])
def test_promoted_vs_unpromoted(fp8bs, oracle_mod, K):
    rng = np.random.default_rng(100 + K)
    M = N = 128
    a, sa = oracle_mod.quant_rowwise(synth.loguniform_rows(rng, (M, K)))
    b, sb = oracle_mod.quant_rowwise(synth.loguniform_rows(rng, (N, K)))
    ref = oracle_mod.gemm(a, sa, b, sb, TILE)
    da, dsa, db, dsb = dev(a), dev(sa), dev(b), dev(sb)
    c_pr = host(fp8bs.gemm(da, dsa, db, dsb, TILE, out_dtype=torch.float32))
    c_un = host(fp8bs.gemm(da, dsa, db, dsb, TILE, out_dtype=torch.float32, promote=False))
    e_pr = gemm_errors(c_pr, ref)
    e_un = gemm_errors(c_un, ref)
    # the CPU 14-bit accumulator model (no promotion) on 256 sampled outputs
    srng = np.random.default_rng(K)
    ms, ns = srng.integers(0, M, 256), srng.integers(0, N, 256)
    emu = oracle_mod.gemm_limited_acc(a, sa, b, sb, TILE, ms, ns, bits=14, group=32,
                                      promote_every=0)
    refs = ref[ms, ns]
    emu_max_rel = float(np.abs(emu - refs).max() / np.abs(refs).max())
    emu_fro = float(np.linalg.norm(emu - refs) / np.linalg.norm(refs))
    print(f"\nK={K:6d}  promoted rel_fro {e_pr[0]:.2e} max_rel {e_pr[1]:.2e} | "
          f"un-promoted (B300 tensor core) rel_fro {e_un[0]:.2e} max_rel {e_un[1]:.2e} | "
          f"14-bit model rel_fro {emu_fro:.2e} max_rel {emu_max_rel:.2e}")
    assert_gemm_f32(c_pr, ref, f"promoted K={K}")
    assert np.isfinite(e_un[0]) and e_un[0] < 0.1


def _pow2_code(e: int) -> int:
    """E4M3 code of 2^e for -9 <= e <= 8 (subnormals 2^-9 .. 2^-7)."""
    return (1 << (e + 9)) if e < -6 else ((e + 7) << 3)


@pytest.mark.parametrize("big_exp,sign", [(0, 1), (0, -1), (4, 1), (8, 1)])
def test_accumulator_width_hand_worked(fp8bs, oracle_mod, big_exp, sign):
    """A direct probe of the tensor-core accumulator: row 0 of A and B hold
    one product 2^big_exp followed by 4095 products of +-2^-18 (2^-9 * 2^-9,
    the smallest E4M3 subnormal squared), all scales 1, K = 4096.  The exact
    sum is 2^big_exp +- 4095 * 2^-18.  The 14-bit model of the pages' H800
    accumulator aligns every group to the big product's exponent and drops
    (or, for negative terms, floors to one unit) every small product, which
    costs 4095 * 2^-18 = 1.6% at big_exp = 0 -- the pages' "nearly 2%".
    Printed: the fraction of the small products each variant keeps.  Asserted:
    the promoted result is the exact sum rounded once to FP32 where that is
    exact (big_exp = 0, whose 128-K partials are exact in FP32), and every
    variant lies between the model and the exact sum."""
    K = 4096
    a = np.zeros((1, K), np.uint8)
    b = np.zeros((128, K), np.uint8)
    hi = big_exp // 2
    a[0, 0], b[0, 0] = _pow2_code(hi), _pow2_code(big_exp - hi)
    tiny = _pow2_code(-9)
    a[0, 1:] = tiny
    b[0, 1:] = tiny | (0x80 if sign < 0 else 0)
    sa = np.ones((K // 128, 1), np.float32)
    sb = np.ones((K // 128, 128), np.float32)
    exact = 2.0 ** big_exp + sign * (K - 1) * 2.0 ** -18
    ref = oracle_mod.gemm(a, sa, b, sb, TILE)[0, 0]
    assert ref == exact
    model = oracle_mod.gemm_limited_acc(a, sa, b, sb, TILE, np.array([0]), np.array([0]),
                                        bits=14, group=32, promote_every=0)[0]
    da, dsa, db, dsb = dev(a), dev(sa), dev(b), dev(sb)
    c_pr = float(host(fp8bs.gemm(da, dsa, db, dsb, TILE, out_dtype=torch.float32))[0, 0])
    c_un = float(host(fp8bs.gemm(da, dsa, db, dsb, TILE, out_dtype=torch.float32,
                                 promote=False))[0, 0])
    small = sign * (K - 1) * 2.0 ** -18

    def kept(v):
        return (v - 2.0 ** big_exp) / small

    print(f"\nbig 2^{big_exp}, small {'+' if sign > 0 else '-'}2^-18 x {K - 1}: exact {exact!r} | "
          f"promoted {c_pr!r} (keeps {kept(c_pr):.4f}) | un-promoted {c_un!r} "
          f"(keeps {kept(c_un):.4f}) | 14-bit model {model!r} (keeps {kept(model):.4f})")
    if big_exp == 0:
        assert c_pr == np.float32(exact)
    lo, hi_ = sorted((model, exact))
    for v in (c_pr, c_un):
        assert lo - abs(exact) * 2.0 ** -23 <= v <= hi_ + abs(exact) * 2.0 ** -23
