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
