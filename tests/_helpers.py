"""Shared helpers of the GPU parity tests: moving seeded inputs to the
device, and the comparison rules.

Comparison rules (stated once):
  * quantizer codes and scales: bit-identical to the oracle;
  * GEMM, FP32 output: relative Frobenius error <= 1e-3 and max-abs error
    / max |C_ref| <= 5e-3 against the oracle's double-precision sum of
    dequantized products;
  * GEMM, BF16 output: the output is FP32 rounded once to bf16, so every
    element must lie within one bf16 ulp of C_ref (plus 1e-5 * max |C_ref|
    for the FP32 accumulation), and the relative Frobenius distance to
    bf16(C_ref) must be <= 1e-3.
"""
import numpy as np
import torch

REL_FRO = 1e-3
MAX_REL = 5e-3


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    t = torch.from_numpy(np.ascontiguousarray(bits).view(np.int16))
    return t.view(torch.bfloat16).cuda()


def dev(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.float().cpu().numpy()
    return t.cpu().numpy()


def assert_codes_equal(gpu: torch.Tensor, ref: np.ndarray, what: str):
    g = host(gpu)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    if not np.array_equal(g, ref):
        bad = np.argwhere(g != ref)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} code mismatches, first at {i}: "
                             f"gpu {g[i]:#04x} oracle {ref[i]:#04x}")


def assert_scales_equal(gpu: torch.Tensor, ref: np.ndarray, what: str):
    g = host(gpu)
    assert g.shape == ref.shape, (what, g.shape, ref.shape)
    gb, rb = g.view(np.uint32), ref.view(np.uint32)
    if not np.array_equal(gb, rb):
        bad = np.argwhere(gb != rb)
        i = tuple(bad[0])
        raise AssertionError(f"{what}: {len(bad)} scale mismatches, first at {i}: "
                             f"gpu {g[i]!r} oracle {ref[i]!r}")


def gemm_errors(c: np.ndarray, ref: np.ndarray):
    c = c.astype(np.float64)
    diff = c - ref
    rel_fro = np.linalg.norm(diff) / max(np.linalg.norm(ref), 1e-300)
    max_rel = np.abs(diff).max() / max(np.abs(ref).max(), 1e-300)
    return float(rel_fro), float(max_rel)


def assert_gemm_f32(c: np.ndarray, ref: np.ndarray, what: str):
    rel_fro, max_rel = gemm_errors(c, ref)
    assert rel_fro <= REL_FRO and max_rel <= MAX_REL, (what, rel_fro, max_rel)
    return rel_fro, max_rel


def bf16_round(v: np.ndarray) -> np.ndarray:
    """Nearest bf16 (ties to even) of float64 values, via torch's float64 ->
    bf16 cast of values first made exact in float32 where possible."""
    return torch.from_numpy(np.asarray(v, np.float64)).to(torch.bfloat16).double().numpy()


def ulp_bf16(v: np.ndarray) -> np.ndarray:
    a = np.abs(v)
    e = np.floor(np.log2(np.where(a > 0, a, 2.0 ** -133)))
    return 2.0 ** np.maximum(e - 7, -133)


def assert_gemm_bf16(c: np.ndarray, ref: np.ndarray, what: str):
    c = c.astype(np.float64)
    slack = ulp_bf16(ref) + 1e-5 * np.abs(ref).max()
    err = np.abs(c - ref)
    if not np.all(err <= slack):
        i = np.unravel_index(np.argmax(err - slack), err.shape)
        raise AssertionError(f"{what}: element {i} gpu {c[i]!r} ref {ref[i]!r}")
    rb = bf16_round(ref)
    rel = np.linalg.norm(c - rb) / max(np.linalg.norm(rb), 1e-300)
    assert rel <= REL_FRO, (what, rel)
    return float(rel)
