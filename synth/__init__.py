"""Seeded synthetic inputs shaped like the pages' workloads.

Shared by the tests, the smoke check and the benchmark.  It holds none of the
method's arithmetic: it only draws random numbers (numpy PCG64, seeded) and
rounds them to bf16 (round-to-nearest-even), returning bf16 bit patterns as
uint16 arrays.  Workload recipes (shapes, distributions, outlier channels)
are listed in WORKLOADS.

Distributions: "N(0, sigma)" means standard deviation sigma; Student-t with
nu=4 is Z / sqrt(chi2_4 / 4) with chi2_4 = -2 ln(U1 U2); "log-uniform row
magnitudes" multiplies each row of U(-1, 1) by 10**U(-2, 2).
"""
from dataclasses import dataclass, field

import numpy as np


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round float32 values to bf16 (nearest, ties to even); uint16 bits."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = (u & 0x7FFFFFFF) > 0x7F800000
    lsb = (u >> 16) & 1
    r = ((u + np.uint32(0x7FFF) + lsb) >> 16).astype(np.uint16)
    return np.where(nan, np.uint16(0x7FC0), r)


def bf16_bits_to_f32(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal(rng, shape, sigma=1.0) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma))


def normal_with_outlier_columns(rng, shape, n_cols, factor, sigma=1.0):
    """N(0, sigma) with n_cols distinct seeded columns multiplied by factor."""
    x = rng.standard_normal(shape, dtype=np.float32) * np.float32(sigma)
    cols = np.sort(rng.choice(shape[1], size=n_cols, replace=False))
    x[:, cols] *= np.float32(factor)
    return f32_to_bf16_bits(x), cols


def student_t4(rng, shape) -> np.ndarray:
    z = rng.standard_normal(shape, dtype=np.float32)
    u1 = rng.random(shape, dtype=np.float32)
    u2 = rng.random(shape, dtype=np.float32)
    # 1 - U keeps the logarithm's argument in (0, 1].
    chi2 = -2.0 * np.log((1.0 - u1) * (1.0 - u2))
    return f32_to_bf16_bits(z / np.sqrt(chi2 / 4.0))


def loguniform_rows(rng, shape) -> np.ndarray:
    u = rng.uniform(-1.0, 1.0, size=shape).astype(np.float32)
    mag = (10.0 ** rng.uniform(-2.0, 2.0, size=(shape[0], 1))).astype(np.float32)
    return f32_to_bf16_bits(u * mag)


@dataclass
class Workload:
    name: str
    seed: int
    M: int
    N: int
    K: int
    out: str  # "f32" or "bf16"
    note: str = ""
    extra: dict = field(default_factory=dict)


# The five workloads.  The seed is the workload's index (tiny = 0).
WORKLOADS = {
    "tiny": Workload("tiny", 0, 128, 256, 512, "f32",
                     "A N(0,1) with 4 seeded outlier columns x50; B N(0,0.02)"),
    "dense": Workload("dense", 1, 4096, 7168, 7168, "bf16",
                      "A N(0,1) with 7 (0.1% of 7168) seeded channels x100; W N(0,0.02)"),
    "moe": Workload("moe", 2, 8192, 4096, 7168, "bf16",
                    "A Student-t nu=4; W N(0,0.02) (gate and up fused, 2x2048)"),
    "bwd": Workload("bwd", 3, 4096, 7168, 2048, "bf16",
                    "X[4096,2048] N(0,1) with 2 channels x100; W[7168,2048] N(0,0.02); "
                    "dY[4096,7168] N(0,1e-3)"),
    "stress": Workload("stress", 4, 8192, 8192, 16384, "f32",
                       "A, B U(-1,1) with per-row magnitudes 10^U(-2,2)"),
}


def make_inputs(name: str, scale_rows: int = None, seed: int = None) -> dict:
    """bf16 bit arrays of a workload.

    Forward workloads return {"A": [M, K], "B": [N, K]}; "bwd" returns
    {"X": [M, K], "W": [N, K], "dY": [M, N]} with M tokens, N output
    features, K input features.  scale_rows, if given, replaces M (the token
    count) to draw a smaller batch of the same distribution; seed, if given,
    replaces the workload's seed (another batch of the same distribution).
    """
    w = WORKLOADS[name]
    rng = np.random.default_rng(w.seed if seed is None else seed)
    M = w.M if scale_rows is None else scale_rows
    if name == "tiny":
        A, _ = normal_with_outlier_columns(rng, (M, w.K), 4, 50.0)
        return {"A": A, "B": normal(rng, (w.N, w.K), 0.02)}
    if name == "dense":
        A, _ = normal_with_outlier_columns(rng, (M, w.K), (w.K * 1) // 1000, 100.0)
        return {"A": A, "B": normal(rng, (w.N, w.K), 0.02)}
    if name == "moe":
        return {"A": student_t4(rng, (M, w.K)), "B": normal(rng, (w.N, w.K), 0.02)}
    if name == "bwd":
        X, _ = normal_with_outlier_columns(rng, (M, w.K), 2, 100.0)
        W = normal(rng, (w.N, w.K), 0.02)
        dY = normal(rng, (M, w.N), 1e-3)
        return {"X": X, "W": W, "dY": dY}
    if name == "stress":
        return {"A": loguniform_rows(rng, (M, w.K)), "B": loguniform_rows(rng, (w.N, w.K))}
    raise KeyError(name)
