"""CPU oracle for fine-grained FP8 quantization and the block-scaled GEMM.

TEST INFRASTRUCTURE ONLY: imported by tests/, the smoke check and the
benchmark's CPU-baseline leg, never by the fp8_fine_grained_18_b300 package.
A thin ctypes layer over the plain C99 code in fp8bs_oracle.c; every
function takes and returns numpy arrays.  bf16 tensors travel as uint16 bit
patterns.  Scale layouts follow fp8bs_oracle.h.
"""
import ctypes
import os

import numpy as np

from . import build as _build

BSCALE_BLOCK_128x128 = 0
BSCALE_TILE_1x128 = 1
GROUP = 128

_lib = None


def lib():
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I = ctypes.c_int64
        L.fp8bs_oracle_e4m3_decode.restype = ctypes.c_double
        L.fp8bs_oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
        L.fp8bs_oracle_e4m3_encode.restype = ctypes.c_uint8
        L.fp8bs_oracle_e4m3_encode.argtypes = [ctypes.c_float]
        L.fp8bs_oracle_e5m6_decode.restype = ctypes.c_double
        L.fp8bs_oracle_e5m6_decode.argtypes = [ctypes.c_uint16]
        L.fp8bs_oracle_e5m6_encode.restype = ctypes.c_uint16
        L.fp8bs_oracle_e5m6_encode.argtypes = [ctypes.c_float]
        L.fp8bs_oracle_e5m6_pack.argtypes = [P, I, P]
        L.fp8bs_oracle_e5m6_unpack.argtypes = [P, I, P]
        L.fp8bs_oracle_quant_act_e5m6_1x128.argtypes = [P, I, I, P, P]
        L.fp8bs_oracle_requant_e5m6_to_128x1.argtypes = [P, P, I, I, P, P]
        L.fp8bs_oracle_bf16_to_float.restype = ctypes.c_float
        L.fp8bs_oracle_bf16_to_float.argtypes = [ctypes.c_uint16]
        L.fp8bs_oracle_double_to_bf16.restype = ctypes.c_uint16
        L.fp8bs_oracle_double_to_bf16.argtypes = [ctypes.c_double]
        L.fp8bs_oracle_quant_act_1x128.argtypes = [P, I, I, P, P]
        L.fp8bs_oracle_quant_act_128x1.argtypes = [P, I, I, P, P]
        L.fp8bs_oracle_quant_f32_1x128.argtypes = [P, I, I, P, P]
        L.fp8bs_oracle_quant_per_tensor.argtypes = [P, I, I, P, P]
        L.fp8bs_oracle_quant_weight_128x128.argtypes = [P, I, I, P, P, P, P]
        L.fp8bs_oracle_requant_1x128_to_128x1.argtypes = [P, P, I, I, P, P]
        L.fp8bs_oracle_quant_rowwise.argtypes = [P, I, I, P, P]
        L.fp8bs_oracle_gemm.argtypes = [P, P, P, P, ctypes.c_int, I, I, I, P]
        L.fp8bs_oracle_gemm_sampled.argtypes = [P, P, P, P, ctypes.c_int, I, I, I, P, P, I, P]
        L.fp8bs_oracle_gemm_limited_acc.argtypes = [
            P, P, P, P, ctypes.c_int, I, I, I, ctypes.c_int, ctypes.c_int,
            ctypes.c_int, P, P, I, P]
        L.fp8bs_oracle_num_threads.restype = ctypes.c_int
        for f in ("quant_act_1x128", "quant_act_128x1", "quant_f32_1x128", "quant_weight_128x128",
                  "requant_1x128_to_128x1", "quant_rowwise", "quant_per_tensor", "gemm", "e5m6_pack", "e5m6_unpack",
                  "quant_act_e5m6_1x128", "requant_e5m6_to_128x1",
                  "gemm_sampled", "gemm_limited_acc"):
            getattr(L, "fp8bs_oracle_" + f).restype = None
        _lib = L
    return _lib


def _p(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a)
    assert a.dtype == dtype, (a.dtype, dtype)
    return a


def num_threads() -> int:
    return lib().fp8bs_oracle_num_threads()


# --- codec ---------------------------------------------------------------

def e4m3_decode(code: int) -> float:
    return lib().fp8bs_oracle_e4m3_decode(int(code))


def e4m3_encode(y: float) -> int:
    return lib().fp8bs_oracle_e4m3_encode(float(np.float32(y)))


def e5m6_decode(code: int) -> float:
    return lib().fp8bs_oracle_e5m6_decode(int(code))


def e5m6_encode(y: float) -> int:
    return lib().fp8bs_oracle_e5m6_encode(float(np.float32(y)))


def e5m6_decode_array(codes: np.ndarray) -> np.ndarray:
    """Elementwise decode (float64) of 12-bit codes via the scalar definition."""
    table = np.array([e5m6_decode(c) for c in range(4096)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint16) & 0xFFF]


def e5m6_pack(codes: np.ndarray) -> np.ndarray:
    """12-bit codes [..., n] (n even) -> bytes [..., 3n/2]."""
    c = np.ascontiguousarray(codes, dtype=np.uint16)
    out = np.empty(c.shape[:-1] + (c.shape[-1] // 2 * 3,), np.uint8)
    lib().fp8bs_oracle_e5m6_pack(_p(c), c.size, _p(out))
    return out


def e5m6_unpack(packed: np.ndarray) -> np.ndarray:
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.empty(p.shape[:-1] + (p.shape[-1] // 3 * 2,), np.uint16)
    lib().fp8bs_oracle_e5m6_unpack(_p(p), out.size, _p(out))
    return out


def quant_act_e5m6_1x128(x_bf16: np.ndarray):
    """bf16 bits [M, K] -> (packed E5M6 uint8 [M, 3K/2], s float32 [K/128, M])."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    packed = np.empty((M, K // 2 * 3), np.uint8)
    s = np.empty((K // GROUP, M), np.float32)
    lib().fp8bs_oracle_quant_act_e5m6_1x128(_p(x), M, K, _p(packed), _p(s))
    return packed, s


def requant_e5m6_to_128x1(packed: np.ndarray, s: np.ndarray):
    """packed [M, 3K/2], s [K/128, M] -> (qT uint8 [K, M], sT float32 [M/128, K])."""
    pk = _c(packed, np.uint8)
    sc = _c(s, np.float32)
    M, K = pk.shape[0], pk.shape[1] // 3 * 2
    qT = np.empty((K, M), np.uint8)
    sT = np.empty((M // GROUP, K), np.float32)
    lib().fp8bs_oracle_requant_e5m6_to_128x1(_p(pk), _p(sc), M, K, _p(qT), _p(sT))
    return qT, sT


def bf16_to_float(bits: int) -> float:
    return lib().fp8bs_oracle_bf16_to_float(int(bits))


def e4m3_decode_array(codes: np.ndarray) -> np.ndarray:
    """Elementwise decode (float64) via the oracle's scalar definition."""
    table = np.array([e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[np.asarray(codes, dtype=np.uint8)]


def double_to_bf16_array(v: np.ndarray) -> np.ndarray:
    L = lib()
    flat = np.asarray(v, dtype=np.float64).ravel()
    out = np.fromiter((L.fp8bs_oracle_double_to_bf16(float(x)) for x in flat),
                      dtype=np.uint16, count=flat.size)
    return out.reshape(np.shape(v))


# --- quantizers ----------------------------------------------------------

def quant_act_1x128(x_bf16: np.ndarray):
    """x: uint16 [M, K] -> (q uint8 [M, K], s float32 [K/128, M])."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // GROUP, M), np.float32)
    lib().fp8bs_oracle_quant_act_1x128(_p(x), M, K, _p(q), _p(s))
    return q, s


def quant_per_tensor(x_bf16: np.ndarray):
    """bf16 bits [rows, cols] -> (q uint8 [rows, cols], s float32 scalar)."""
    x = _c(x_bf16, np.uint16)
    rows, cols = x.shape
    q = np.empty((rows, cols), np.uint8)
    s = np.empty(1, np.float32)
    lib().fp8bs_oracle_quant_per_tensor(_p(x), rows, cols, _p(q), _p(s))
    return q, s[0]


def quant_f32_1x128(x: np.ndarray):
    """x: float32 [M, K] -> (q uint8 [M, K], s float32 [K/128, M])."""
    x = _c(x, np.float32)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // GROUP, M), np.float32)
    lib().fp8bs_oracle_quant_f32_1x128(_p(x), M, K, _p(q), _p(s))
    return q, s


def quant_act_128x1(x_bf16: np.ndarray):
    """x: uint16 [M, N] -> (qT uint8 [N, M], sT float32 [M/128, N])."""
    x = _c(x_bf16, np.uint16)
    M, N = x.shape
    qT = np.empty((N, M), np.uint8)
    sT = np.empty((M // GROUP, N), np.float32)
    lib().fp8bs_oracle_quant_act_128x1(_p(x), M, N, _p(qT), _p(sT))
    return qT, sT


def quant_weight_128x128(w_bf16: np.ndarray, transposed: bool = False):
    """w: uint16 [N, K] -> (q [N, K], s [N/128, K/128]) (+ qT [K, N], sT [K/128, N/128])."""
    w = _c(w_bf16, np.uint16)
    N, K = w.shape
    q = np.empty((N, K), np.uint8)
    s = np.empty((N // GROUP, K // GROUP), np.float32)
    qT = np.empty((K, N), np.uint8) if transposed else None
    sT = np.empty((K // GROUP, N // GROUP), np.float32) if transposed else None
    lib().fp8bs_oracle_quant_weight_128x128(_p(w), N, K, _p(q), _p(s), _p(qT), _p(sT))
    return (q, s, qT, sT) if transposed else (q, s)


def requant_1x128_to_128x1(q: np.ndarray, s: np.ndarray):
    """q: uint8 [M, K], s: float32 [K/128, M] -> (qT [K, M], sT [M/128, K])."""
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    M, K = q.shape
    qT = np.empty((K, M), np.uint8)
    sT = np.empty((M // GROUP, K), np.float32)
    lib().fp8bs_oracle_requant_1x128_to_128x1(_p(q), _p(s), M, K, _p(qT), _p(sT))
    return qT, sT


def quant_rowwise(x_bf16: np.ndarray):
    """x: uint16 [M, K] -> (q [M, K], s [K/128, M] with every K-group equal)."""
    x = _c(x_bf16, np.uint16)
    M, K = x.shape
    q = np.empty((M, K), np.uint8)
    s = np.empty((K // GROUP, M), np.float32)
    lib().fp8bs_oracle_quant_rowwise(_p(x), M, K, _p(q), _p(s))
    return q, s


# --- GEMM ----------------------------------------------------------------

def gemm(a, sa, b, sb, bkind=BSCALE_BLOCK_128x128) -> np.ndarray:
    """C = sum of dequantized products in float64, [M, N]."""
    a = _c(a, np.uint8); b = _c(b, np.uint8)
    sa = _c(sa, np.float32); sb = _c(sb, np.float32)
    M, K = a.shape
    N = b.shape[0]
    c = np.empty((M, N), np.float64)
    lib().fp8bs_oracle_gemm(_p(a), _p(sa), _p(b), _p(sb), int(bkind), M, N, K, _p(c))
    return c


def gemm_sampled(a, sa, b, sb, bkind, ms, ns) -> np.ndarray:
    a = _c(a, np.uint8); b = _c(b, np.uint8)
    sa = _c(sa, np.float32); sb = _c(sb, np.float32)
    ms = _c(np.asarray(ms, np.int64), np.int64)
    ns = _c(np.asarray(ns, np.int64), np.int64)
    M, K = a.shape
    N = b.shape[0]
    out = np.empty(ms.size, np.float64)
    lib().fp8bs_oracle_gemm_sampled(_p(a), _p(sa), _p(b), _p(sb), int(bkind), M, N, K,
                                    _p(ms), _p(ns), ms.size, _p(out))
    return out


def gemm_limited_acc(a, sa, b, sb, bkind, ms, ns, bits=14, group=32,
                     promote_every=0) -> np.ndarray:
    """Parity unpinned: the limited-precision accumulator model (see header)."""
    a = _c(a, np.uint8); b = _c(b, np.uint8)
    sa = _c(sa, np.float32); sb = _c(sb, np.float32)
    ms = _c(np.asarray(ms, np.int64), np.int64)
    ns = _c(np.asarray(ns, np.int64), np.int64)
    M, K = a.shape
    N = b.shape[0]
    out = np.empty(ms.size, np.float64)
    lib().fp8bs_oracle_gemm_limited_acc(_p(a), _p(sa), _p(b), _p(sb), int(bkind), M, N, K,
                                        int(bits), int(group), int(promote_every),
                                        _p(ms), _p(ns), ms.size, _p(out))
    return out
