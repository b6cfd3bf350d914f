"""Python binding of libfp8bs: fine-grained FP8 quantization and the
block-scaled FP8 GEMM on B300 (sm_103a).

Argument marshalling only.  Every call goes through the C ABI declared in
include/fp8bs.h (loaded with ctypes from libfp8bs.so next to this file);
PyTorch supplies device memory and the current CUDA stream.  There is no
fallback: if the library is missing, importing this package fails.

Layouts (see include/fp8bs.h): codes are uint8 tensors holding E4M3 bits;
1x128-group scales of X[rows][cols] are float32 [cols/128, rows]; weight
block scales of W[N][K] are float32 [N/128, K/128].
"""
import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8bs.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED_SHAPE, ERR_MISALIGNED, ERR_ARCH, ERR_CUDA, ERR_TIMEOUT = range(7)
OUT_BF16, OUT_F32, OUT_E4M3_1x128 = 0, 1, 2
TILE_AUTO, TILE_128x128, TILE_128x256 = -1, 0, 1
TILE_256x128_PAIR, TILE_256x160_PAIR, TILE_256x192_PAIR = 2, 3, 4
TILE_256x224_PAIR, TILE_256x256_PAIR, TILE_256x192_PAIR_W12 = 5, 6, 7
TILE_256x256_PAIR_W16, TILE_256x192_PAIR_W16, TILE_256x128_PAIR_W16 = 8, 9, 10
TILES = tuple(range(11))
BSCALE_BLOCK_128x128, BSCALE_TILE_1x128 = 0, 1
GROUP = 128

if not os.path.exists(LIB_PATH):
    raise ImportError(f"libfp8bs.so is not built ({LIB_PATH}); run "
                      "`python fp8_fine_grained_18_b300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)
_P, _I64, _I = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int

_SIGS = {
    "fp8bs_quant_act_1x128": [_P, _I64, _I64, _I, _P, _P, _P],
    "fp8bs_quant_weight_128x128": [_P, _I64, _I64, _P, _P, _P, _P, _P],
    "fp8bs_quant_act_dual": [_P, _I64, _I64, _P, _P, _P, _P, _P],
    "fp8bs_quant_act_and_weight": [_P, _I64, _I64, _P, _P, _P, _I64, _I64, _P, _P, _P],
    "fp8bs_quant_act_e5m6": [_P, _I64, _I64, _P, _P, _P, _P, _P],
    "fp8bs_requant_e5m6_to_128x1": [_P, _P, _I64, _I64, _P, _P, _P],
    "fp8bs_quant_per_tensor": [_P, _I64, _I64, _P, _P, _P, _I64, _P],
    "fp8bs_requant_1x128_to_128x1": [_P, _P, _I64, _I64, _P, _P, _P],
    "fp8bs_gemm": [_P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _I, _P],
    "fp8bs_gemm_ex": [_P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _I, _I, _P],
    "fp8bs_gemm_tiled": [_P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _I, _I, _I, _P],
    "fp8bs_gemm_quant_out": [_P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _P, _P],
    "fp8bs_gemm_streamk_workspace": [_I, _I64, _I64, _I64, _I, _P],
    "fp8bs_gemm_streamk": [_P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _I, _P, ctypes.c_size_t, _P],
    "fp8bs_gemm_streamk_noalloc": [_P, _P, _P, _P, _I, _I64, _I64, _I64, _P, _I, _P],
    "fp8bs_debug_gemm_stall": [_P, _P, _P, _P, _I64, _I64, _I64, _P, _I, _I, _P],
    "fp8bs_get_device_error": [_P],
    "fp8bs_status_string": [_I],
    "fp8bs_last_cuda_error": [],
    "fp8bs_version": [],
}
for _name, _args in _SIGS.items():
    _f = getattr(_lib, _name)
    _f.argtypes = _args
    _f.restype = ctypes.c_char_p if _name == "fp8bs_status_string" else ctypes.c_int


class Fp8bsError(RuntimeError):
    def __init__(self, status: int, where: str):
        msg = _lib.fp8bs_status_string(status).decode()
        if status == ERR_CUDA:
            msg += f" (cudaError {_lib.fp8bs_last_cuda_error()})"
        super().__init__(f"{where}: {msg}")
        self.status = status


def lib():
    """The raw ctypes handle of libfp8bs.so."""
    return _lib


def _check(status: int, where: str):
    if status != OK:
        raise Fp8bsError(status, where)


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _empty(shape, dtype, like):
    return torch.empty(shape, dtype=dtype, device=like.device)


def quant_act_1x128(x: torch.Tensor, transpose_out: bool = False, q=None, scales=None):
    """bf16 x[M, K] -> (codes uint8, scales float32).

    transpose_out=False: codes [M, K], scales [K/128, M] (1x128 tiles).
    transpose_out=True:  codes [K, M], scales [M/128, K] (128x1 tiles of x,
    i.e. 1x128 tiles of x transposed).
    """
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    M, K = x.shape
    if transpose_out:
        q = _empty((K, M), torch.uint8, x) if q is None else q
        scales = _empty((M // GROUP, K), torch.float32, x) if scales is None else scales
    else:
        q = _empty((M, K), torch.uint8, x) if q is None else q
        scales = _empty((K // GROUP, M), torch.float32, x) if scales is None else scales
    _check(_lib.fp8bs_quant_act_1x128(_ptr(x), M, K, int(transpose_out), _ptr(q), _ptr(scales),
                                      _stream(x)), "fp8bs_quant_act_1x128")
    return q, scales


def quant_act_dual(x: torch.Tensor, q=None, scales=None, qT=None, scalesT=None):
    """bf16 x[M, K] -> (codes [M, K], scales [K/128, M], codesT [K, M],
    scalesT [M/128, K]): both tilings of quant_act_1x128 from one read."""
    assert x.dtype == torch.bfloat16 and x.dim() == 2 and x.is_contiguous()
    M, K = x.shape
    q = _empty((M, K), torch.uint8, x) if q is None else q
    scales = _empty((K // GROUP, M), torch.float32, x) if scales is None else scales
    qT = _empty((K, M), torch.uint8, x) if qT is None else qT
    scalesT = _empty((M // GROUP, K), torch.float32, x) if scalesT is None else scalesT
    _check(_lib.fp8bs_quant_act_dual(_ptr(x), M, K, _ptr(q), _ptr(scales), _ptr(qT),
                                     _ptr(scalesT), _stream(x)), "fp8bs_quant_act_dual")
    return q, scales, qT, scalesT


def quant_weight_128x128(w: torch.Tensor, transposed: bool = False, q=None, scales=None,
                         qT=None, scalesT=None):
    """bf16 w[N, K] -> (codes [N, K], scales [N/128, K/128]) and, with
    transposed=True, also (codesT [K, N], scalesT [K/128, N/128])."""
    assert w.dtype == torch.bfloat16 and w.dim() == 2 and w.is_contiguous()
    N, K = w.shape
    q = _empty((N, K), torch.uint8, w) if q is None else q
    scales = _empty((N // GROUP, K // GROUP), torch.float32, w) if scales is None else scales
    if transposed:
        qT = _empty((K, N), torch.uint8, w) if qT is None else qT
        scalesT = _empty((K // GROUP, N // GROUP), torch.float32, w) if scalesT is None else scalesT
    _check(_lib.fp8bs_quant_weight_128x128(_ptr(w), N, K, _ptr(q), _ptr(scales),
                                           _ptr(qT if transposed else None),
                                           _ptr(scalesT if transposed else None), _stream(w)),
           "fp8bs_quant_weight_128x128")
    return (q, scales, qT, scalesT) if transposed else (q, scales)


def quant_act_and_weight(x: torch.Tensor, w: torch.Tensor, q=None, scales=None, qw=None,
                         w_scales=None):
    """Q1 of x bf16 [M, K] and Q2 of w bf16 [N, Kw] in one launch.

    Returns (q, scales, qw, w_scales) as quant_act_1x128 and
    quant_weight_128x128 would."""
    assert x.dtype == torch.bfloat16 and w.dtype == torch.bfloat16
    assert x.is_contiguous() and w.is_contiguous()
    M, K = x.shape
    N, Kw = w.shape
    q = _empty((M, K), torch.uint8, x) if q is None else q
    scales = _empty((K // GROUP, M), torch.float32, x) if scales is None else scales
    qw = _empty((N, Kw), torch.uint8, w) if qw is None else qw
    w_scales = _empty((N // GROUP, Kw // GROUP), torch.float32, w) if w_scales is None else w_scales
    _check(_lib.fp8bs_quant_act_and_weight(_ptr(x), M, K, _ptr(q), _ptr(scales), _ptr(w), N, Kw,
                                           _ptr(qw), _ptr(w_scales), _stream(x)),
           "fp8bs_quant_act_and_weight")
    return q, scales, qw, w_scales


def quant_act_e5m6(x: torch.Tensor, with_e4m3: bool = True, packed=None, scales=None, q=None,
                   q_scales=None):
    """E5M6 cache of x bf16 [M, K] with 1x128 scales, plus (with_e4m3) the
    E4M3 1x128 codes from the same read.

    Returns (packed uint8 [M, 3K/2], scales float32 [K/128, M], q, q_scales);
    q and q_scales are None without with_e4m3."""
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    M, K = x.shape
    packed = _empty((M, K // 2 * 3), torch.uint8, x) if packed is None else packed
    scales = _empty((K // GROUP, M), torch.float32, x) if scales is None else scales
    if with_e4m3:
        q = _empty((M, K), torch.uint8, x) if q is None else q
        q_scales = _empty((K // GROUP, M), torch.float32, x) if q_scales is None else q_scales
    else:
        q = q_scales = None
    _check(_lib.fp8bs_quant_act_e5m6(_ptr(x), M, K, _ptr(packed), _ptr(scales), _ptr(q),
                                     _ptr(q_scales), _stream(x)), "fp8bs_quant_act_e5m6")
    return packed, scales, q, q_scales


def requant_e5m6_to_128x1(packed: torch.Tensor, scales: torch.Tensor, qT=None, scalesT=None):
    """E5M6 cache [M, 3K/2] + scales [K/128, M] -> (qT uint8 [K, M], scalesT [M/128, K])."""
    M, K = packed.shape[0], packed.shape[1] // 3 * 2
    qT = _empty((K, M), torch.uint8, packed) if qT is None else qT
    scalesT = _empty((M // GROUP, K), torch.float32, packed) if scalesT is None else scalesT
    _check(_lib.fp8bs_requant_e5m6_to_128x1(_ptr(packed), _ptr(scales), M, K, _ptr(qT),
                                            _ptr(scalesT), _stream(packed)),
           "fp8bs_requant_e5m6_to_128x1")
    return qT, scalesT


def quant_per_tensor(x: torch.Tensor, q=None, scale=None, bcast_shape=None, bcast=None):
    """Per-tensor baseline: x bf16 [rows, cols] -> (q uint8, scale float32 [1],
    bcast float32 of bcast_shape filled with the scale, or None)."""
    assert x.dtype == torch.bfloat16 and x.is_contiguous()
    rows, cols = x.shape
    q = _empty((rows, cols), torch.uint8, x) if q is None else q
    scale = _empty((1,), torch.float32, x) if scale is None else scale
    if bcast is None and bcast_shape is not None:
        bcast = _empty(tuple(bcast_shape), torch.float32, x)
    nb = 0 if bcast is None else bcast.numel()
    _check(_lib.fp8bs_quant_per_tensor(_ptr(x), rows, cols, _ptr(q), _ptr(scale),
                                       _ptr(bcast) if bcast is not None else None, nb,
                                       _stream(x)), "fp8bs_quant_per_tensor")
    return q, scale, bcast


def requant_1x128_to_128x1(q: torch.Tensor, scales: torch.Tensor, qT=None, scalesT=None):
    """codes q[M, K] with scales [K/128, M] -> (qT [K, M], scalesT [M/128, K])."""
    assert q.dtype == torch.uint8 and scales.dtype == torch.float32
    M, K = q.shape
    qT = _empty((K, M), torch.uint8, q) if qT is None else qT
    scalesT = _empty((M // GROUP, K), torch.float32, q) if scalesT is None else scalesT
    _check(_lib.fp8bs_requant_1x128_to_128x1(_ptr(q), _ptr(scales), M, K, _ptr(qT), _ptr(scalesT),
                                             _stream(q)), "fp8bs_requant_1x128_to_128x1")
    return qT, scalesT


def gemm(a: torch.Tensor, sa: torch.Tensor, b: torch.Tensor, sb: torch.Tensor,
         bkind: int = BSCALE_BLOCK_128x128, out_dtype=torch.bfloat16, promote: bool = True,
         out=None, tile: int = TILE_AUTO):
    """C[M, N] = block-scaled a[M, K] * b[N, K]^T (bf16 or float32 out).

    tile: TILE_AUTO (per-shape choice) or one of the TILE_* shapes."""
    assert a.dtype == torch.uint8 and b.dtype == torch.uint8
    M, K = a.shape
    N = b.shape[0]
    odt = OUT_BF16 if out_dtype == torch.bfloat16 else OUT_F32
    c = _empty((M, N), out_dtype, a) if out is None else out
    _check(_lib.fp8bs_gemm_tiled(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), int(bkind), M, N, K,
                                 _ptr(c), odt, int(bool(promote)), int(tile), _stream(a)),
           "fp8bs_gemm")
    return c


def gemm_streamk_workspace(M: int, N: int, K: int, bkind: int = BSCALE_BLOCK_128x128,
                           out_dtype=torch.bfloat16) -> int:
    """Workspace bytes gemm_streamk needs for this problem on the current
    device (0: it runs as gemm)."""
    n = ctypes.c_size_t(0)
    odt = OUT_BF16 if out_dtype == torch.bfloat16 else OUT_F32
    _check(_lib.fp8bs_gemm_streamk_workspace(int(bkind), M, N, K, odt, ctypes.addressof(n)),
           "fp8bs_gemm_streamk_workspace")
    return n.value


def gemm_streamk(a: torch.Tensor, sa: torch.Tensor, b: torch.Tensor, sb: torch.Tensor,
                 bkind: int = BSCALE_BLOCK_128x128, out_dtype=torch.bfloat16, workspace=None,
                 out=None):
    """gemm (promoted) with stream-K scheduling of an uneven last wave.
    workspace: a uint8 CUDA tensor of at least gemm_streamk_workspace bytes
    (allocated here when None)."""
    assert a.dtype == torch.uint8 and b.dtype == torch.uint8
    M, K = a.shape
    N = b.shape[0]
    odt = OUT_BF16 if out_dtype == torch.bfloat16 else OUT_F32
    c = _empty((M, N), out_dtype, a) if out is None else out
    if workspace is None:
        need = gemm_streamk_workspace(M, N, K, bkind, out_dtype)
        workspace = _empty((max(need, 1),), torch.uint8, a) if need else None
    ws_ptr = _ptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() if workspace is not None else 0
    _check(_lib.fp8bs_gemm_streamk(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), int(bkind), M, N, K,
                                   _ptr(c), odt, ws_ptr, ws_bytes, _stream(a)),
           "fp8bs_gemm_streamk")
    return c


def gemm_streamk_noalloc(a: torch.Tensor, sa: torch.Tensor, b: torch.Tensor, sb: torch.Tensor,
                         bkind: int = BSCALE_BLOCK_128x128, out_dtype=torch.bfloat16, out=None):
    """gemm_streamk on the library's fixed scratch (fp8bs_gemm_streamk_noalloc):
    no workspace argument; see include/fp8bs.h for its limit and set-up."""
    assert a.dtype == torch.uint8 and b.dtype == torch.uint8
    M, K = a.shape
    N = b.shape[0]
    odt = OUT_BF16 if out_dtype == torch.bfloat16 else OUT_F32
    c = _empty((M, N), out_dtype, a) if out is None else out
    _check(_lib.fp8bs_gemm_streamk_noalloc(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), int(bkind), M, N,
                                           K, _ptr(c), odt, _stream(a)),
           "fp8bs_gemm_streamk_noalloc")
    return c


def gemm_quant_out(a: torch.Tensor, sa: torch.Tensor, b: torch.Tensor, sb: torch.Tensor,
                   bkind: int = BSCALE_BLOCK_128x128, out=None, out_scales=None):
    """The promoted GEMM with its FP32 result quantized 1x128 in the epilogue.

    Returns (c uint8 [M, N] E4M3 codes, c_scales float32 [N/128, M])."""
    assert a.dtype == torch.uint8 and b.dtype == torch.uint8
    M, K = a.shape
    N = b.shape[0]
    c = _empty((M, N), torch.uint8, a) if out is None else out
    cs = _empty((N // GROUP, M), torch.float32, a) if out_scales is None else out_scales
    _check(_lib.fp8bs_gemm_quant_out(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), int(bkind), M, N, K,
                                     _ptr(c), _ptr(cs), _stream(a)), "fp8bs_gemm_quant_out")
    return c, cs


def debug_gemm_stall(a, sa, b, sb, skip_iter: int, out=None, tile: int = TILE_AUTO):
    """Test support: see fp8bs_debug_gemm_stall in include/fp8bs.h."""
    M, K = a.shape
    N = b.shape[0]
    c = _empty((M, N), torch.float32, a) if out is None else out
    _check(_lib.fp8bs_debug_gemm_stall(_ptr(a), _ptr(sa), _ptr(b), _ptr(sb), M, N, K, _ptr(c),
                                       int(skip_iter), int(tile), _stream(a)),
           "fp8bs_debug_gemm_stall")
    return c


def get_device_error(device=None) -> int:
    """Synchronizes the current stream; returns OK or ERR_TIMEOUT (and clears it)."""
    dev = torch.device("cuda") if device is None else torch.device(device)
    s = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    return _lib.fp8bs_get_device_error(s)


def version() -> int:
    return _lib.fp8bs_version()
