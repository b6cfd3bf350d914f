"""Host-side checks of the C ABI (no GPU needed): the library loads, exports
every entry point include/fp8bs.h declares, and rejects invalid arguments
synchronously, before any CUDA call."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp8bs.h")


@pytest.fixture(scope="module")
def libfp8bs():
    import __graft_entry__
    __graft_entry__._load_builder().build()
    import fp8_fine_grained_18_b300 as m
    return m


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8bs_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared_functions()
    for required in ("fp8bs_quant_act_1x128", "fp8bs_quant_weight_128x128",
                     "fp8bs_requant_1x128_to_128x1", "fp8bs_quant_act_dual", "fp8bs_gemm",
                     "fp8bs_gemm_ex", "fp8bs_gemm_quant_out", "fp8bs_quant_per_tensor",
                     "fp8bs_quant_act_e5m6", "fp8bs_requant_e5m6_to_128x1",
                     "fp8bs_quant_act_and_weight",
                     "fp8bs_status_string", "fp8bs_get_device_error"):
        assert required in names


def test_library_exports_every_declared_symbol(libfp8bs):
    lib = ctypes.CDLL(libfp8bs.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing


def test_status_strings(libfp8bs):
    lib = libfp8bs.lib()
    for s in range(7):
        assert lib.fp8bs_status_string(s)
    assert lib.fp8bs_status_string(0) == b"ok"
    assert lib.fp8bs_version() >= 100


FAKE = ctypes.c_void_p(0x10000)      # never dereferenced: rejected first
FAKE_ODD = ctypes.c_void_p(0x10008)  # 8-byte aligned only


def test_quant_argument_errors(libfp8bs):
    L, m = libfp8bs.lib(), libfp8bs
    # no-ops need no pointers
    assert L.fp8bs_quant_act_1x128(None, 0, 128, 0, None, None, None) == m.OK
    assert L.fp8bs_quant_act_1x128(None, 5, 0, 0, None, None, None) == m.OK
    assert L.fp8bs_quant_act_1x128(FAKE, -1, 128, 0, FAKE, FAKE, None) == m.ERR_INVALID_ARG
    assert L.fp8bs_quant_act_1x128(FAKE, 4, 128, 2, FAKE, FAKE, None) == m.ERR_INVALID_ARG
    assert L.fp8bs_quant_act_1x128(None, 4, 128, 0, FAKE, FAKE, None) == m.ERR_INVALID_ARG
    assert L.fp8bs_quant_act_1x128(FAKE, 4, 100, 0, FAKE, FAKE, None) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_quant_act_1x128(FAKE, 100, 128, 1, FAKE, FAKE, None) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_quant_act_1x128(FAKE_ODD, 4, 128, 0, FAKE, FAKE, None) == m.ERR_MISALIGNED
    assert L.fp8bs_quant_weight_128x128(FAKE, 128, 128, FAKE, FAKE, FAKE, None, None) == m.ERR_INVALID_ARG
    assert L.fp8bs_quant_weight_128x128(FAKE, 100, 128, FAKE, FAKE, None, None, None) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_quant_weight_128x128(FAKE, 128, 128, FAKE, FAKE_ODD, None, None, None) == m.ERR_MISALIGNED
    assert L.fp8bs_requant_1x128_to_128x1(FAKE, FAKE, 128, 128, FAKE, None, None) == m.ERR_INVALID_ARG
    assert L.fp8bs_quant_act_dual(None, 0, 128, None, None, None, None, None) == m.OK
    assert L.fp8bs_quant_act_dual(FAKE, 128, 128, FAKE, FAKE, FAKE, None, None) == m.ERR_INVALID_ARG
    assert L.fp8bs_quant_act_dual(FAKE, 100, 128, FAKE, FAKE, FAKE, FAKE, None) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_quant_act_dual(FAKE, 128, 128, FAKE_ODD, FAKE, FAKE, FAKE, None) == m.ERR_MISALIGNED
    assert L.fp8bs_requant_1x128_to_128x1(FAKE, FAKE, 129, 128, FAKE, FAKE, None) == m.ERR_UNSUPPORTED_SHAPE
    aw = L.fp8bs_quant_act_and_weight
    assert aw(None, 0, 128, None, None, None, 0, 128, None, None, None) == m.OK
    assert aw(FAKE, -1, 128, FAKE, FAKE, FAKE, 128, 128, FAKE, FAKE, None) == m.ERR_INVALID_ARG
    assert aw(FAKE, 4, 128, FAKE, FAKE, None, 128, 128, FAKE, FAKE, None) == m.ERR_INVALID_ARG
    assert aw(FAKE, 4, 128, FAKE, FAKE, FAKE, 100, 128, FAKE, FAKE, None) == m.ERR_UNSUPPORTED_SHAPE
    assert aw(FAKE, 4, 96, FAKE, FAKE, FAKE, 128, 128, FAKE, FAKE, None) == m.ERR_UNSUPPORTED_SHAPE
    assert aw(FAKE, 4, 128, FAKE, FAKE, FAKE_ODD, 128, 128, FAKE, FAKE, None) == m.ERR_MISALIGNED
    # an empty operand defers to the other call's checks
    assert aw(FAKE, 0, 128, None, None, FAKE, 100, 128, FAKE, FAKE, None) == m.ERR_UNSUPPORTED_SHAPE
    e5 = L.fp8bs_quant_act_e5m6
    assert e5(None, 0, 128, None, None, None, None, None) == m.OK
    assert e5(FAKE, 4, 128, FAKE, FAKE, FAKE, None, None) == m.ERR_INVALID_ARG  # q without scales
    assert e5(FAKE, 4, 128, None, FAKE, None, None, None) == m.ERR_INVALID_ARG
    assert e5(FAKE, 4, 96, FAKE, FAKE, None, None, None) == m.ERR_UNSUPPORTED_SHAPE
    assert e5(FAKE, 4, 128, FAKE_ODD, FAKE, None, None, None) == m.ERR_MISALIGNED
    r5 = L.fp8bs_requant_e5m6_to_128x1
    assert r5(None, None, 0, 128, None, None, None) == m.OK
    assert r5(FAKE, FAKE, 128, 128, FAKE, None, None) == m.ERR_INVALID_ARG
    assert r5(FAKE, FAKE, 100, 128, FAKE, FAKE, None) == m.ERR_UNSUPPORTED_SHAPE
    assert r5(FAKE, FAKE_ODD, 128, 128, FAKE, FAKE, None) == m.ERR_MISALIGNED
    pt = L.fp8bs_quant_per_tensor
    assert pt(None, 0, 16, None, None, None, 0, None) == m.OK
    assert pt(FAKE, -1, 16, FAKE, FAKE, None, 0, None) == m.ERR_INVALID_ARG
    assert pt(FAKE, 4, 16, FAKE, FAKE, None, 5, None) == m.ERR_INVALID_ARG      # n_bcast without array
    assert pt(FAKE, 4, 16, FAKE, FAKE, FAKE, -1, None) == m.ERR_INVALID_ARG
    assert pt(FAKE, 4, 16, FAKE, None, None, 0, None) == m.ERR_INVALID_ARG
    assert pt(FAKE, 4, 24, FAKE, FAKE, None, 0, None) == m.ERR_UNSUPPORTED_SHAPE
    assert pt(FAKE_ODD, 4, 16, FAKE, FAKE, None, 0, None) == m.ERR_MISALIGNED
    assert pt(FAKE, 4, 16, FAKE, ctypes.c_void_p(0x10002), None, 0, None) == m.ERR_MISALIGNED


def test_gemm_argument_errors(libfp8bs):
    L, m = libfp8bs.lib(), libfp8bs
    args = lambda M, N, K, bk=0, out=0, pr=1, a=FAKE, c=FAKE: (  # noqa: E731
        a, FAKE, FAKE, FAKE, bk, M, N, K, c, out, pr, None)
    assert L.fp8bs_gemm_ex(*args(0, 256, 128)) == m.OK
    assert L.fp8bs_gemm_ex(*args(8, 0, 128)) == m.OK
    assert L.fp8bs_gemm_ex(*args(-1, 256, 128)) == m.ERR_INVALID_ARG
    assert L.fp8bs_gemm_ex(*args(8, 256, 128, bk=2)) == m.ERR_INVALID_ARG
    assert L.fp8bs_gemm_ex(*args(8, 256, 128, out=3)) == m.ERR_INVALID_ARG
    # E4M3 output needs the scale array: only fp8bs_gemm_quant_out gives one
    assert L.fp8bs_gemm_ex(*args(8, 256, 128, out=m.OUT_E4M3_1x128)) == m.ERR_INVALID_ARG
    qargs = lambda M, N, K, cs=FAKE: (FAKE, FAKE, FAKE, FAKE, 0, M, N, K, FAKE, cs, None)  # noqa: E731
    assert L.fp8bs_gemm_quant_out(*qargs(0, 256, 128)) == m.OK
    assert L.fp8bs_gemm_quant_out(*qargs(8, 256, 128, cs=None)) == m.ERR_INVALID_ARG
    assert L.fp8bs_gemm_quant_out(*qargs(8, 144, 128)) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_gemm_quant_out(*qargs(8, 256, 100)) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_gemm_quant_out(*qargs(8, 256, 128, cs=FAKE_ODD)) == m.ERR_MISALIGNED
    assert L.fp8bs_gemm_ex(*args(8, 256, 128, pr=2)) == m.ERR_INVALID_ARG
    assert L.fp8bs_gemm_ex(*args(8, 256, 128, a=None)) == m.ERR_INVALID_ARG
    assert L.fp8bs_gemm_ex(*args(8, 256, 100)) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_gemm_ex(*args(8, 256, 0)) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_gemm_ex(*args(8, 250, 128)) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_gemm_ex(*args(8, 256, 128, c=FAKE_ODD)) == m.ERR_MISALIGNED
    assert L.fp8bs_debug_gemm_stall(FAKE, FAKE, FAKE, FAKE, 8, 256, 128, FAKE, -1, -1, None) == m.ERR_INVALID_ARG
    targs = lambda tile: (FAKE, FAKE, FAKE, FAKE, 0, 8, 256, 128, FAKE, 0, 1, tile, None)  # noqa: E731
    assert L.fp8bs_gemm_tiled(*targs(-2)) == m.ERR_INVALID_ARG
    assert L.fp8bs_gemm_tiled(*targs(13)) == m.ERR_INVALID_ARG
    assert L.fp8bs_gemm_tiled(FAKE, FAKE, FAKE, FAKE, 0, 8, 256, 100, FAKE, 0, 1, 2, None) == \
        m.ERR_UNSUPPORTED_SHAPE


def test_valid_call_without_gpu_reports_cuda_or_arch(libfp8bs):
    """On a machine without a usable sm_103 device a valid call must fail
    with a status, not crash (this is what the CPU suite sees)."""
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    L, m = libfp8bs.lib(), libfp8bs
    st = L.fp8bs_quant_act_1x128(FAKE, 4, 128, 0, FAKE, FAKE, None)
    assert st in (m.ERR_CUDA, m.ERR_ARCH)


def test_maximum_sizes_rejected(libfp8bs):
    """Sizes past what the kernels index (32-bit rows and tile counts, 65535
    grid rows) are refused before anything is launched."""
    L, m = libfp8bs.lib(), libfp8bs
    big = 1 << 31
    assert L.fp8bs_quant_act_1x128(FAKE, big, 128, 0, FAKE, FAKE, None) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_quant_act_1x128(FAKE, 1 << 30, 128, 1, FAKE, FAKE, None) == \
        m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_quant_act_1x128(FAKE, 1 << 29, 1 << 20, 1, FAKE, FAKE, None) == \
        m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_quant_act_1x128(FAKE, 128, 128 * 65536, 0, FAKE, FAKE, None) == \
        m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_quant_weight_128x128(FAKE, 128 * 65536, 128, FAKE, FAKE, None, None, None) == \
        m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_requant_1x128_to_128x1(FAKE, FAKE, 1 << 30, 128, FAKE, FAKE, None) == \
        m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_requant_1x128_to_128x1(FAKE, FAKE, 128, 1 << 30, FAKE, FAKE, None) == \
        m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_quant_act_dual(FAKE, 1 << 30, 128, FAKE, FAKE, FAKE, FAKE, None) == \
        m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_quant_act_e5m6(FAKE, big, 128, FAKE, FAKE, None, None, None) == \
        m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_requant_e5m6_to_128x1(FAKE, FAKE, 1 << 30, 128, FAKE, FAKE, None) == \
        m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_quant_act_and_weight(FAKE, big, 128, FAKE, FAKE, FAKE, 128, 128, FAKE, FAKE,
                                        None) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_quant_per_tensor(FAKE, 1 << 30, 1 << 16, FAKE, FAKE, None, 0, None) == \
        m.ERR_UNSUPPORTED_SHAPE
    gargs = lambda M, N, K: (FAKE, FAKE, FAKE, FAKE, 0, M, N, K, FAKE, 0, 1, None)  # noqa: E731
    assert L.fp8bs_gemm_ex(*gargs(big, 256, 128)) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_gemm_ex(*gargs(8, big, 128)) == m.ERR_UNSUPPORTED_SHAPE
    assert L.fp8bs_gemm_ex(*gargs(8, 256, big)) == m.ERR_UNSUPPORTED_SHAPE


def test_python_binding_covers_every_declared_function(libfp8bs):
    """Every call the header declares has a typed ctypes binding."""
    missing = [n for n in _declared_functions() if n not in libfp8bs._SIGS]
    assert not missing, missing
