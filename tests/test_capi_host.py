"""Host-side checks of the C ABI: the library loads, exports every function
include/fp4attn.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fp4attn.h")


@pytest.fixture(scope="module")
def L():
    import __graft_entry__

    __graft_entry__.build()
    import blackwell_nvfp4_quantize_gb300 as fa

    return fa.lib()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fp4attn_[a-z0-9_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = declared_functions()
    assert len(names) >= 8
    for n in names:
        assert hasattr(L, n), n


def test_status_strings(L):
    import blackwell_nvfp4_quantize_gb300 as fa

    for s in range(5):
        assert len(fa.status_string(s)) > 0
    assert fa.status_string(99) == "unknown status"


def test_size_queries(L):
    import blackwell_nvfp4_quantize_gb300 as fa

    assert fa.nvfp4_bytes(1, 40, 32768, 128) == (40 * 32768 * 64, 40 * 256 * 2 * 512)
    assert fa.mxfp4_v_bytes(1, 40, 32768, 128) == (40 * 128 * 32768 // 2, 40 * 256 * 512)
    assert fa.nvfp4_bytes(2, 3, 77, 64) == (2 * 3 * 77 * 32, 6 * 1 * 512)
    assert fa.mxfp4_v_bytes(2, 3, 77, 64) == (6 * 64 * 64, 6 * 512)
    with pytest.raises(fa.Fp4AttnError) as e:
        fa.nvfp4_bytes(1, 1, 128, 96)
    assert e.value.status == fa.FP4ATTN_ERR_UNSUPPORTED
    with pytest.raises(fa.Fp4AttnError) as e:
        fa.nvfp4_bytes(0, 1, 128, 64)
    assert e.value.status == fa.FP4ATTN_ERR_INVALID_ARG


def test_argument_errors_without_gpu(L):
    import blackwell_nvfp4_quantize_gb300 as fa

    n = None
    assert L.fp4attn_quant_qk_nvfp4(n, n, n, n, 1, 1, 128, 64, n) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_quant_qk_nvfp4(n, n, n, n, 1, 1, 128, 80, n) == fa.FP4ATTN_ERR_UNSUPPORTED
    assert L.fp4attn_quant_v_mxfp4(n, n, n, 1, 1, 128, 64, n) == fa.FP4ATTN_ERR_INVALID_ARG
    # misaligned pointers are rejected
    assert L.fp4attn_quant_v_mxfp4(ctypes.c_void_p(0x1001), ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000),
                                   1, 1, 128, 64, n) == fa.FP4ATTN_ERR_INVALID_ARG
    q = fa._NVFP4(0x1000, 0x2000, 0x3000)
    v = fa._MXFP4(0x4000, 0x5000)
    good = ctypes.c_void_p(0x6000)
    args = (ctypes.byref(q), ctypes.byref(q), ctypes.byref(v), good, good, 1, 1, 128, 64)
    assert L.fp4attn_fwd_directp(*args, ctypes.c_float(float("nan")), n) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_fwd_directp(*args, ctypes.c_float(-1.0), n) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_fwd_directp(ctypes.byref(q), ctypes.byref(q), ctypes.byref(v), good, good, 1, 1, 128, 32,
                                 ctypes.c_float(0.1), n) == fa.FP4ATTN_ERR_UNSUPPORTED
    bad = fa._NVFP4(0x1000, 0, 0x3000)
    assert L.fp4attn_fwd_directp(ctypes.byref(bad), ctypes.byref(q), ctypes.byref(v), good, good, 1, 1, 128, 64,
                                 ctypes.c_float(0.1), n) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_debug_dump_p(*args, ctypes.c_float(0.1), 0, 0, 100, 64, good, good, good, n) == \
        fa.FP4ATTN_ERR_INVALID_ARG  # rows beyond N
    assert L.fp4attn_fwd_directp(ctypes.byref(q), ctypes.byref(q), ctypes.byref(v), good, good, 300, 300, 128, 64,
                                 ctypes.c_float(0.1), n) == fa.FP4ATTN_ERR_UNSUPPORTED  # B*H > 65535


def test_no_torch_types_in_header():
    src = open(HEADER).read()
    assert "torch" not in src and "at::" not in src and "Tensor" not in src


def test_causal_argument_errors_without_gpu(L):
    import blackwell_nvfp4_quantize_gb300 as fa

    n = None
    q = fa._NVFP4(0x1000, 0x2000, 0x3000)
    v = fa._MXFP4(0x4000, 0x5000)
    good = ctypes.c_void_p(0x6000)
    args = (ctypes.byref(q), ctypes.byref(q), ctypes.byref(v), good, good, 1, 1, 128, 64)
    assert L.fp4attn_fwd_directp_causal(*args, ctypes.c_float(float("inf")), n) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_fwd_directp_causal(ctypes.byref(q), ctypes.byref(q), ctypes.byref(v), good, good, 1, 1, 128,
                                        48, ctypes.c_float(0.1), n) == fa.FP4ATTN_ERR_UNSUPPORTED
    assert L.fp4attn_debug_dump_p_causal(*args, ctypes.c_float(0.1), 0, 1, 0, 8, good, good, good, n) == \
        fa.FP4ATTN_ERR_INVALID_ARG  # h beyond H
    # the one-call training forward checks every argument before launching
    assert L.fp4attn_fwd_directp_causal_save(n, good, good, ctypes.byref(q), ctypes.byref(q), ctypes.byref(v),
                                             good, good, 1, 1, 128, 64, ctypes.c_float(0.1), n) == \
        fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_fwd_directp_causal_save(ctypes.c_void_p(0x7001), good, good, ctypes.byref(q), ctypes.byref(q),
                                             ctypes.byref(v), good, good, 1, 1, 128, 64, ctypes.c_float(0.1), n) == \
        fa.FP4ATTN_ERR_INVALID_ARG
    bad = fa._NVFP4(0x1000, 0x2000, 0)
    assert L.fp4attn_fwd_directp_causal_save(good, good, good, ctypes.byref(q), ctypes.byref(bad), ctypes.byref(v),
                                             good, good, 1, 1, 128, 64, ctypes.c_float(0.1), n) == \
        fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_fwd_directp_causal_save(good, good, good, ctypes.byref(q), ctypes.byref(q), ctypes.byref(v),
                                             good, good, 1, 1, 128, 64, ctypes.c_float(0.0), n) == \
        fa.FP4ATTN_ERR_INVALID_ARG


def test_fp8pv_argument_errors_without_gpu(L):
    import blackwell_nvfp4_quantize_gb300 as fa

    n = None
    q = fa._NVFP4(0x1000, 0x2000, 0x3000)
    v = fa._MXFP4(0x4000, 0x5000)
    good = ctypes.c_void_p(0x6000)
    assert fa.mxfp8_v_bytes(1, 40, 32768, 128) == (40 * 128 * 32768, 40 * 256 * 512)
    assert fa.mxfp8_v_bytes(2, 3, 77, 64) == (6 * 64 * 128, 6 * 512)
    assert L.fp4attn_quant_v_mxfp8(n, good, good, 1, 1, 128, 64, n) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_quant_v_mxfp8(good, good, good, 1, 1, 128, 96, n) == fa.FP4ATTN_ERR_UNSUPPORTED
    args = (ctypes.byref(q), ctypes.byref(q), ctypes.byref(v), good, good, 1, 1, 128, 64)
    assert L.fp4attn_fwd_directp_fp8pv(*args, ctypes.c_float(0.0), 0, n) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_fwd_directp_fp8pv(ctypes.byref(q), ctypes.byref(q), None, good, good, 1, 1, 128, 64,
                                       ctypes.c_float(0.1), 1, n) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_debug_dump_p_fp8pv(*args, ctypes.c_float(0.1), 0, 0, 0, 100, 64, good, good, good, n) == \
        fa.FP4ATTN_ERR_INVALID_ARG  # rows beyond N


def test_mma_peak_argument_errors(L):
    import blackwell_nvfp4_quantize_gb300 as fa

    assert L.fp4attn_debug_mma_peak(3, 16, None) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_debug_mma_peak(-1, 16, None) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_debug_mma_peak(0, 0, None) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_debug_mma_peak(1, (1 << 26) + 1, None) == fa.FP4ATTN_ERR_INVALID_ARG


def test_noalloc_debug_argument_errors(L):
    import blackwell_nvfp4_quantize_gb300 as fa

    assert L.fp4attn_debug_noalloc_timeout(None, 16, 100, None) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_debug_noalloc_timeout(ctypes.c_void_p(0x1008), 16, 100, None) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_debug_noalloc_timeout(ctypes.c_void_p(0x1000), 0, 100, None) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_debug_noalloc_timeout(ctypes.c_void_p(0x1000), 16, 0, None) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_debug_status_word_exists(None) == fa.FP4ATTN_ERR_INVALID_ARG
