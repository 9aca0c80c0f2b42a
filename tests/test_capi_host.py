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


def test_backward_argument_errors_without_gpu(L):
    import blackwell_nvfp4_quantize_gb300 as fa

    n = None
    good = ctypes.c_void_p(0x6000)
    # FP8 operand quantizers: null / misaligned pointers, bad format, bad D
    for fn in (L.fp4attn_quant_mxfp8_t, L.fp4attn_quant_mxfp8_rows):
        assert fn(n, good, good, 0, 1, 1, 128, 64, n) == fa.FP4ATTN_ERR_INVALID_ARG
        assert fn(good, ctypes.c_void_p(0x6004), good, 0, 1, 1, 128, 64, n) == fa.FP4ATTN_ERR_INVALID_ARG
        assert fn(good, good, good, 2, 1, 1, 128, 64, n) == fa.FP4ATTN_ERR_INVALID_ARG
        assert fn(good, good, good, -1, 1, 1, 128, 64, n) == fa.FP4ATTN_ERR_INVALID_ARG
        assert fn(good, good, good, 1, 1, 1, 128, 96, n) == fa.FP4ATTN_ERR_UNSUPPORTED
    # sizes
    assert fa.mxfp8_rows_bytes(1, 40, 32768, 128) == (40 * 32768 * 128, 40 * 256 * 512)
    assert fa.mxfp8_rows_bytes(2, 3, 77, 64) == (6 * 77 * 64, 6 * 512)
    assert fa.bwd_workspace_bytes(2, 3, 77, 64) == (6 * 128 * 4, 6 * 128 * 4)
    with pytest.raises(fa.Fp4AttnError):
        fa.bwd_workspace_bytes(1, 1, 0, 64)
    # prep
    assert L.fp4attn_bwd_prep(good, good, good, good, n, 1, 1, 128, 64, n) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_bwd_prep(good, good, ctypes.c_void_p(0x6002), good, good, 1, 1, 128, 64, n) == \
        fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_bwd_prep(good, good, good, good, good, 1, 1, 128, 80, n) == fa.FP4ATTN_ERR_UNSUPPORTED
    # the backward: every operand struct, workspace and output is checked first
    q = fa._NVFP4(0x1000, 0x2000, 0x3000)
    f8 = fa._MXFP4(0x4000, 0x5000)
    f8_bad = fa._MXFP4(0x4000, 0)
    ops = [ctypes.byref(f8)] * 5

    def call(q1=q, k1=q, fp8=ops, nl2=good, delta=good, dq=good, dk=good, dv=good, D=64, scale=0.1):
        return L.fp4attn_bwd_directp_causal(ctypes.byref(q1), ctypes.byref(k1), *fp8, nl2, delta, dq, dk, dv, 1, 1,
                                            128, D, ctypes.c_float(scale), n)

    assert call(k1=fa._NVFP4(0x1000, 0x2000, 0)) == fa.FP4ATTN_ERR_INVALID_ARG
    for i in range(5):
        bad_ops = list(ops)
        bad_ops[i] = ctypes.byref(f8_bad)
        assert call(fp8=bad_ops) == fa.FP4ATTN_ERR_INVALID_ARG, i
    assert call(nl2=n) == fa.FP4ATTN_ERR_INVALID_ARG
    assert call(dv=ctypes.c_void_p(0x6008)) == fa.FP4ATTN_ERR_INVALID_ARG
    assert call(scale=float("nan")) == fa.FP4ATTN_ERR_INVALID_ARG
    assert call(scale=-1.0) == fa.FP4ATTN_ERR_INVALID_ARG
    assert call(D=32) == fa.FP4ATTN_ERR_UNSUPPORTED


def test_host_batch_workspace_and_argument_errors_without_gpu(L):
    import blackwell_nvfp4_quantize_gb300 as fa

    def up(x):
        return (x + 255) // 256 * 256

    # two slots of bf16 Q, K, V, O and fp32 LSE; NVFP4 Q and K (payload,
    # atoms, 4-byte g, each region 256-aligned); V payload and atoms
    for (B, H, N, D) in [(1, 40, 32768, 128), (2, 3, 77, 64)]:
        tiles = (N + 127) // 128
        slot = 4 * up(B * H * N * D * 2) + up(B * H * N * 4)
        qk = up(B * H * N * D // 2) + up(B * H * tiles * (D // 64) * 512) + 256
        for fp8pv in (False, True):
            vpay = up(B * H * D * tiles * (128 if fp8pv else 64))
            want = 2 * slot + 2 * qk + vpay + up(B * H * tiles * 512)
            for causal in (False, True):
                assert fa.host_batch_workspace_bytes(B, H, N, D, causal, fp8pv) == want
    sz = ctypes.c_size_t()
    assert L.fp4attn_fwd_host_batch_workspace_bytes(1, 1, 128, 64, 4, ctypes.byref(sz)) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_fwd_host_batch_workspace_bytes(1, 1, 128, 64, 0, None) == fa.FP4ATTN_ERR_INVALID_ARG
    assert L.fp4attn_fwd_host_batch_workspace_bytes(1, 1, 128, 80, 0, ctypes.byref(sz)) == fa.FP4ATTN_ERR_UNSUPPORTED

    # the batch call: everything is checked before a stream is made or a copy queued
    need = fa.host_batch_workspace_bytes(1, 1, 128, 64)
    h = ctypes.c_void_p(0x7000)
    arr = lambda *p: (ctypes.c_void_p * len(p))(*p)
    two = arr(h, h)
    hole = arr(h, None)

    def call(n=2, q=two, k=two, v=two, o=two, lse=two, D=64, scale=0.125, flags=0, ws=0x100000, nbytes=need):
        return L.fp4attn_fwd_host_batch(n, q, k, v, o, lse, 1, 1, 128, D, ctypes.c_float(scale), flags,
                                        ctypes.c_void_p(ws), nbytes, None)

    assert call(n=0) == fa.FP4ATTN_ERR_INVALID_ARG
    assert call(q=None) == fa.FP4ATTN_ERR_INVALID_ARG
    for name in ("q", "k", "v", "o", "lse"):
        assert call(**{name: hole}) == fa.FP4ATTN_ERR_INVALID_ARG, name
    assert call(flags=4) == fa.FP4ATTN_ERR_INVALID_ARG
    assert call(scale=float("inf")) == fa.FP4ATTN_ERR_INVALID_ARG
    assert call(scale=0.0) == fa.FP4ATTN_ERR_INVALID_ARG
    assert call(ws=0) == fa.FP4ATTN_ERR_INVALID_ARG
    assert call(ws=0x100010) == fa.FP4ATTN_ERR_INVALID_ARG          # not 256-aligned
    assert call(nbytes=need - 1) == fa.FP4ATTN_ERR_INVALID_ARG
    assert call(flags=fa.FP4ATTN_HB_FP8PV) == fa.FP4ATTN_ERR_INVALID_ARG  # the FP8 V needs more bytes
    assert call(D=96) == fa.FP4ATTN_ERR_UNSUPPORTED
