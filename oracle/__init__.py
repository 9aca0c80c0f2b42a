"""CPU oracle for the Direct-P FP4 attention forward -- TEST INFRASTRUCTURE ONLY.

Plain C (``fp4attn_oracle.c``) behind ctypes, numpy in and out.  Only the
test-suite, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline leg
may import this package; the CUDA library never does, and shares no code with
it.  What each function computes, and the reading of the method it follows,
is documented in ``fp4attn_oracle.h``.  Source of the method:
"Hardware-Aware FP4 FlashAttention-4", neuraltrendhub.com summary page,
section "What the paper found", and the paper's abstract.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp4attn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (ISO C11, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_HERE, "fp4attn_oracle.h"))
    ):
        tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared",
               "-pthread", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    build()
    lib = ctypes.CDLL(_LIB_PATH)
    u8p = ctypes.POINTER(ctypes.c_uint8)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    i32p = ctypes.POINTER(ctypes.c_int32)
    i64p = ctypes.POINTER(ctypes.c_int64)
    f32p = ctypes.POINTER(ctypes.c_float)
    f64p = ctypes.POINTER(ctypes.c_double)
    c_int, c_size = ctypes.c_int, ctypes.c_size_t
    lib.orc_e2m1_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e2m1_decode.restype = ctypes.c_double
    lib.orc_e2m1_encode.argtypes = [ctypes.c_double]
    lib.orc_e2m1_encode.restype = ctypes.c_uint8
    lib.orc_e4m3_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e4m3_decode.restype = ctypes.c_double
    lib.orc_e4m3_encode.argtypes = [ctypes.c_double]
    lib.orc_e4m3_encode.restype = ctypes.c_uint8
    lib.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
    lib.orc_e8m0_decode.restype = ctypes.c_double
    lib.orc_sf_index.argtypes = [c_size, c_int, c_int, c_int, c_int]
    lib.orc_sf_index.restype = c_size
    lib.orc_nvfp4_sf_bytes.argtypes = [c_int] * 4
    lib.orc_nvfp4_sf_bytes.restype = c_size
    lib.orc_mxfp4_sf_bytes.argtypes = [c_int] * 4
    lib.orc_mxfp4_sf_bytes.restype = c_size
    lib.orc_quant_nvfp4.argtypes = [u16p, c_int, c_int, c_int, c_int, u8p, u8p, f32p, c_int]
    lib.orc_quant_nvfp4.restype = None
    lib.orc_quant_mxfp4_v.argtypes = [u16p, c_int, c_int, c_int, c_int, u8p, u8p, c_int]
    lib.orc_quant_mxfp4_v.restype = None
    lib.orc_quant_mxfp8_v.argtypes = [u16p, c_int, c_int, c_int, c_int, u8p, u8p, c_int]
    lib.orc_quant_mxfp8_v.restype = None
    lib.orc_directp_rows.argtypes = [u8p, u8p, ctypes.c_float, u8p, u8p, ctypes.c_float, u8p, u8p,
                                     c_int, c_int, c_int, c_int, ctypes.c_float, c_int, c_int, i64p, c_int,
                                     f64p, f64p, u8p, i32p, i32p, c_int]
    lib.orc_directp_rows.restype = None
    lib.orc_directp_rows_ex.argtypes = [u8p, u8p, ctypes.c_float, u8p, u8p, ctypes.c_float, u8p, u8p,
                                        c_int, c_int, c_int, c_int, ctypes.c_float, c_int, c_int, c_int, i64p, c_int,
                                        f64p, f64p, u8p, i32p, i32p, c_int]
    lib.orc_directp_rows_ex.restype = None
    lib.orc_directp_map_row_f64.argtypes = [f64p, c_int, ctypes.c_double, c_int, u8p, i32p, i32p, f64p]
    lib.orc_directp_map_row_f64.restype = None
    lib.orc_directp_map_row.argtypes = [f32p, c_int, ctypes.c_float, c_int, u8p, i32p, i32p, f64p]
    lib.orc_directp_map_row.restype = None
    lib.orc_exact_rows.argtypes = [u16p, u16p, u16p, c_int, c_int, c_int, c_int, ctypes.c_double, c_int,
                                   i64p, c_int, f64p, f64p, c_int]
    lib.orc_exact_rows.restype = None
    _lib = lib
    return lib


def _ptr(a: np.ndarray, ctype):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def default_threads() -> int:
    return max(1, os.cpu_count() or 1)


# ---- formats -------------------------------------------------------------

def e2m1_decode(code: int) -> float:
    return _load().orc_e2m1_decode(code)


def e2m1_encode(y: float) -> int:
    return _load().orc_e2m1_encode(float(y))


def e4m3_decode(code: int) -> float:
    return _load().orc_e4m3_decode(code)


def e4m3_encode(y: float) -> int:
    return _load().orc_e4m3_encode(float(y))


def e8m0_decode(code: int) -> float:
    return _load().orc_e8m0_decode(code)


def sf_index(bh: int, n_row_tiles: int, row: int, kblock: int, kblocks_per_row: int) -> int:
    return _load().orc_sf_index(bh, n_row_tiles, row, kblock, kblocks_per_row)


def nvfp4_sf_bytes(B, H, N, D) -> int:
    return _load().orc_nvfp4_sf_bytes(B, H, N, D)


def mxfp4_sf_bytes(B, H, N, D) -> int:
    return _load().orc_mxfp4_sf_bytes(B, H, N, D)


# ---- quantizers ----------------------------------------------------------

def quant_nvfp4(x_bf16_bits: np.ndarray, threads: int | None = None):
    """x: uint16 bf16 bit patterns [B,H,N,D] -> (payload [B,H,N,D/2] u8, sf u8, g float)."""
    lib = _load()
    x = np.ascontiguousarray(x_bf16_bits, dtype=np.uint16)
    B, H, N, D = x.shape
    payload = np.zeros((B, H, N, D // 2), dtype=np.uint8)
    sf = np.zeros(lib.orc_nvfp4_sf_bytes(B, H, N, D), dtype=np.uint8)
    g = ctypes.c_float(0.0)
    lib.orc_quant_nvfp4(_ptr(x, ctypes.c_uint16), B, H, N, D, _ptr(payload, ctypes.c_uint8),
                        _ptr(sf, ctypes.c_uint8), ctypes.byref(g), threads or default_threads())
    return payload, sf, np.float32(g.value)


def quant_mxfp4_v(v_bf16_bits: np.ndarray, threads: int | None = None):
    """v: uint16 bf16 bit patterns [B,H,N,D] -> (payload_t [B,H,D,Npad/2] u8, sf u8)."""
    lib = _load()
    v = np.ascontiguousarray(v_bf16_bits, dtype=np.uint16)
    B, H, N, D = v.shape
    npad = (N + 127) // 128 * 128
    payload_t = np.zeros((B, H, D, npad // 2), dtype=np.uint8)
    sf = np.zeros(lib.orc_mxfp4_sf_bytes(B, H, N, D), dtype=np.uint8)
    lib.orc_quant_mxfp4_v(_ptr(v, ctypes.c_uint16), B, H, N, D, _ptr(payload_t, ctypes.c_uint8),
                          _ptr(sf, ctypes.c_uint8), threads or default_threads())
    return payload_t, sf


def quant_mxfp8_v(v_bf16_bits: np.ndarray, threads: int | None = None):
    """v: uint16 bf16 bit patterns [B,H,N,D] -> (payload_t [B,H,D,Npad] u8 E4M3 codes, sf u8)."""
    lib = _load()
    v = np.ascontiguousarray(v_bf16_bits, dtype=np.uint16)
    B, H, N, D = v.shape
    npad = (N + 127) // 128 * 128
    payload_t = np.zeros((B, H, D, npad), dtype=np.uint8)
    sf = np.zeros(lib.orc_mxfp4_sf_bytes(B, H, N, D), dtype=np.uint8)
    lib.orc_quant_mxfp8_v(_ptr(v, ctypes.c_uint16), B, H, N, D, _ptr(payload_t, ctypes.c_uint8),
                          _ptr(sf, ctypes.c_uint8), threads or default_threads())
    return payload_t, sf


PV_MXFP4, PV_MXFP8 = 0, 1


# ---- attention -----------------------------------------------------------

def directp_rows(q, k, v, shape, softmax_scale, rows, threads=None, want_codes=False, causal=False,
                 pv_fmt=PV_MXFP4, f64_decisions=False):
    """Direct-P forward for selected rows.

    q, k: (payload, sf, g) as returned by quant_nvfp4; v: (payload_t, sf) from
    quant_mxfp4_v (pv_fmt PV_MXFP4: E2M1 P and V) or quant_mxfp8_v (PV_MXFP8:
    E4M3 P and V).  rows: int64 flat row ids (b*H + h)*N + i.  causal: row i
    sees keys 0..i.  f64_decisions: take the mapping's decisions in fp64 (S,
    c, X and X - K_b not rounded to fp32) instead of the kernel's fp32.
    Returns dict with o [R,D] f64, lse [R] f64 and, when want_codes, codes
    [R,Npad] u8 (one code per byte), kshift [R,Npad/32] i32, m [R] i32.
    """
    lib = _load()
    B, H, N, D = shape
    npad = (N + 127) // 128 * 128
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    R = rows.shape[0]
    o = np.zeros((R, D), dtype=np.float64)
    lse = np.zeros((R,), dtype=np.float64)
    out = {"o": o, "lse": lse}
    codes = kshift = m = None
    if want_codes:
        codes = np.zeros((R, npad), dtype=np.uint8)
        kshift = np.zeros((R, npad // 32), dtype=np.int32)
        m = np.zeros((R,), dtype=np.int32)
        out.update(codes=codes, kshift=kshift, m=m)
    qp, qsf, gq = [np.ascontiguousarray(t) for t in q[:2]] + [q[2]]
    kp, ksf, gk = [np.ascontiguousarray(t) for t in k[:2]] + [k[2]]
    vp, vsf = [np.ascontiguousarray(t) for t in v]
    null_u8 = ctypes.POINTER(ctypes.c_uint8)()
    null_i32 = ctypes.POINTER(ctypes.c_int32)()
    lib.orc_directp_rows_ex(
        _ptr(qp, ctypes.c_uint8), _ptr(qsf, ctypes.c_uint8), float(gq),
        _ptr(kp, ctypes.c_uint8), _ptr(ksf, ctypes.c_uint8), float(gk),
        _ptr(vp, ctypes.c_uint8), _ptr(vsf, ctypes.c_uint8),
        B, H, N, D, float(softmax_scale), int(bool(causal)), int(pv_fmt), int(bool(f64_decisions)),
        _ptr(rows, ctypes.c_int64), R,
        _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
        _ptr(codes, ctypes.c_uint8) if want_codes else null_u8,
        _ptr(kshift, ctypes.c_int32) if want_codes else null_i32,
        _ptr(m, ctypes.c_int32) if want_codes else null_i32,
        threads or default_threads())
    return out


def directp_map_row(s: np.ndarray, c: float, pv_fmt=PV_MXFP4):
    """One row of fp32 scores -> (codes u8[n], kshift i32[ceil(n/32)], M, l); E2M1 or E4M3 codes."""
    lib = _load()
    s = np.ascontiguousarray(s, dtype=np.float32)
    n = s.shape[0]
    codes = np.zeros((n,), dtype=np.uint8)
    ks = np.zeros(((n + 31) // 32,), dtype=np.int32)
    m = ctypes.c_int32(0)
    l = ctypes.c_double(0.0)
    lib.orc_directp_map_row(_ptr(s, ctypes.c_float), n, float(c), int(pv_fmt), _ptr(codes, ctypes.c_uint8),
                            _ptr(ks, ctypes.c_int32), ctypes.byref(m), ctypes.byref(l))
    return codes, ks, int(m.value), float(l.value)


def directp_map_row_f64(s: np.ndarray, c: float, pv_fmt=PV_MXFP4):
    """One row of fp64 scores mapped with fp64 decisions -> (codes, kshift, M, l)."""
    lib = _load()
    s = np.ascontiguousarray(s, dtype=np.float64)
    n = s.shape[0]
    codes = np.zeros((n,), dtype=np.uint8)
    ks = np.zeros(((n + 31) // 32,), dtype=np.int32)
    m = ctypes.c_int32(0)
    l = ctypes.c_double(0.0)
    lib.orc_directp_map_row_f64(_ptr(s, ctypes.c_double), n, float(c), int(pv_fmt), _ptr(codes, ctypes.c_uint8),
                                _ptr(ks, ctypes.c_int32), ctypes.byref(m), ctypes.byref(l))
    return codes, ks, int(m.value), float(l.value)


def exact_rows(q_bits, k_bits, v_bits, softmax_scale, rows, threads=None, causal=False):
    """Unquantized fp64 softmax attention for selected rows of bf16 inputs
    (causal: row i sees keys 0..i)."""
    lib = _load()
    q = np.ascontiguousarray(q_bits, dtype=np.uint16)
    k = np.ascontiguousarray(k_bits, dtype=np.uint16)
    v = np.ascontiguousarray(v_bits, dtype=np.uint16)
    B, H, N, D = q.shape
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    R = rows.shape[0]
    o = np.zeros((R, D), dtype=np.float64)
    lse = np.zeros((R,), dtype=np.float64)
    lib.orc_exact_rows(_ptr(q, ctypes.c_uint16), _ptr(k, ctypes.c_uint16), _ptr(v, ctypes.c_uint16),
                       B, H, N, D, float(softmax_scale), int(bool(causal)), _ptr(rows, ctypes.c_int64), R,
                       _ptr(o, ctypes.c_double), _ptr(lse, ctypes.c_double),
                       threads or default_threads())
    return o, lse
