"""Direct-P FP4 attention forward for GB300 (sm_103a).

Thin Python binding over the C ABI of ``libfp4attn.so`` (declared in
``include/fp4attn.h``).  PyTorch supplies device memory and streams only; every
step of the computation runs in the library's CUDA kernels.  The binding
raises if the library has not been built -- there is no fallback.

Method: "Hardware-Aware FP4 FlashAttention-4" (Direct-P for noncausal
inference): NVFP4 Q/K, MXFP4 V along keys, scores mapped directly to MXFP4
E2M1 probability codes, denominator from the same rounded probabilities, O
and LSE as outputs; its causal training forward, which keeps the quantized
Q/K and the LSE for a backward pass; and the FP8 P/V variant (E4M3
probability codes, MXFP8 V) kept for training.
"""
from __future__ import annotations

import ctypes
import math
import os
from dataclasses import dataclass

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfp4attn.so")

FP4ATTN_OK = 0
FP4ATTN_ERR_INVALID_ARG = 1
FP4ATTN_ERR_UNSUPPORTED = 2
FP4ATTN_ERR_CUDA = 3
FP4ATTN_ERR_TIMEOUT = 4

_lib = None


class Fp4AttnError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (what, status_string(status), status))


class _NVFP4(ctypes.Structure):
    _fields_ = [("payload", ctypes.c_void_p), ("sf", ctypes.c_void_p), ("g", ctypes.c_void_p)]


class _MXFP4(ctypes.Structure):
    _fields_ = [("payload_t", ctypes.c_void_p), ("sf", ctypes.c_void_p)]


def lib():
    """The loaded C library (ctypes.CDLL).  Raises if it is not built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError("libfp4attn.so is not built (%s); run __graft_entry__.build() or "
                           "python -m blackwell_nvfp4_quantize_gb300.build" % LIB_PATH)
    L = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fp4attn_status_string.argtypes = [i]
    L.fp4attn_status_string.restype = ctypes.c_char_p
    L.fp4attn_nvfp4_bytes.argtypes = [i, i, i, i, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    L.fp4attn_mxfp4_v_bytes.argtypes = [i, i, i, i, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    L.fp4attn_quant_qk_nvfp4.argtypes = [vp, vp, vp, vp, i, i, i, i, vp]
    L.fp4attn_quant_v_mxfp4.argtypes = [vp, vp, vp, i, i, i, i, vp]
    L.fp4attn_fwd_directp.argtypes = [ctypes.POINTER(_NVFP4), ctypes.POINTER(_NVFP4), ctypes.POINTER(_MXFP4),
                                      vp, vp, i, i, i, i, f, vp]
    L.fp4attn_debug_dump_p.argtypes = [ctypes.POINTER(_NVFP4), ctypes.POINTER(_NVFP4), ctypes.POINTER(_MXFP4),
                                       vp, vp, i, i, i, i, f, i, i, i, i, vp, vp, vp, vp]
    L.fp4attn_device_status.argtypes = [vp]
    L.fp4attn_fwd_directp_noalloc.argtypes = [ctypes.POINTER(_NVFP4), ctypes.POINTER(_NVFP4),
                                              ctypes.POINTER(_MXFP4), vp, vp, i, i, i, i, f, vp]
    L.fp4attn_debug_cvt_transitions.argtypes = [i, ctypes.c_uint32, ctypes.c_uint32, vp, i, vp, vp]
    L.fp4attn_fwd_directp_causal.argtypes = L.fp4attn_fwd_directp.argtypes
    L.fp4attn_debug_dump_p_causal.argtypes = L.fp4attn_debug_dump_p.argtypes
    L.fp4attn_fwd_directp_causal_save.argtypes = [vp, vp, vp, ctypes.POINTER(_NVFP4), ctypes.POINTER(_NVFP4),
                                                  ctypes.POINTER(_MXFP4), vp, vp, i, i, i, i, f, vp]
    L.fp4attn_mxfp8_v_bytes.argtypes = [i, i, i, i, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    L.fp4attn_quant_v_mxfp8.argtypes = [vp, vp, vp, i, i, i, i, vp]
    L.fp4attn_fwd_directp_fp8pv.argtypes = [ctypes.POINTER(_NVFP4), ctypes.POINTER(_NVFP4), ctypes.POINTER(_MXFP4),
                                            vp, vp, i, i, i, i, f, i, vp]
    L.fp4attn_debug_dump_p_fp8pv.argtypes = [ctypes.POINTER(_NVFP4), ctypes.POINTER(_NVFP4),
                                             ctypes.POINTER(_MXFP4), vp, vp, i, i, i, i, f, i, i, i, i, i, vp, vp,
                                             vp, vp]
    L.fp4attn_debug_wait_timeout.argtypes = [i, vp]
    L.fp4attn_debug_mma_peak.argtypes = [i, i, vp]
    L.fp4attn_debug_noalloc_timeout.argtypes = [vp, ctypes.c_longlong, i, vp]
    L.fp4attn_debug_status_word_exists.argtypes = [ctypes.POINTER(i)]
    L.fp4attn_quant_mxfp8_t.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
    L.fp4attn_quant_mxfp8_rows.argtypes = [vp, vp, vp, i, i, i, i, i, vp]
    L.fp4attn_mxfp8_rows_bytes.argtypes = [i, i, i, i, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    L.fp4attn_bwd_workspace_bytes.argtypes = [i, i, i, i, ctypes.POINTER(sz), ctypes.POINTER(sz)]
    L.fp4attn_bwd_prep.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, vp]
    L.fp4attn_bwd_directp_causal.argtypes = [ctypes.POINTER(_NVFP4), ctypes.POINTER(_NVFP4)] + \
        [ctypes.POINTER(_MXFP4)] * 5 + [vp, vp, vp, vp, vp, i, i, i, i, ctypes.c_float, vp]
    L.fp4attn_fwd_host_batch_workspace_bytes.argtypes = [i, i, i, i, i, ctypes.POINTER(sz)]
    L.fp4attn_fwd_host_batch.argtypes = [i, ctypes.POINTER(vp), ctypes.POINTER(vp), ctypes.POINTER(vp),
                                         ctypes.POINTER(vp), ctypes.POINTER(vp), i, i, i, i, ctypes.c_float, i,
                                         vp, sz, vp]
    for name in ("fp4attn_debug_wait_timeout", "fp4attn_debug_mma_peak", "fp4attn_debug_noalloc_timeout",
                 "fp4attn_debug_status_word_exists", "fp4attn_mxfp8_v_bytes", "fp4attn_quant_v_mxfp8", "fp4attn_fwd_directp_fp8pv",
                 "fp4attn_debug_dump_p_fp8pv", "fp4attn_fwd_directp_causal", "fp4attn_debug_dump_p_causal", "fp4attn_fwd_directp_causal_save",
                 "fp4attn_fwd_directp_noalloc", "fp4attn_debug_cvt_transitions", "fp4attn_nvfp4_bytes", "fp4attn_mxfp4_v_bytes", "fp4attn_quant_qk_nvfp4",
                 "fp4attn_quant_v_mxfp4", "fp4attn_fwd_directp", "fp4attn_debug_dump_p",
                 "fp4attn_device_status"):
        getattr(L, name).restype = i
    _lib = L
    return L


def status_string(status: int) -> str:
    return lib().fp4attn_status_string(status).decode()


def _check(status: int, what: str):
    if status != FP4ATTN_OK:
        raise Fp4AttnError(status, what)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


@dataclass
class NVFP4Tensor:
    """Q or K in NVFP4: payload [B,H,N,D/2] u8, scale atoms u8, g (1 fp32), on one device."""
    payload: torch.Tensor
    sf: torch.Tensor
    g: torch.Tensor
    shape: tuple

    def _c(self):
        return _NVFP4(self.payload.data_ptr(), self.sf.data_ptr(), self.g.data_ptr())


@dataclass
class MXFP4Tensor:
    """V in MXFP4 along keys: payload_t [B,H,D,Npad/2] u8, scale atoms u8."""
    payload_t: torch.Tensor
    sf: torch.Tensor
    shape: tuple

    def _c(self):
        return _MXFP4(self.payload_t.data_ptr(), self.sf.data_ptr())


@dataclass
class MXFP8Tensor:
    """V in MXFP8 along keys (FP8 P/V variant): payload_t [B,H,D,Npad] u8 E4M3 codes, scale atoms u8."""
    payload_t: torch.Tensor
    sf: torch.Tensor
    shape: tuple

    def _c(self):  # same two pointers as the MXFP4 struct
        return _MXFP4(self.payload_t.data_ptr(), self.sf.data_ptr())


def nvfp4_bytes(B, H, N, D):
    p, s = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().fp4attn_nvfp4_bytes(B, H, N, D, ctypes.byref(p), ctypes.byref(s)), "fp4attn_nvfp4_bytes")
    return p.value, s.value


def mxfp4_v_bytes(B, H, N, D):
    p, s = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().fp4attn_mxfp4_v_bytes(B, H, N, D, ctypes.byref(p), ctypes.byref(s)), "fp4attn_mxfp4_v_bytes")
    return p.value, s.value


def mxfp8_v_bytes(B, H, N, D):
    p, s = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().fp4attn_mxfp8_v_bytes(B, H, N, D, ctypes.byref(p), ctypes.byref(s)), "fp4attn_mxfp8_v_bytes")
    return p.value, s.value


def _check_input(x: torch.Tensor, name: str):
    if not (x.is_cuda and x.dtype == torch.bfloat16 and x.dim() == 4 and x.is_contiguous()):
        raise ValueError("%s must be a contiguous CUDA bf16 tensor [B,H,N,D]" % name)


# The C ABI takes plain pointers and cannot see buffer sizes: everything a
# kernel will read or write is checked here, before the call, so that a
# mismatched buffer raises instead of being read or written past its end.

def _check_buffer(t: torch.Tensor, name: str, dtype, numel: int, device):
    if not isinstance(t, torch.Tensor) or t.dtype != dtype or t.numel() != numel or not t.is_contiguous():
        raise ValueError("%s must be a contiguous %s tensor of %d elements" % (name, dtype, numel))
    if t.device != device:
        raise ValueError("%s is on %s, the operands on %s" % (name, t.device, device))


def _check_quantized(t, name: str, shape, kind):
    """t is a kind (NVFP4Tensor / MXFP4Tensor / MXFP8Tensor) of the given
    shape whose buffers hold exactly the bytes the library reads."""
    if not isinstance(t, kind):
        raise ValueError("%s must be a %s" % (name, kind.__name__))
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s has shape %s, expected %s" % (name, tuple(t.shape), tuple(shape)))
    B, H, N, D = shape
    if kind is NVFP4Tensor:
        pb, sb = nvfp4_bytes(B, H, N, D)
        dev = t.payload.device
        _check_buffer(t.payload, name + ".payload", torch.uint8, pb, dev)
        _check_buffer(t.g, name + ".g", torch.float32, 1, dev)
    else:
        pb, sb = (mxfp4_v_bytes if kind is MXFP4Tensor else mxfp8_v_bytes)(B, H, N, D)
        dev = t.payload_t.device
        _check_buffer(t.payload_t, name + ".payload_t", torch.uint8, pb, dev)
    _check_buffer(t.sf, name + ".sf", torch.uint8, sb, dev)
    return dev


def _check_fwd_args(q, k, v, v_kind, o, lse):
    """Operands of one shape on one device; O bf16 [B,H,N,D] and LSE fp32
    [B,H,N] (when given) on that device."""
    if not isinstance(q, NVFP4Tensor):
        raise ValueError("q must be an NVFP4Tensor")
    shape = tuple(q.shape)
    dev = _check_quantized(q, "q", shape, NVFP4Tensor)
    for t, name, kind in ((k, "k", NVFP4Tensor), (v, "v", v_kind)):
        if _check_quantized(t, name, shape, kind) != dev:
            raise ValueError("q, k and v must be on one device")
    B, H, N, D = shape
    if o is not None:
        _check_buffer(o, "o", torch.bfloat16, B * H * N * D, dev)
    if lse is not None:
        _check_buffer(lse, "lse", torch.float32, B * H * N, dev)
    if dev.type != "cuda":
        raise ValueError("the operands must be CUDA tensors")


def empty_nvfp4(shape, device) -> NVFP4Tensor:
    B, H, N, D = shape
    pb, sb = nvfp4_bytes(B, H, N, D)
    return NVFP4Tensor(torch.empty((B, H, N, D // 2), dtype=torch.uint8, device=device),
                       torch.empty((sb,), dtype=torch.uint8, device=device),
                       torch.empty((1,), dtype=torch.float32, device=device), tuple(shape))


def empty_mxfp4(shape, device) -> MXFP4Tensor:
    B, H, N, D = shape
    pb, sb = mxfp4_v_bytes(B, H, N, D)
    npad = (N + 127) // 128 * 128
    return MXFP4Tensor(torch.empty((B, H, D, npad // 2), dtype=torch.uint8, device=device),
                       torch.empty((sb,), dtype=torch.uint8, device=device), tuple(shape))


def empty_mxfp8(shape, device) -> MXFP8Tensor:
    B, H, N, D = shape
    pb, sb = mxfp8_v_bytes(B, H, N, D)
    npad = (N + 127) // 128 * 128
    return MXFP8Tensor(torch.empty((B, H, D, npad), dtype=torch.uint8, device=device),
                       torch.empty((sb,), dtype=torch.uint8, device=device), tuple(shape))


def quant_qk_nvfp4(x: torch.Tensor, out: NVFP4Tensor | None = None, stream=None) -> NVFP4Tensor:
    """fp4attn_quant_qk_nvfp4 on a CUDA bf16 [B,H,N,D] tensor."""
    _check_input(x, "x")
    B, H, N, D = x.shape
    out = out or empty_nvfp4(x.shape, x.device)
    if _check_quantized(out, "out", x.shape, NVFP4Tensor) != x.device:
        raise ValueError("out must be on the device of x")
    _check(lib().fp4attn_quant_qk_nvfp4(_ptr(x), _ptr(out.payload), _ptr(out.sf), _ptr(out.g),
                                        B, H, N, D, ctypes.c_void_p(_stream(stream))), "fp4attn_quant_qk_nvfp4")
    return out


def quant_v_mxfp4(v: torch.Tensor, out: MXFP4Tensor | None = None, stream=None) -> MXFP4Tensor:
    """fp4attn_quant_v_mxfp4 on a CUDA bf16 [B,H,N,D] tensor."""
    _check_input(v, "v")
    B, H, N, D = v.shape
    out = out or empty_mxfp4(v.shape, v.device)
    if _check_quantized(out, "out", v.shape, MXFP4Tensor) != v.device:
        raise ValueError("out must be on the device of v")
    _check(lib().fp4attn_quant_v_mxfp4(_ptr(v), _ptr(out.payload_t), _ptr(out.sf), B, H, N, D,
                                       ctypes.c_void_p(_stream(stream))), "fp4attn_quant_v_mxfp4")
    return out


def quant_v_mxfp8(v: torch.Tensor, out: MXFP8Tensor | None = None, stream=None) -> MXFP8Tensor:
    """fp4attn_quant_v_mxfp8 on a CUDA bf16 [B,H,N,D] tensor (FP8 P/V variant)."""
    _check_input(v, "v")
    B, H, N, D = v.shape
    out = out or empty_mxfp8(v.shape, v.device)
    if _check_quantized(out, "out", v.shape, MXFP8Tensor) != v.device:
        raise ValueError("out must be on the device of v")
    _check(lib().fp4attn_quant_v_mxfp8(_ptr(v), _ptr(out.payload_t), _ptr(out.sf), B, H, N, D,
                                       ctypes.c_void_p(_stream(stream))), "fp4attn_quant_v_mxfp8")
    return out


def fwd_directp_fp8pv(q: NVFP4Tensor, k: NVFP4Tensor, v: MXFP8Tensor, softmax_scale: float | None = None,
                      causal: bool = False, o: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                      stream=None):
    """fp4attn_fwd_directp_fp8pv: Direct-P with E4M3 probability codes and MXFP8 V; (O, LSE)."""
    _check_fwd_args(q, k, v, MXFP8Tensor, o, lse)
    B, H, N, D = q.shape
    dev = q.payload.device
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    o = o if o is not None else torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev)
    lse = lse if lse is not None else torch.empty((B, H, N), dtype=torch.float32, device=dev)
    qc, kc, vc = q._c(), k._c(), v._c()
    _check(lib().fp4attn_fwd_directp_fp8pv(ctypes.byref(qc), ctypes.byref(kc), ctypes.byref(vc), _ptr(o),
                                           _ptr(lse), B, H, N, D, float(softmax_scale), int(bool(causal)),
                                           ctypes.c_void_p(_stream(stream))), "fp4attn_fwd_directp_fp8pv")
    return o, lse


def _fwd(name, q, k, v, softmax_scale, o, lse, stream):
    _check_fwd_args(q, k, v, MXFP4Tensor, o, lse)
    B, H, N, D = q.shape
    dev = q.payload.device
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    o = o if o is not None else torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev)
    lse = lse if lse is not None else torch.empty((B, H, N), dtype=torch.float32, device=dev)
    qc, kc, vc = q._c(), k._c(), v._c()
    _check(getattr(lib(), name)(ctypes.byref(qc), ctypes.byref(kc), ctypes.byref(vc), _ptr(o), _ptr(lse),
                                B, H, N, D, float(softmax_scale), ctypes.c_void_p(_stream(stream))), name)
    return o, lse


def fwd_directp(q: NVFP4Tensor, k: NVFP4Tensor, v: MXFP4Tensor, softmax_scale: float | None = None,
                o: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """fp4attn_fwd_directp: returns (O bf16 [B,H,N,D], LSE fp32 [B,H,N])."""
    return _fwd("fp4attn_fwd_directp", q, k, v, softmax_scale, o, lse, stream)


def fwd_directp_causal(q: NVFP4Tensor, k: NVFP4Tensor, v: MXFP4Tensor, softmax_scale: float | None = None,
                       o: torch.Tensor | None = None, lse: torch.Tensor | None = None, stream=None):
    """fp4attn_fwd_directp_causal (query i sees keys 0..i): returns (O, LSE)."""
    return _fwd("fp4attn_fwd_directp_causal", q, k, v, softmax_scale, o, lse, stream)


def fwd_directp_causal_save(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, softmax_scale: float | None = None,
                            q_saved: NVFP4Tensor | None = None, k_saved: NVFP4Tensor | None = None,
                            v_quant: MXFP4Tensor | None = None, o: torch.Tensor | None = None,
                            lse: torch.Tensor | None = None, stream=None):
    """fp4attn_fwd_directp_causal_save: quantizes Q, K, V and runs the causal
    forward in one call.  Returns (O, LSE, q_saved, k_saved, v_quant); the
    quantized Q/K and the LSE are what a backward pass reconstructs P from."""
    for x, name in ((q, "q"), (k, "k"), (v, "v")):
        _check_input(x, name)
    if not (q.shape == k.shape == v.shape and q.device == k.device == v.device):
        raise ValueError("q, k and v must have one shape and one device")
    B, H, N, D = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    q_saved = q_saved or empty_nvfp4(q.shape, q.device)
    k_saved = k_saved or empty_nvfp4(k.shape, k.device)
    v_quant = v_quant or empty_mxfp4(v.shape, v.device)
    o = o if o is not None else torch.empty((B, H, N, D), dtype=torch.bfloat16, device=q.device)
    lse = lse if lse is not None else torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    for t, name, kind in ((q_saved, "q_saved", NVFP4Tensor), (k_saved, "k_saved", NVFP4Tensor),
                          (v_quant, "v_quant", MXFP4Tensor)):
        if _check_quantized(t, name, q.shape, kind) != q.device:
            raise ValueError("%s must be on the device of q" % name)
    _check_buffer(o, "o", torch.bfloat16, B * H * N * D, q.device)
    _check_buffer(lse, "lse", torch.float32, B * H * N, q.device)
    qc, kc, vc = q_saved._c(), k_saved._c(), v_quant._c()
    _check(lib().fp4attn_fwd_directp_causal_save(_ptr(q), _ptr(k), _ptr(v), ctypes.byref(qc), ctypes.byref(kc),
                                                 ctypes.byref(vc), _ptr(o), _ptr(lse), B, H, N, D,
                                                 float(softmax_scale), ctypes.c_void_p(_stream(stream))),
           "fp4attn_fwd_directp_causal_save")
    return o, lse, q_saved, k_saved, v_quant


def fwd_directp_noalloc(q: NVFP4Tensor, k: NVFP4Tensor, v: MXFP4Tensor, o: torch.Tensor, lse: torch.Tensor,
                        softmax_scale: float | None = None, stream=None):
    """fp4attn_fwd_directp_noalloc: the same forward with no device allocation
    anywhere on its path; the caller provides O and LSE.  A bounded wait that
    gives up shows as NaN in every LSE entry instead of a status code."""
    if o is None or lse is None:
        raise ValueError("fwd_directp_noalloc writes into caller-provided o and lse: both are required")
    _check_fwd_args(q, k, v, MXFP4Tensor, o, lse)
    B, H, N, D = q.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    qc, kc, vc = q._c(), k._c(), v._c()
    _check(lib().fp4attn_fwd_directp_noalloc(ctypes.byref(qc), ctypes.byref(kc), ctypes.byref(vc), _ptr(o),
                                             _ptr(lse), B, H, N, D, float(softmax_scale),
                                             ctypes.c_void_p(_stream(stream))), "fp4attn_fwd_directp_noalloc")
    return o, lse


def debug_dump_p(q: NVFP4Tensor, k: NVFP4Tensor, v, b: int, h: int, row0: int, nrows: int,
                 softmax_scale: float | None = None, stream=None, causal: bool = False):
    """fp4attn_debug_dump_p (or fp4attn_debug_dump_p_causal; with an MXFP8Tensor v,
    fp4attn_debug_dump_p_fp8pv): (O, LSE, codes [nrows, Npad/2] u8 -- [nrows, Npad] E4M3 bytes
    for FP8 P/V --, kshift [nrows, Npad/32] i32, O of the dumped rows in fp32 [nrows, D])."""
    B, H, N, D = q.shape
    dev = q.payload.device
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    npad = (N + 127) // 128 * 128
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    fp8 = isinstance(v, MXFP8Tensor)
    _check_fwd_args(q, k, v, MXFP8Tensor if fp8 else MXFP4Tensor, None, None)
    if not (0 <= b < B and 0 <= h < H and 0 <= row0 and nrows > 0 and row0 + nrows <= N):
        raise ValueError("dump rows (b=%d, h=%d, rows %d..%d) outside [B=%d, H=%d, N=%d]"
                         % (b, h, row0, row0 + nrows, B, H, N))
    codes = torch.zeros((nrows, npad if fp8 else npad // 2), dtype=torch.uint8, device=dev)
    kshift = torch.zeros((nrows, npad // 32), dtype=torch.int32, device=dev)
    o32 = torch.zeros((nrows, D), dtype=torch.float32, device=dev)
    qc, kc, vc = q._c(), k._c(), v._c()
    if fp8:
        _check(lib().fp4attn_debug_dump_p_fp8pv(ctypes.byref(qc), ctypes.byref(kc), ctypes.byref(vc), _ptr(o),
                                                _ptr(lse), B, H, N, D, float(softmax_scale), int(bool(causal)), b, h,
                                                row0, nrows, _ptr(codes), _ptr(kshift), _ptr(o32),
                                                ctypes.c_void_p(_stream(stream))), "fp4attn_debug_dump_p_fp8pv")
        return o, lse, codes, kshift, o32
    name = "fp4attn_debug_dump_p_causal" if causal else "fp4attn_debug_dump_p"
    _check(getattr(lib(), name)(ctypes.byref(qc), ctypes.byref(kc), ctypes.byref(vc), _ptr(o), _ptr(lse),
                                B, H, N, D, float(softmax_scale), b, h, row0, nrows, _ptr(codes),
                                _ptr(kshift), _ptr(o32), ctypes.c_void_p(_stream(stream))), name)
    return o, lse, codes, kshift, o32


def device_status(stream=None) -> int:
    """fp4attn_device_status: FP4ATTN_OK, or FP4ATTN_ERR_TIMEOUT if a bounded wait gave up."""
    return lib().fp4attn_device_status(ctypes.c_void_p(_stream(stream)))


def debug_noalloc_timeout(lse: torch.Tensor, limit_us: int, stream=None) -> None:
    """fp4attn_debug_noalloc_timeout: a bounded wait on the allocation-free
    entry point's status word gives up after limit_us, and its report kernel
    sets every entry of lse (a CUDA fp32 tensor) to NaN."""
    if not (isinstance(lse, torch.Tensor) and lse.is_cuda and lse.dtype == torch.float32 and lse.is_contiguous()):
        raise ValueError("lse must be a contiguous CUDA fp32 tensor")
    _check(lib().fp4attn_debug_noalloc_timeout(_ptr(lse), lse.numel(), int(limit_us), ctypes.c_void_p(_stream(stream))),
           "fp4attn_debug_noalloc_timeout")


def debug_status_word_exists() -> bool:
    """fp4attn_debug_status_word_exists: has the library created its
    per-device status block on the current device?"""
    e = ctypes.c_int(-1)
    _check(lib().fp4attn_debug_status_word_exists(ctypes.byref(e)), "fp4attn_debug_status_word_exists")
    return bool(e.value)


def debug_wait_timeout(limit_us: int, stream=None) -> None:
    """fp4attn_debug_wait_timeout: a bounded wait that nothing completes gives up after limit_us."""
    _check(lib().fp4attn_debug_wait_timeout(int(limit_us), ctypes.c_void_p(_stream(stream))),
           "fp4attn_debug_wait_timeout")


MMA_PEAK_KINDS = {"nvf4": 0, "mxf4": 1, "mxf8": 2}


def debug_mma_peak(kind: str, iters: int = 1 << 20, launches: int = 3, stream=None):
    """fp4attn_debug_mma_peak: dense TFLOP/s of the block-scaled product `kind`
    ("nvf4": QK^T form, "mxf4": PV form, "mxf8": FP8 PV form), timed with CUDA
    events over `launches` launches after one warm-up launch."""
    st = torch.cuda.current_stream() if stream is None else stream
    code = MMA_PEAK_KINDS[kind]
    _check(lib().fp4attn_debug_mma_peak(code, int(iters), ctypes.c_void_p(_stream(st))), "fp4attn_debug_mma_peak")
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(st)
    for _ in range(launches):
        _check(lib().fp4attn_debug_mma_peak(code, int(iters), ctypes.c_void_p(_stream(st))),
               "fp4attn_debug_mma_peak")
    e1.record(st)
    e1.synchronize()
    ms = e0.elapsed_time(e1) / launches
    sms = torch.cuda.get_device_properties(torch.cuda.current_device()).multi_processor_count
    return sms * float(iters) * 2.0 * 128 ** 3 / (ms * 1e-3) / 1e12


def debug_cvt_transitions(fmt: int, lo: int, hi: int, capacity: int = 4096, stream=None):
    """fp4attn_debug_cvt_transitions: sorted list of (bit pattern, code) where the conversion changes."""
    pairs = torch.zeros((capacity, 2), dtype=torch.int64).to(torch.int32).cuda()
    count = torch.zeros((1,), dtype=torch.int32, device=pairs.device)
    _check(lib().fp4attn_debug_cvt_transitions(fmt, lo, hi, _ptr(pairs), capacity, _ptr(count),
                                               ctypes.c_void_p(_stream(stream))), "fp4attn_debug_cvt_transitions")
    n = int(count.item())
    if n > capacity:
        raise RuntimeError("more transitions (%d) than capacity (%d)" % (n, capacity))
    out = pairs[:n].cpu().numpy().view("uint32")
    return sorted((int(a), int(b)) for a, b in out)


def attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, softmax_scale: float | None = None, stream=None,
              causal: bool = False, fp8pv: bool = False):
    """Quantize Q, K (NVFP4) and V (MXFP4, or MXFP8 with fp8pv) and run the Direct-P forward: (O, LSE)."""
    qq = quant_qk_nvfp4(q, stream=stream)
    kq = quant_qk_nvfp4(k, stream=stream)
    if fp8pv:
        return fwd_directp_fp8pv(qq, kq, quant_v_mxfp8(v, stream=stream), softmax_scale, causal=causal, stream=stream)
    vq = quant_v_mxfp4(v, stream=stream)
    fwd = fwd_directp_causal if causal else fwd_directp
    return fwd(qq, kq, vq, softmax_scale, stream=stream)


# ---- forwards from host memory -------------------------------------------------

FP4ATTN_HB_CAUSAL, FP4ATTN_HB_FP8PV = 1, 2


def _hb_flags(causal: bool, fp8pv: bool) -> int:
    return (FP4ATTN_HB_CAUSAL if causal else 0) | (FP4ATTN_HB_FP8PV if fp8pv else 0)


def host_batch_workspace_bytes(B, H, N, D, causal: bool = False, fp8pv: bool = False) -> int:
    n = ctypes.c_size_t()
    _check(lib().fp4attn_fwd_host_batch_workspace_bytes(B, H, N, D, _hb_flags(causal, fp8pv), ctypes.byref(n)),
           "fp4attn_fwd_host_batch_workspace_bytes")
    return n.value


def empty_host_batch_workspace(shape, device, causal: bool = False, fp8pv: bool = False) -> torch.Tensor:
    """A device workspace for fwd_host_batch (u8, 256-byte aligned)."""
    B, H, N, D = shape
    ws = torch.empty((host_batch_workspace_bytes(B, H, N, D, causal, fp8pv),), dtype=torch.uint8, device=device)
    if ws.data_ptr() % 256:
        raise RuntimeError("the allocator returned a workspace that is not 256-byte aligned")
    return ws


def fwd_host_batch(qs, ks, vs, os_, lses, softmax_scale: float | None = None, causal: bool = False,
                   fp8pv: bool = False, workspace: torch.Tensor | None = None, stream=None) -> None:
    """fp4attn_fwd_host_batch: step i quantizes the host tensors qs[i], ks[i],
    vs[i] (CPU bf16 [B,H,N,D], pinned for overlap) on the workspace's device,
    runs the forward and writes os_[i] (CPU bf16) and lses[i] (CPU fp32
    [B,H,N]).  Asynchronous on `stream`: the outputs are complete, and the
    inputs free, once that stream has synchronised."""
    n = len(qs)
    if n < 1 or not (len(ks) == len(vs) == len(os_) == len(lses) == n):
        raise ValueError("qs, ks, vs, os_ and lses must hold the same number (>= 1) of tensors")
    shape = tuple(qs[0].shape)
    if len(shape) != 4:
        raise ValueError("inputs must be [B,H,N,D]")
    B, H, N, D = shape
    for seq, name, dtype, numel in ((qs, "qs", torch.bfloat16, B * H * N * D), (ks, "ks", torch.bfloat16, B * H * N * D),
                                    (vs, "vs", torch.bfloat16, B * H * N * D), (os_, "os_", torch.bfloat16, B * H * N * D),
                                    (lses, "lses", torch.float32, B * H * N)):
        for j, t in enumerate(seq):
            _check_buffer(t, "%s[%d]" % (name, j), dtype, numel, torch.device("cpu"))
    if workspace is None:
        raise ValueError("fwd_host_batch needs a device workspace (empty_host_batch_workspace)")
    need = host_batch_workspace_bytes(B, H, N, D, causal, fp8pv)
    if not (workspace.is_cuda and workspace.dtype == torch.uint8 and workspace.is_contiguous()
            and workspace.numel() >= need):
        raise ValueError("workspace must be a contiguous CUDA u8 tensor of at least %d bytes" % need)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    arr = lambda seq: (ctypes.c_void_p * n)(*[t.data_ptr() for t in seq])
    with torch.cuda.device(workspace.device):
        _check(lib().fp4attn_fwd_host_batch(n, arr(qs), arr(ks), arr(vs), arr(os_), arr(lses), B, H, N, D,
                                            float(softmax_scale), _hb_flags(causal, fp8pv), _ptr(workspace),
                                            workspace.numel(), ctypes.c_void_p(_stream(stream))),
               "fp4attn_fwd_host_batch")


# ---- causal backward ---------------------------------------------------------

FP8_E4M3, FP8_E5M2 = 0, 1


@dataclass
class FP8Tensor:
    """An MXFP8 operand of the backward: payload u8 and scale atoms u8.
    layout "rows": [B,H,N,D] codes, blocks along D; "t": [B,H,D,Npad] codes,
    blocks along the sequence.  fmt: FP8_E4M3 or FP8_E5M2."""
    payload: torch.Tensor
    sf: torch.Tensor
    shape: tuple
    layout: str
    fmt: int

    def _c(self):  # the C struct has the same two pointers as the MXFP4 one
        return _MXFP4(self.payload.data_ptr(), self.sf.data_ptr())


def mxfp8_rows_bytes(B, H, N, D):
    p, s = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().fp4attn_mxfp8_rows_bytes(B, H, N, D, ctypes.byref(p), ctypes.byref(s)), "fp4attn_mxfp8_rows_bytes")
    return p.value, s.value


def bwd_workspace_bytes(B, H, N, D):
    a, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check(lib().fp4attn_bwd_workspace_bytes(B, H, N, D, ctypes.byref(a), ctypes.byref(b)),
           "fp4attn_bwd_workspace_bytes")
    return a.value, b.value


def empty_fp8(shape, layout: str, fmt: int, device) -> FP8Tensor:
    B, H, N, D = shape
    if layout == "rows":
        pb, sb = mxfp8_rows_bytes(B, H, N, D)
        payload = torch.empty((B, H, N, D), dtype=torch.uint8, device=device)
    elif layout == "t":
        pb, sb = mxfp8_v_bytes(B, H, N, D)
        payload = torch.empty((B, H, D, (N + 127) // 128 * 128), dtype=torch.uint8, device=device)
    else:
        raise ValueError("layout must be 'rows' or 't'")
    return FP8Tensor(payload, torch.empty((sb,), dtype=torch.uint8, device=device), tuple(shape), layout, fmt)


def _check_fp8(t, name: str, shape, layout: str, fmt: int | None = None):
    if not isinstance(t, FP8Tensor):
        raise ValueError("%s must be an FP8Tensor" % name)
    if tuple(t.shape) != tuple(shape) or t.layout != layout or (fmt is not None and t.fmt != fmt):
        raise ValueError("%s must be a %s-layout %s FP8Tensor of shape %s" %
                         (name, layout, {0: "E4M3", 1: "E5M2"}.get(fmt, "FP8"), tuple(shape)))
    B, H, N, D = shape
    pb, sb = (mxfp8_rows_bytes if layout == "rows" else mxfp8_v_bytes)(B, H, N, D)
    dev = t.payload.device
    _check_buffer(t.payload, name + ".payload", torch.uint8, pb, dev)
    _check_buffer(t.sf, name + ".sf", torch.uint8, sb, dev)
    return dev


def _quant_fp8(name, layout, x, fmt, out, stream):
    _check_input(x, "x")
    if fmt not in (FP8_E4M3, FP8_E5M2):
        raise ValueError("fmt must be FP8_E4M3 or FP8_E5M2")
    B, H, N, D = x.shape
    out = out or empty_fp8(x.shape, layout, fmt, x.device)
    if _check_fp8(out, "out", x.shape, layout, fmt) != x.device:
        raise ValueError("out must be on the device of x")
    _check(getattr(lib(), name)(_ptr(x), _ptr(out.payload), _ptr(out.sf), int(fmt), B, H, N, D,
                                ctypes.c_void_p(_stream(stream))), name)
    return out


def quant_mxfp8_rows(x: torch.Tensor, fmt: int, out: FP8Tensor | None = None, stream=None) -> FP8Tensor:
    """fp4attn_quant_mxfp8_rows: MXFP8 along D, row-major."""
    return _quant_fp8("fp4attn_quant_mxfp8_rows", "rows", x, fmt, out, stream)


def quant_mxfp8_t(x: torch.Tensor, fmt: int, out: FP8Tensor | None = None, stream=None) -> FP8Tensor:
    """fp4attn_quant_mxfp8_t: MXFP8 along the sequence, token-inner."""
    return _quant_fp8("fp4attn_quant_mxfp8_t", "t", x, fmt, out, stream)


def bwd_prep(o: torch.Tensor, dout: torch.Tensor, lse: torch.Tensor, nl2: torch.Tensor | None = None,
             delta: torch.Tensor | None = None, stream=None):
    """fp4attn_bwd_prep: returns (nl2, delta), fp32 [B,H,Npad] each (nl2 = -LSE log2 e)."""
    _check_input(o, "o")
    _check_input(dout, "dout")
    if o.shape != dout.shape or o.device != dout.device:
        raise ValueError("o and dout must have one shape and device")
    B, H, N, D = o.shape
    _check_buffer(lse, "lse", torch.float32, B * H * N, o.device)
    npad = (N + 127) // 128 * 128
    nl2 = nl2 if nl2 is not None else torch.empty((B, H, npad), dtype=torch.float32, device=o.device)
    delta = delta if delta is not None else torch.empty((B, H, npad), dtype=torch.float32, device=o.device)
    _check_buffer(nl2, "nl2", torch.float32, B * H * npad, o.device)
    _check_buffer(delta, "delta", torch.float32, B * H * npad, o.device)
    _check(lib().fp4attn_bwd_prep(_ptr(o), _ptr(dout), _ptr(lse), _ptr(nl2), _ptr(delta), B, H, N, D,
                                  ctypes.c_void_p(_stream(stream))), "fp4attn_bwd_prep")
    return nl2, delta


def bwd_directp_causal(q_saved: NVFP4Tensor, k_saved: NVFP4Tensor, v_rows: FP8Tensor, do_rows: FP8Tensor,
                       do_t: FP8Tensor, q_t: FP8Tensor, k_t: FP8Tensor, nl2: torch.Tensor, delta: torch.Tensor,
                       softmax_scale: float | None = None, dq: torch.Tensor | None = None,
                       dk: torch.Tensor | None = None, dv: torch.Tensor | None = None, stream=None):
    """fp4attn_bwd_directp_causal: returns (dQ, dK, dV), fp32 [B,H,N,D]."""
    if not isinstance(q_saved, NVFP4Tensor):
        raise ValueError("q_saved must be an NVFP4Tensor")
    shape = tuple(q_saved.shape)
    dev = _check_quantized(q_saved, "q_saved", shape, NVFP4Tensor)
    if _check_quantized(k_saved, "k_saved", shape, NVFP4Tensor) != dev:
        raise ValueError("the operands must be on one device")
    for t, name, layout, fmt in ((v_rows, "v_rows", "rows", FP8_E4M3), (do_rows, "do_rows", "rows", FP8_E5M2),
                                 (do_t, "do_t", "t", FP8_E5M2), (q_t, "q_t", "t", FP8_E4M3),
                                 (k_t, "k_t", "t", FP8_E4M3)):
        if _check_fp8(t, name, shape, layout, fmt) != dev:
            raise ValueError("the operands must be on one device")
    B, H, N, D = shape
    npad = (N + 127) // 128 * 128
    _check_buffer(nl2, "nl2", torch.float32, B * H * npad, dev)
    _check_buffer(delta, "delta", torch.float32, B * H * npad, dev)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(D)
    outs = []
    for t, name in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        t = t if t is not None else torch.empty((B, H, N, D), dtype=torch.float32, device=dev)
        _check_buffer(t, name, torch.float32, B * H * N * D, dev)
        outs.append(t)
    if dev.type != "cuda":
        raise ValueError("the operands must be CUDA tensors")
    qc, kc = q_saved._c(), k_saved._c()
    cs = [t._c() for t in (v_rows, do_rows, do_t, q_t, k_t)]
    _check(lib().fp4attn_bwd_directp_causal(ctypes.byref(qc), ctypes.byref(kc), *[ctypes.byref(c) for c in cs],
                                            _ptr(nl2), _ptr(delta), *[_ptr(t) for t in outs], B, H, N, D,
                                            float(softmax_scale), ctypes.c_void_p(_stream(stream))),
           "fp4attn_bwd_directp_causal")
    return tuple(outs)


def attention_backward_causal(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, o: torch.Tensor,
                              lse: torch.Tensor, dout: torch.Tensor, q_saved: NVFP4Tensor, k_saved: NVFP4Tensor,
                              softmax_scale: float | None = None, stream=None):
    """The causal backward from the training forward's state (fwd_directp_causal_save: q_saved, k_saved, o,
    lse) and the bf16 inputs q, k, v and output gradient dout: quantizes the FP8 operands (E4M3 V rows,
    E5M2 dO rows and dO^T, E4M3 Q^T and K^T), computes nl2 and Delta, and returns (dQ, dK, dV) fp32."""
    for x, name in ((q, "q"), (k, "k"), (v, "v"), (o, "o"), (dout, "dout")):
        _check_input(x, name)
        if x.shape != q.shape or x.device != q.device:
            raise ValueError("q, k, v, o and dout must have one shape and device")
    v_rows = quant_mxfp8_rows(v, FP8_E4M3, stream=stream)
    do_rows = quant_mxfp8_rows(dout, FP8_E5M2, stream=stream)
    do_t = quant_mxfp8_t(dout, FP8_E5M2, stream=stream)
    q_t = quant_mxfp8_t(q, FP8_E4M3, stream=stream)
    k_t = quant_mxfp8_t(k, FP8_E4M3, stream=stream)
    nl2, delta = bwd_prep(o, dout, lse, stream=stream)
    return bwd_directp_causal(q_saved, k_saved, v_rows, do_rows, do_t, q_t, k_t, nl2, delta, softmax_scale,
                              stream=stream)
