"""The allocation-free forward entry point against the regular one.

fp4attn_fwd_directp_noalloc exists for callers that cannot let a library
allocate device memory -- processes that reserved nearly all of it for their
own pool, frameworks that forbid allocations outside their allocator, loops
that cannot afford an allocation's implicit synchronisation.  It must produce
what fp4attn_fwd_directp produces.  This file is named so that pytest collects
it last, and it works both alone in a fresh process and after the other tests.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from blackwell_nvfp4_quantize_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

O_TOL = 2e-2           # as in the forward parity tests
BF16_REL = 2.0 ** -8   # stored O is bf16
LSE_TOL = 1e-3


@pytest.mark.parametrize("B,H,N,D", [(1, 1, 256, 64), (1, 3, 333, 128), (2, 2, 1024, 128)])
def test_noalloc_matches_regular_entry_point_twice(B, H, N, D):
    import blackwell_nvfp4_quantize_gb300 as fa

    L = fa.lib()
    q, k, v = wl.make_custom(B, H, N, D, seed=4000 + N + D, kind="normal", scale=1.5)
    qq, kq, vq = fa.quant_qk_nvfp4(q.cuda()), fa.quant_qk_nvfp4(k.cuda()), fa.quant_v_mxfp4(v.cuda())
    scale = 1.0 / math.sqrt(D)
    o_ref, lse_ref = fa.fwd_directp(qq, kq, vq, scale)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FP4ATTN_OK
    o_ref = o_ref.float().cpu().numpy()
    lse_ref = lse_ref.cpu().numpy()
    qc, kc, vc = qq._c(), kq._c(), vq._c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    for call in range(2):
        o = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        status = L.fp4attn_fwd_directp_noalloc(ctypes.byref(qc), ctypes.byref(kc), ctypes.byref(vc),
                                               ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
                                               B, H, N, D, ctypes.c_float(scale), stream)
        assert status == fa.FP4ATTN_OK, fa.status_string(status)
        torch.cuda.synchronize()
        o_np = o.float().cpu().numpy()
        lse_np = lse.cpu().numpy()
        assert np.all(np.isfinite(o_np)) and np.all(np.isfinite(lse_np)), "call %d left NaN" % call
        assert np.all(np.abs(o_np - o_ref) <= O_TOL + BF16_REL * np.abs(o_ref)), "call %d" % call
        assert np.max(np.abs(lse_np - lse_ref)) <= LSE_TOL, "call %d" % call


def test_noalloc_rejects_bad_arguments():
    import blackwell_nvfp4_quantize_gb300 as fa

    L = fa.lib()
    q = fa._NVFP4(0x1000, 0x2000, 0x3000)
    v = fa._MXFP4(0x4000, 0x5000)
    good = ctypes.c_void_p(0x6000)
    assert L.fp4attn_fwd_directp_noalloc(ctypes.byref(q), ctypes.byref(q), ctypes.byref(v), good, good, 1, 1,
                                         128, 96, ctypes.c_float(0.1), None) == fa.FP4ATTN_ERR_UNSUPPORTED
    assert L.fp4attn_fwd_directp_noalloc(ctypes.byref(q), ctypes.byref(q), ctypes.byref(v), None, good, 1, 1,
                                         128, 64, ctypes.c_float(0.1), None) == fa.FP4ATTN_ERR_INVALID_ARG
