"""The allocation-free forward entry point, fp4attn_fwd_directp_noalloc.

It exists for callers that cannot let a library allocate device memory:
processes that reserved nearly all of the GPU's memory for their own pool,
frameworks that route every allocation through their own allocator, loops
that cannot take an allocation's implicit synchronisation.  It runs the same
kernel as fp4attn_fwd_directp with its status word in a static device array,
so its outputs must be bit-identical to the regular entry point's.

This file is named so that pytest collects it last; it passes alone in a
fresh process and after the other tests.
"""
import ctypes
import json
import math
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from blackwell_nvfp4_quantize_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def _call_c_abi(fa, qq, kq, vq, o, lse, scale):
    B, H, N, D = qq.shape
    qc, kc, vc = qq._c(), kq._c(), vq._c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return fa.lib().fp4attn_fwd_directp_noalloc(ctypes.byref(qc), ctypes.byref(kc), ctypes.byref(vc),
                                                ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
                                                B, H, N, D, ctypes.c_float(scale), stream)


@pytest.mark.parametrize("B,H,N,D", [(1, 1, 256, 64), (1, 3, 333, 128), (2, 2, 1024, 128)])
def test_noalloc_bit_identical_to_regular_entry_point_twice(B, H, N, D):
    import blackwell_nvfp4_quantize_gb300 as fa

    q, k, v = wl.make_custom(B, H, N, D, seed=4000 + N + D, kind="normal", scale=1.5)
    qq, kq, vq = fa.quant_qk_nvfp4(q.cuda()), fa.quant_qk_nvfp4(k.cuda()), fa.quant_v_mxfp4(v.cuda())
    scale = 1.0 / math.sqrt(D)
    o_ref, lse_ref = fa.fwd_directp(qq, kq, vq, scale)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FP4ATTN_OK
    for call in range(2):
        o = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        if call == 0:
            status = _call_c_abi(fa, qq, kq, vq, o, lse, scale)
            assert status == fa.FP4ATTN_OK, fa.status_string(status)
        else:
            fa.fwd_directp_noalloc(qq, kq, vq, o, lse, scale)  # the Python wrapper of the same call
        torch.cuda.synchronize()
        assert torch.equal(o, o_ref), "call %d: O differs from fp4attn_fwd_directp" % call
        assert torch.equal(lse, lse_ref), "call %d: LSE differs from fp4attn_fwd_directp" % call


def test_noalloc_first_in_a_fresh_process_creates_no_status_block():
    # In a fresh process the quantizers and then the allocation-free forward
    # (twice) run before anything else; the library's per-device status block
    # -- its only cudaMalloc -- must not exist afterwards.  The regular forward
    # run after them creates it and gives bit-identical outputs.
    r = subprocess.run([sys.executable, os.path.join(HERE, "_noalloc_fresh.py")], capture_output=True, text=True,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    out = json.loads(r.stdout.strip().splitlines()[-1])
    assert out["status"] == [0, 0], out
    assert out["before"] is False and out["after_noalloc"] is False, out
    assert out["after_regular"] is True, out
    assert out["equal"] == [True, True], out


def test_noalloc_timeout_shows_as_nan_then_recovers():
    # The entry point's only failure signal: a bounded wait that gave up turns
    # every LSE entry into NaN.  Driven without a fault: a wait on the static
    # status word that nothing completes gives up after 20 ms.  The next call
    # clears the word and computes normally.
    import blackwell_nvfp4_quantize_gb300 as fa

    B, H, N, D = 1, 2, 300, 64
    q, k, v = wl.make_custom(B, H, N, D, seed=77, kind="normal", scale=1.5)
    qq, kq, vq = fa.quant_qk_nvfp4(q.cuda()), fa.quant_qk_nvfp4(k.cuda()), fa.quant_v_mxfp4(v.cuda())
    lse = torch.zeros((B, H, N), dtype=torch.float32, device="cuda")
    fa.debug_noalloc_timeout(lse, 20000)
    torch.cuda.synchronize()
    assert bool(torch.isnan(lse).all()), "a timed-out wait must turn every LSE entry into NaN"
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16, device="cuda")
    fa.fwd_directp_noalloc(qq, kq, vq, o, lse)
    o_ref, lse_ref = fa.fwd_directp(qq, kq, vq)
    torch.cuda.synchronize()
    assert bool(torch.isfinite(lse).all()) and np.isfinite(o.float().cpu().numpy()).all()
    assert torch.equal(o, o_ref) and torch.equal(lse, lse_ref)


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
