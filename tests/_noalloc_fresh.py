"""Run by tests/test_zz_no_alloc.py in a fresh process: the allocation-free
forward is the first forward call of the process, so whether the library's
per-device status block exists afterwards shows whether that call created it.
Prints one JSON line."""
import ctypes
import json
import math
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import blackwell_nvfp4_quantize_gb300 as fa  # noqa: E402
from blackwell_nvfp4_quantize_gb300 import workloads as wl  # noqa: E402


def main():
    torch.cuda.set_device(0)
    B, H, N, D = 1, 3, 333, 128
    q, k, v = wl.make_custom(B, H, N, D, seed=4242, kind="normal", scale=1.5)
    qq, kq, vq = fa.quant_qk_nvfp4(q.cuda()), fa.quant_qk_nvfp4(k.cuda()), fa.quant_v_mxfp4(v.cuda())
    torch.cuda.synchronize()
    before = fa.debug_status_word_exists()
    L = fa.lib()
    qc, kc, vc = qq._c(), kq._c(), vq._c()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    outs = []
    for _ in range(2):
        o = torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device="cuda")
        st = L.fp4attn_fwd_directp_noalloc(ctypes.byref(qc), ctypes.byref(kc), ctypes.byref(vc),
                                           ctypes.c_void_p(o.data_ptr()), ctypes.c_void_p(lse.data_ptr()),
                                           B, H, N, D, ctypes.c_float(1.0 / math.sqrt(D)), stream)
        outs.append((st, o, lse))
    torch.cuda.synchronize()
    after_noalloc = fa.debug_status_word_exists()
    o_ref, lse_ref = fa.fwd_directp(qq, kq, vq)
    torch.cuda.synchronize()
    after_regular = fa.debug_status_word_exists()
    print(json.dumps({
        "status": [st for st, _, _ in outs],
        "before": before, "after_noalloc": after_noalloc, "after_regular": after_regular,
        "equal": [bool(torch.equal(o, o_ref) and torch.equal(lse, lse_ref)) for _, o, lse in outs],
    }))


if __name__ == "__main__":
    main()
