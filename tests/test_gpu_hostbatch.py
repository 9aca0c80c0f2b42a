"""The host-memory batch entry point (fp4attn_fwd_host_batch): each step's O
and LSE equal, bit for bit, what the device-resident calls compute on the
same inputs (same kernels), and agree with the oracle run end to end from the
bf16 inputs (oracle quantizers, oracle forward) within the forward's parity
bar: O max-abs 2e-2 plus the bf16 rounding of the output, LSE 1e-3.  Enough
steps run that both device slots are reused (steps i and i+2 share one)."""
import numpy as np
import pytest
import torch

import oracle
from blackwell_nvfp4_quantize_gb300 import workloads as wl
from _gpu_common import BF16_REL, LSE_TOL, O_TOL

pytestmark = pytest.mark.gpu


def _device_path(fa, q, k, v, scale, causal, fp8pv):
    qq, kq = fa.quant_qk_nvfp4(q.cuda()), fa.quant_qk_nvfp4(k.cuda())
    if fp8pv:
        return fa.fwd_directp_fp8pv(qq, kq, fa.quant_v_mxfp8(v.cuda()), scale, causal=causal)
    fwd = fa.fwd_directp_causal if causal else fa.fwd_directp
    return fwd(qq, kq, fa.quant_v_mxfp4(v.cuda()), scale)


def _oracle_path(q, k, v, scale, causal, fp8pv):
    B, H, N, D = q.shape
    qb, kb, vb = (wl.bf16_bits(t) for t in (q, k, v))
    vq = oracle.quant_mxfp8_v(vb) if fp8pv else oracle.quant_mxfp4_v(vb)
    return oracle.directp_rows(oracle.quant_nvfp4(qb), oracle.quant_nvfp4(kb), vq, (B, H, N, D), scale,
                               np.arange(B * H * N, dtype=np.int64), causal=causal,
                               pv_fmt=oracle.PV_MXFP8 if fp8pv else oracle.PV_MXFP4)


@pytest.mark.parametrize("shape", [(1, 2, 200, 64), (2, 3, 77, 128), (1, 1, 384, 128)])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("fp8pv", [False, True])
def test_host_batch_matches_device_path_and_oracle(shape, causal, fp8pv):
    import blackwell_nvfp4_quantize_gb300 as fa

    B, H, N, D = shape
    steps = 5
    scale = 1.0 / np.sqrt(D)
    ins = [wl.make_custom(B, H, N, D, seed=100 + 7 * i, kind="normal", scale=1.0 + 0.25 * i) for i in range(steps)]
    qs, ks, vs = ([t[j].pin_memory() for t in ins] for j in range(3))
    os_ = [torch.full((B, H, N, D), float("nan"), dtype=torch.bfloat16).pin_memory() for _ in range(steps)]
    lses = [torch.full((B, H, N), float("nan"), dtype=torch.float32).pin_memory() for _ in range(steps)]
    ws = fa.empty_host_batch_workspace(shape, "cuda", causal=causal, fp8pv=fp8pv)
    stream = torch.cuda.Stream()
    fa.fwd_host_batch(qs, ks, vs, os_, lses, scale, causal=causal, fp8pv=fp8pv, workspace=ws, stream=stream)
    stream.synchronize()
    assert fa.device_status() == fa.FP4ATTN_OK
    for i in range(steps):
        o_ref, lse_ref = _device_path(fa, ins[i][0], ins[i][1], ins[i][2], scale, causal, fp8pv)
        torch.cuda.synchronize()
        assert torch.equal(os_[i], o_ref.cpu()), "step %d: O differs from the device path" % i
        assert torch.equal(lses[i], lse_ref.cpu()), "step %d: LSE differs from the device path" % i
    # the first and the last step against the oracle run end to end
    for i in (0, steps - 1):
        ref = _oracle_path(ins[i][0], ins[i][1], ins[i][2], scale, causal, fp8pv)
        o = os_[i].float().numpy().reshape(-1, D)
        err_o = float(np.max(np.abs(o - ref["o"]) - BF16_REL * np.abs(ref["o"])))
        err_l = float(np.max(np.abs(lses[i].numpy().reshape(-1) - ref["lse"])))
        assert err_o <= O_TOL, (i, err_o)
        assert err_l <= LSE_TOL, (i, err_l)


def test_host_batch_pageable_buffers_and_one_step():
    # unpinned host memory still gives the right result (the copies are then
    # staged by the driver and do not overlap), and nsteps = 1 has no slot reuse
    import blackwell_nvfp4_quantize_gb300 as fa

    B, H, N, D = 1, 2, 130, 128
    q, k, v = wl.make_custom(B, H, N, D, seed=5, kind="normal", scale=1.5)
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16)
    lse = torch.empty((B, H, N), dtype=torch.float32)
    ws = fa.empty_host_batch_workspace((B, H, N, D), "cuda")
    fa.fwd_host_batch([q], [k], [v], [o], [lse], workspace=ws)
    torch.cuda.current_stream().synchronize()
    o_ref, lse_ref = _device_path(fa, q, k, v, 1.0 / np.sqrt(D), False, False)
    assert torch.equal(o, o_ref.cpu()) and torch.equal(lse, lse_ref.cpu())


def test_host_batch_orders_after_and_before_the_callers_stream():
    # work queued on the stream before the call is done before the first
    # upload reads its host buffer; work queued after it sees every output
    import blackwell_nvfp4_quantize_gb300 as fa

    B, H, N, D = 1, 1, 256, 64
    q, k, v = wl.make_custom(B, H, N, D, seed=11, kind="normal")
    q_h, k_h, v_h = (t.pin_memory() for t in (q, k, v))
    q_dev = q.cuda()
    q_h.zero_()
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(2_000_000)        # keep the stream busy before the copy back
        q_h.copy_(q_dev, non_blocking=True)  # the input is only complete once this ran
    o = torch.empty((B, H, N, D), dtype=torch.bfloat16).pin_memory()
    lse = torch.empty((B, H, N), dtype=torch.float32).pin_memory()
    ws = fa.empty_host_batch_workspace((B, H, N, D), "cuda")
    fa.fwd_host_batch([q_h], [k_h], [v_h], [o], [lse], workspace=ws, stream=stream)
    o_dev = torch.empty((B, H, N, D), dtype=torch.bfloat16, device="cuda")
    with torch.cuda.stream(stream):
        o_dev.copy_(o, non_blocking=True)    # queued after the call: sees the finished O
    stream.synchronize()
    o_ref, _ = _device_path(fa, q, k, v, 1.0 / np.sqrt(D), False, False)
    torch.cuda.synchronize()
    assert torch.equal(o, o_ref.cpu())
    assert torch.equal(o_dev, o_ref)
