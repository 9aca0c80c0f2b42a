"""Parity of the Direct-P forward kernel with the oracle, on identical
quantized operands (the GPU's own quantized buffers feed the oracle):
  probability codes agree on >= 99.9% of entries (ties may flip with fp32
  accumulation order), block shifts likewise, O within max-abs 2e-2 and LSE
  within 1e-3.  Cosine similarity against unquantized fp64 attention is
  reported, not asserted (beyond a loose sanity floor)."""
import math

import numpy as np
import pytest
import torch

import oracle
from blackwell_nvfp4_quantize_gb300 import workloads as wl
from _gpu_common import cosine, mx_to_np, nv_to_np, sample_rows, unpack_codes

pytestmark = pytest.mark.gpu

O_TOL = 2e-2
LSE_TOL = 1e-3
CODE_AGREE = 0.999
# O is stored in bf16 (round to nearest even: relative error <= 2^-9).  The
# 2e-2 absolute bound applies to O as computed (fp32, before that store, read
# through the dump entry point); the stored bf16 O is checked against
# 2e-2 plus its own rounding, and to be exactly the rounding of the fp32 value.
BF16_REL = 2.0 ** -8


def _quantize(q, k, v):
    import blackwell_nvfp4_quantize_gb300 as fa

    return fa.quant_qk_nvfp4(q.cuda()), fa.quant_qk_nvfp4(k.cuda()), fa.quant_v_mxfp4(v.cuda())


def _run_and_check(q, k, v, scale, dump_slices, sample, label):
    """dump_slices: list of (b, h, row0, nrows) compared in full (codes, block
    shifts, fp32 O before its bf16 store, LSE); sample: flat row ids whose
    stored bf16 O and LSE are compared."""
    import blackwell_nvfp4_quantize_gb300 as fa

    B, H, N, D = q.shape
    qq, kq, vq = _quantize(q, k, v)
    o, lse = fa.fwd_directp(qq, kq, vq, scale)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FP4ATTN_OK
    qn, kn, vn = nv_to_np(qq), nv_to_np(kq), mx_to_np(vq)
    o_np = o.float().cpu().numpy().reshape(-1, D)
    lse_np = lse.cpu().numpy().reshape(-1)
    assert np.all(np.isfinite(o_np)) and np.all(np.isfinite(lse_np))
    # stored bf16 O / LSE on sampled rows: 2e-2 plus the bf16 rounding of the output
    ref = oracle.directp_rows(qn, kn, vn, (B, H, N, D), scale, sample)
    err_o16 = float(np.max(np.abs(o_np[sample] - ref["o"]) - BF16_REL * np.abs(ref["o"])))
    err_l = float(np.max(np.abs(lse_np[sample] - ref["lse"])))
    # codes, block shifts and fp32 O through the dump entry point (same kernel and launch shape)
    agree = total = kagree = ktotal = 0
    err_o32 = 0.0
    for (b, h, row0, nrows) in dump_slices:
        o2, lse2, codes, kshift, o32 = fa.debug_dump_p(qq, kq, vq, b, h, row0, nrows, scale)
        torch.cuda.synchronize()
        # the dump variant computes the same O / LSE, and O is the bf16 rounding of its fp32 value
        assert torch.equal(o2, o) and torch.equal(lse2, lse)
        assert torch.equal(o32.to(torch.bfloat16), o2.reshape(-1, D)[(b * H + h) * N + row0:][:nrows])
        rows = np.arange(nrows, dtype=np.int64) + (b * H + h) * N + row0
        r = oracle.directp_rows(qn, kn, vn, (B, H, N, D), scale, rows, want_codes=True)
        err_o32 = max(err_o32, float(np.max(np.abs(o32.cpu().numpy() - r["o"]))))
        err_l = max(err_l, float(np.max(np.abs(lse_np[rows] - r["lse"]))))
        gc = unpack_codes(codes.cpu().numpy())
        agree += int(np.sum(gc[:, :N] == r["codes"][:, :N]))
        total += nrows * N
        nblk = (N + 31) // 32
        gk = kshift.cpu().numpy()[:, :nblk]
        kagree += int(np.sum(gk == r["kshift"][:, :nblk]))
        ktotal += gk.size
        assert np.all(gc[:, N:] == 0)
    frac = agree / max(total, 1)
    kfrac = kagree / max(ktotal, 1)
    print("%s: max|dO32|=%.3g max|dO16|-bf16=%.3g max|dLSE|=%.3g codes agree %.6f kshift agree %.6f"
          % (label, err_o32, err_o16, err_l, frac, kfrac))
    assert err_o32 <= O_TOL, err_o32
    assert err_o16 <= O_TOL, err_o16
    assert err_l <= LSE_TOL, err_l
    if total:
        assert frac >= CODE_AGREE, frac
        assert kfrac >= CODE_AGREE, kfrac
    return o_np, lse_np


def test_workload1_full():
    w = wl.WORKLOADS[1]
    q, k, v = wl.make_inputs(w)
    B, H, N, D = w.shape
    o, lse = _run_and_check(q, k, v, w.softmax_scale, [(0, 0, 0, N)], np.arange(B * H * N, dtype=np.int64),
                            "workload 1")
    # report: cosine against unquantized fp64 attention
    ex_o, _ = oracle.exact_rows(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), w.softmax_scale,
                                np.arange(B * H * N))
    cos = cosine(o, ex_o)
    print("workload 1: cosine vs fp64 unquantized attention %.5f" % cos)
    assert cos > 0.95


@pytest.mark.parametrize("idx", [2, 3, 5, 4])
def test_workloads_sampled(idx):
    w = wl.WORKLOADS[idx]
    q, k, v = wl.make_inputs(w)
    B, H, N, D = w.shape
    heads = sorted({0, B * H - 1, (B * H) // 2})
    sample = sample_rows(B, H, N, heads, 48 if idx == 4 else 96, seed=idx)
    last_b, last_h = divmod(B * H - 1, H)
    dumps = [(0, 0, 0, 128), (last_b, last_h, N - 128, 128)]
    o, lse = _run_and_check(q, k, v, w.softmax_scale, dumps, sample, "workload %d" % idx)
    ex_o, _ = oracle.exact_rows(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), w.softmax_scale,
                                sample[:64])
    print("workload %d: cosine vs fp64 unquantized attention %.5f" % (idx, cosine(o[sample[:64]], ex_o)))


@pytest.mark.parametrize("N", [1, 33, 77, 128, 200, 383])
@pytest.mark.parametrize("D", [64, 128])
def test_ragged_lengths(N, D):
    q, k, v = wl.make_custom(1, 2, N, D, seed=7 + N, kind="normal", scale=1.5)
    B, H = 1, 2
    _run_and_check(q, k, v, 1.0 / math.sqrt(D), [(0, 1, 0, N)], np.arange(B * H * N, dtype=np.int64),
                   "ragged N=%d D=%d" % (N, D))


@pytest.mark.parametrize("D", [64, 128])
def test_all_equal_scores(D):
    # Q = 0: every score is 0, every code is 6 (4.0) with scale 2^-2, O = mean of V-hat, LSE = ln N
    N = 256
    q, k, v = wl.make_custom(1, 1, N, D, seed=3, kind="zero_q")
    o, lse = _run_and_check(q, k, v, 0.125, [(0, 0, 0, N)], np.arange(N, dtype=np.int64), "zero q D=%d" % D)
    assert np.max(np.abs(lse - math.log(N))) < 1e-5


def test_large_scale_rows():
    # wide dynamic range of scores: many rescales of O, many zero codes
    q, k, v = wl.make_custom(1, 2, 640, 128, seed=12, kind="normal", scale=4.0)
    _run_and_check(q, k, v, 1.0 / math.sqrt(128), [(0, 0, 0, 640)], np.arange(2 * 640, dtype=np.int64),
                   "scale 4")


def test_timeout_status_word_is_clear():
    import blackwell_nvfp4_quantize_gb300 as fa

    assert fa.device_status() == fa.FP4ATTN_OK
