"""Parity of the Direct-P forward kernel with the oracle, on identical
quantized operands (the GPU's own quantized buffers feed the oracle):
  probability codes agree on >= 99.9% of entries (ties may flip with fp32
  accumulation order), block shifts likewise, O within max-abs 2e-2 and LSE
  within 1e-3.  Cosine similarity against unquantized fp64 attention is
  reported, not asserted (beyond a loose sanity floor)."""
import math

import numpy as np
import pytest

import oracle
from blackwell_nvfp4_quantize_gb300 import workloads as wl
from _gpu_common import cosine, run_and_check, sample_rows

pytestmark = pytest.mark.gpu


def test_workload1_full():
    w = wl.WORKLOADS[1]
    q, k, v = wl.make_inputs(w)
    B, H, N, D = w.shape
    o, lse = run_and_check(q, k, v, w.softmax_scale, [(0, 0, 0, N)], np.arange(B * H * N, dtype=np.int64),
                           "workload 1")
    # report: cosine against unquantized fp64 attention
    ex_o, _ = oracle.exact_rows(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), w.softmax_scale,
                                np.arange(B * H * N))
    cos = cosine(o, ex_o)
    print("workload 1: cosine vs fp64 unquantized attention %.5f" % cos)
    assert cos > 0.95


@pytest.mark.parametrize("idx", [2, 3, 5, 4])
def test_workloads_sampled(idx):
    # every head: rows 0 and N-1 and 16 more spread over the sequence (the two
    # largest workloads) or 48; codes, shifts and fp32 O in full for 128-row
    # slices at the start, the end and the middle of the head range
    w = wl.WORKLOADS[idx]
    q, k, v = wl.make_inputs(w)
    B, H, N, D = w.shape
    sample = sample_rows(B, H, N, range(B * H), 16 if idx in (4, 5) else 48, seed=idx)
    last_b, last_h = divmod(B * H - 1, H)
    mid_b, mid_h = divmod((B * H) // 2, H)
    dumps = [(0, 0, 0, 128), (last_b, last_h, N - 128, 128), (mid_b, mid_h, N // 2 - 64, 128)]
    o, lse = run_and_check(q, k, v, w.softmax_scale, dumps, sample, "workload %d" % idx)
    sub = sample[:: max(1, len(sample) // 64)][:64]
    ex_o, _ = oracle.exact_rows(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), w.softmax_scale, sub)
    print("workload %d: cosine vs fp64 unquantized attention %.5f" % (idx, cosine(o[sub], ex_o)))


@pytest.mark.parametrize("N", [1, 33, 77, 128, 200, 383])
@pytest.mark.parametrize("D", [64, 128])
def test_ragged_lengths(N, D):
    q, k, v = wl.make_custom(1, 2, N, D, seed=7 + N, kind="normal", scale=1.5)
    B, H = 1, 2
    run_and_check(q, k, v, 1.0 / math.sqrt(D), [(0, 1, 0, N)], np.arange(B * H * N, dtype=np.int64),
                  "ragged N=%d D=%d" % (N, D))


@pytest.mark.parametrize("D", [64, 128])
def test_all_equal_scores(D):
    # Q = 0: every score is 0, every code is 6 (4.0) with scale 2^-2, O = mean of V-hat, LSE = ln N
    N = 256
    q, k, v = wl.make_custom(1, 1, N, D, seed=3, kind="zero_q")
    o, lse = run_and_check(q, k, v, 0.125, [(0, 0, 0, N)], np.arange(N, dtype=np.int64), "zero q D=%d" % D)
    assert np.max(np.abs(lse - math.log(N))) < 1e-5


def test_large_scale_rows():
    # wide dynamic range of scores: many rescales of O, many zero codes
    q, k, v = wl.make_custom(1, 2, 640, 128, seed=12, kind="normal", scale=4.0)
    run_and_check(q, k, v, 1.0 / math.sqrt(128), [(0, 0, 0, 640)], np.arange(2 * 640, dtype=np.int64),
                  "scale 4")


def test_timeout_status_word_is_clear():
    import blackwell_nvfp4_quantize_gb300 as fa

    assert fa.device_status() == fa.FP4ATTN_OK


def test_side_streams_and_preallocated_outputs():
    # every call is asynchronous on the caller's stream: two forwards on two
    # side streams at once, into preallocated outputs, give the results of the
    # default-stream call
    import torch

    import blackwell_nvfp4_quantize_gb300 as fa

    q, k, v = wl.make_custom(1, 4, 1000, 128, seed=77, kind="normal", scale=1.5)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    o_ref, lse_ref = fa.attention(qc, kc, vc)
    oc_ref, lsec_ref = fa.attention(qc, kc, vc, causal=True)
    torch.cuda.synchronize()
    s1, s2 = torch.cuda.Stream(), torch.cuda.Stream()
    o1, o2 = torch.empty_like(o_ref), torch.empty_like(o_ref)
    l1, l2 = torch.empty_like(lse_ref), torch.empty_like(lse_ref)
    with torch.cuda.stream(s1):
        q1, k1, v1 = fa.quant_qk_nvfp4(qc, stream=s1), fa.quant_qk_nvfp4(kc, stream=s1), fa.quant_v_mxfp4(vc, stream=s1)
        fa.fwd_directp(q1, k1, v1, o=o1, lse=l1, stream=s1)
    with torch.cuda.stream(s2):
        q2, k2, v2 = fa.quant_qk_nvfp4(qc, stream=s2), fa.quant_qk_nvfp4(kc, stream=s2), fa.quant_v_mxfp4(vc, stream=s2)
        fa.fwd_directp_causal(q2, k2, v2, o=o2, lse=l2, stream=s2)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FP4ATTN_OK
    assert torch.equal(o1, o_ref) and torch.equal(l1, lse_ref)
    assert torch.equal(o2, oc_ref) and torch.equal(l2, lsec_ref)


@pytest.mark.parametrize("causal", [False, True])
def test_most_heads(causal):
    # B*H = 65535, the most heads one launch takes (one grid row per head);
    # a ragged 17-row sequence per head, so every head ends in a partial tile
    import torch

    B, H, N, D = 3, 21845, 17, 64
    q, k, v = wl.make_custom(B, H, N, D, seed=55, kind="normal", scale=1.5)
    heads = [0, 1, H - 1, H, 2 * H + 7, B * H - 1]
    sample = sample_rows(B, H, N, heads, N, seed=55)
    run_and_check(q, k, v, 1.0 / math.sqrt(D), [(B - 1, H - 1, 0, N)], sample,
                  "65535 heads causal=%d" % causal, causal=causal)
    del q, k, v
    torch.cuda.empty_cache()
