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
    w = wl.WORKLOADS[idx]
    q, k, v = wl.make_inputs(w)
    B, H, N, D = w.shape
    heads = sorted({0, B * H - 1, (B * H) // 2})
    sample = sample_rows(B, H, N, heads, 48 if idx == 4 else 96, seed=idx)
    last_b, last_h = divmod(B * H - 1, H)
    dumps = [(0, 0, 0, 128), (last_b, last_h, N - 128, 128)]
    o, lse = run_and_check(q, k, v, w.softmax_scale, dumps, sample, "workload %d" % idx)
    ex_o, _ = oracle.exact_rows(wl.bf16_bits(q), wl.bf16_bits(k), wl.bf16_bits(v), w.softmax_scale,
                                sample[:64])
    print("workload %d: cosine vs fp64 unquantized attention %.5f" % (idx, cosine(o[sample[:64]], ex_o)))


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
