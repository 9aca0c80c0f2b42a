"""Parity of the FP8 P/V variant ("Hardware-Aware FP4 FlashAttention-4",
"What the paper found": training keeps FP8 probabilities and values) with the
oracle: the MXFP8 V quantizer bit-exact on full tensors, and the forward with
E4M3 probability codes and MXFP8 V -- noncausal and causal -- at the same bar
as the E2M1 forward (codes and block shifts >= 99.9% equal, O max-abs 2e-2,
LSE 1e-3), on identical quantized operands."""
import math

import numpy as np
import pytest
import torch

import oracle
from blackwell_nvfp4_quantize_gb300 import workloads as wl
from _gpu_common import mx_to_np, run_and_check, sample_rows

pytestmark = pytest.mark.gpu


def _check_mxfp8(v, heads=None):
    """GPU MXFP8 V against the oracle; heads: check only the first `heads` heads (per-head blocks)."""
    import blackwell_nvfp4_quantize_gb300 as fa

    t = fa.quant_v_mxfp8(v.cuda())
    p, sf = mx_to_np(t)
    B, H, N, D = v.shape
    if heads is None:
        rp, rsf = oracle.quant_mxfp8_v(wl.bf16_bits(v))
    else:
        assert B == 1
        rp, rsf = oracle.quant_mxfp8_v(wl.bf16_bits(v[:, :heads].contiguous()))
        p = p[:, :heads]
        sf = sf[:rsf.size]
    assert np.array_equal(sf, rsf), "scale atoms differ at %s" % np.argwhere(sf != rsf)[:5].tolist()
    assert np.array_equal(p, rp), "payload differs at %s" % np.argwhere(p != rp)[:5].tolist()


@pytest.mark.parametrize("idx", [1, 2, 3, 5, 4])
def test_mxfp8_quantizer_bit_exact_on_workloads(idx):
    w = wl.WORKLOADS[idx]
    _, _, v = wl.make_inputs(w)
    _check_mxfp8(v)
    torch.cuda.empty_cache()


@pytest.mark.parametrize("N", [1, 31, 77, 128, 129, 300])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("kind", ["normal", "wide", "zeros"])
def test_mxfp8_quantizer_edge_cases(N, D, kind):
    _, _, v = wl.make_custom(2, 3, N, D, seed=200 + N + D, kind=kind, scale=3.0)
    _check_mxfp8(v)


def test_mxfp8_hand_worked_block(golden_dir):
    import json
    import os

    import blackwell_nvfp4_quantize_gb300 as fa

    g = json.load(open(os.path.join(golden_dir, "mxfp8_block.json")))
    bits = [int(x, 16) if x.startswith("0x") else int(x) for x in g["v_bf16_bits"]]
    v = torch.tensor(bits, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).reshape(g["shape"])
    # the quantizer needs D in {64, 128}: the fixture's channel is channel 0 of a 64-channel tensor
    v64 = torch.zeros((1, 1, 64, 64), dtype=torch.bfloat16)
    v64[..., 0] = v[..., 0]
    t = fa.quant_v_mxfp8(v64.cuda())
    p = t.payload_t.cpu().numpy()
    want = [int(x, 16) if x.startswith("0x") else int(x) for x in g["codes_first_64"]]
    assert p[0, 0, 0, :64].tolist() == want
    assert t.sf.cpu().numpy()[:4].tolist() == g["scale_bytes_row0"]


@pytest.mark.parametrize("causal", [False, True])
def test_fp8pv_workload1_full(causal):
    w = wl.WORKLOADS[1]
    q, k, v = wl.make_inputs(w)
    B, H, N, D = w.shape
    run_and_check(q, k, v, w.softmax_scale, [(0, 0, 0, N)], np.arange(B * H * N, dtype=np.int64),
                  "fp8pv workload 1 causal=%d" % causal, causal=causal, fp8pv=True)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("idx", [2, 3, 5, 4])
def test_fp8pv_workloads_sampled(idx, causal):
    w = wl.WORKLOADS[idx]
    q, k, v = wl.make_inputs(w)
    B, H, N, D = w.shape
    sample = sample_rows(B, H, N, range(B * H), 16 if idx in (4, 5) else 32, seed=300 + idx)
    last_b, last_h = divmod(B * H - 1, H)
    mid_b, mid_h = divmod((B * H) // 2, H)
    dumps = [(0, 0, 0, 64), (last_b, last_h, N - 64, 64), (mid_b, mid_h, N // 2 - 64, 128)]
    run_and_check(q, k, v, w.softmax_scale, dumps, sample, "fp8pv workload %d causal=%d" % (idx, causal),
                  causal=causal, fp8pv=True)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 33, 128, 200, 383, 640])
@pytest.mark.parametrize("D", [64, 128])
def test_fp8pv_ragged_lengths(N, D, causal):
    q, k, v = wl.make_custom(1, 2, N, D, seed=27 + N, kind="normal", scale=1.5)
    run_and_check(q, k, v, 1.0 / math.sqrt(D), [(0, 1, 0, N)], np.arange(2 * N, dtype=np.int64),
                  "fp8pv ragged N=%d D=%d causal=%d" % (N, D, causal), causal=causal, fp8pv=True)


@pytest.mark.parametrize("D", [64, 128])
def test_fp8pv_all_equal_scores(D):
    # Q = 0: every score 0, every code E4M3(256) = 0x78 at scale 2^-8, O = mean of V-hat, LSE = ln N
    N = 256
    q, k, v = wl.make_custom(1, 1, N, D, seed=3, kind="zero_q")
    o, lse = run_and_check(q, k, v, 0.125, [(0, 0, 0, N)], np.arange(N, dtype=np.int64), "fp8pv zero q D=%d" % D,
                           fp8pv=True)
    assert np.max(np.abs(lse - math.log(N))) < 1e-5


def test_fp8pv_large_scale_rows():
    q, k, v = wl.make_custom(1, 2, 640, 128, seed=12, kind="normal", scale=4.0)
    run_and_check(q, k, v, 1.0 / math.sqrt(128), [(0, 0, 0, 640)], np.arange(2 * 640, dtype=np.int64),
                  "fp8pv scale 4", fp8pv=True)
