"""Parity of the causal Direct-P forward (query i sees keys 0..i; the causal
training forward of "Hardware-Aware FP4 FlashAttention-4", "What the paper
found") with the oracle's causal rows, on identical quantized operands, at
the same bar as the noncausal forward.  The cases cover both query-tile
pairings of the kernel (an even number of query tiles, and an odd number with
a lone middle tile), partial last tiles, and the one-call entry point that
quantizes Q/K/V, keeps the quantized Q/K and runs the causal forward."""
import math

import numpy as np
import pytest
import torch

from blackwell_nvfp4_quantize_gb300 import workloads as wl
from _gpu_common import quantize, run_and_check, sample_rows

pytestmark = pytest.mark.gpu


def test_causal_workload1_full():
    w = wl.WORKLOADS[1]
    q, k, v = wl.make_inputs(w)
    B, H, N, D = w.shape
    run_and_check(q, k, v, w.softmax_scale, [(0, 0, 0, N)], np.arange(B * H * N, dtype=np.int64),
                  "causal workload 1", causal=True)


@pytest.mark.parametrize("idx", [2, 3, 5, 4])
def test_causal_workloads_sampled(idx):
    w = wl.WORKLOADS[idx]
    q, k, v = wl.make_inputs(w)
    B, H, N, D = w.shape
    # every head, rows spread over the sequence (short early rows and full
    # late rows alike); full slices at the first rows, the last rows and the
    # middle of a middle head
    sample = sample_rows(B, H, N, range(B * H), 16 if idx in (4, 5) else 48, seed=100 + idx)
    last_b, last_h = divmod(B * H - 1, H)
    mid_b, mid_h = divmod((B * H) // 2, H)
    dumps = [(0, 0, 0, 128), (last_b, last_h, N - 128, 128), (mid_b, mid_h, N // 2 - 64, 128)]
    run_and_check(q, k, v, w.softmax_scale, dumps, sample, "causal workload %d" % idx, causal=True)


@pytest.mark.parametrize("N", [1, 33, 128, 129, 200, 256, 383, 640, 700])
@pytest.mark.parametrize("D", [64, 128])
def test_causal_ragged_lengths(N, D):
    q, k, v = wl.make_custom(1, 2, N, D, seed=17 + N, kind="normal", scale=1.5)
    run_and_check(q, k, v, 1.0 / math.sqrt(D), [(0, 1, 0, N)], np.arange(2 * N, dtype=np.int64),
                  "causal ragged N=%d D=%d" % (N, D), causal=True)


def test_causal_large_scale_rows():
    # wide dynamic range: many rescales, many zero codes, short early rows
    q, k, v = wl.make_custom(2, 2, 896, 128, seed=19, kind="normal", scale=4.0)
    run_and_check(q, k, v, 1.0 / math.sqrt(128), [(1, 1, 0, 896)], np.arange(4 * 896, dtype=np.int64),
                  "causal scale 4", causal=True)


@pytest.mark.parametrize("shape", [(1, 3, 520, 64), (2, 2, 1024, 128)])
def test_causal_save_matches_separate_calls(shape):
    import blackwell_nvfp4_quantize_gb300 as fa

    B, H, N, D = shape
    q, k, v = wl.make_custom(B, H, N, D, seed=23 + N, kind="normal", scale=1.0)
    qc, kc, vc = q.cuda(), k.cuda(), v.cuda()
    for _ in range(2):  # two calls in a row give the same bytes
        o, lse, qs, ks, vs = fa.fwd_directp_causal_save(qc, kc, vc)
        qq, kq, vq = quantize(q, k, v)
        o2, lse2 = fa.fwd_directp_causal(qq, kq, vq)
        torch.cuda.synchronize()
        assert fa.device_status() == fa.FP4ATTN_OK
        assert torch.equal(qs.payload, qq.payload) and torch.equal(qs.sf, qq.sf) and torch.equal(qs.g, qq.g)
        assert torch.equal(ks.payload, kq.payload) and torch.equal(ks.sf, kq.sf) and torch.equal(ks.g, kq.g)
        assert torch.equal(vs.payload_t, vq.payload_t) and torch.equal(vs.sf, vq.sf)
        assert torch.equal(o, o2) and torch.equal(lse, lse2)


def test_causal_last_row_matches_noncausal():
    import blackwell_nvfp4_quantize_gb300 as fa

    q, k, v = wl.make_custom(1, 2, 384, 128, seed=29, kind="normal", scale=1.5)
    qq, kq, vq = quantize(q, k, v)
    oc, lc = fa.fwd_directp_causal(qq, kq, vq)
    on, ln = fa.fwd_directp(qq, kq, vq)
    torch.cuda.synchronize()
    # the last row sees every key in both forwards (each within the parity bar of the same oracle row)
    assert torch.allclose(lc[:, :, -1], ln[:, :, -1], atol=2e-3, rtol=0)
    assert torch.allclose(oc[:, :, -1].float(), on[:, :, -1].float(), atol=4e-2, rtol=0)
    # the first row sees only key 0 and differs
    assert not torch.equal(lc[:, :, 0], ln[:, :, 0])


@pytest.mark.parametrize("causal,fp8pv", [(False, False), (True, False), (False, True), (True, True)])
def test_long_single_head(causal, fp8pv):
    # one head with 200000 keys (1563 key tiles, the last one partial): every
    # index of the kernels and the dump stays in range; rows spread over the
    # sequence, both ends included
    N, D = 200000, 128
    q, k, v = wl.make_custom(1, 1, N, D, seed=41, kind="normal", scale=1.0)
    rng = np.random.default_rng(41)
    sample = np.unique(np.concatenate([[0, 1, 127, 128, N - 129, N - 1], rng.choice(N, 10, replace=False)]))
    run_and_check(q, k, v, 1.0 / math.sqrt(D), [(0, 0, N - 64, 64)], sample.astype(np.int64),
                  "long head causal=%d fp8pv=%d" % (causal, fp8pv), causal=causal, fp8pv=fp8pv)
