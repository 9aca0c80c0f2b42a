"""Pins for the oracle's causal rows (the causal forward of "Hardware-Aware FP4
FlashAttention-4", "What the paper found": query i sees keys 0..i).

Checked against: a library softmax-attention (scipy) under the causal mask
for the unquantized pass; and, for Direct-P, facts the mask fixes without
reference to the oracle's arithmetic -- the last row sees every key, so it
equals the noncausal row; row 0 sees only key 0, so its output is v-hat_0
exactly; and a row sees nothing past itself, so it equals the last row of the
same sequence cut right after it (quantized identically by planting the
tensor-wide maximum in row 0 and cutting on a V block boundary).
"""
import math

import numpy as np
import pytest
import scipy.special

import oracle
from blackwell_nvfp4_quantize_gb300 import workloads as wl

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _dec_codes(codes):
    codes = np.asarray(codes)
    v = E2M1[codes & 7]
    return np.where(codes & 8, -v, v)


def _quant(qb, kb, vb):
    return oracle.quant_nvfp4(qb), oracle.quant_nvfp4(kb), oracle.quant_mxfp4_v(vb)


def _decode_v_row0(vq, N, D, bh):
    npad = (N + 127) // 128 * 128
    pay = vq[0].reshape(-1, npad // 2)
    out = np.empty(D)
    for d in range(D):
        code = int(pay[bh * D + d][0] & 0xF)
        e = int(vq[1][(bh * (npad // 128)) * 512 + (d % 32) * 16 + (d // 32) * 4]) - 127
        out[d] = _dec_codes(code) * 2.0 ** e
    return out


def test_causal_stage_a_equals_library_softmax_attention():
    q, k, v = wl.make_custom(1, 2, 80, 64, seed=31, scale=2.0)
    qb, kb, vb = (wl.bf16_bits(t) for t in (q, k, v))
    B, H, N, D = q.shape
    ss = 1.0 / math.sqrt(D)
    rows = np.arange(B * H * N, dtype=np.int64)
    o, lse = oracle.exact_rows(qb, kb, vb, ss, rows, causal=True)
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    logits = ss * np.einsum("bhnd,bhmd->bhnm", qd, kd)
    logits = np.where(np.tril(np.ones((N, N), dtype=bool)), logits, -np.inf)
    p = scipy.special.softmax(logits, axis=-1)
    o_ref = np.einsum("bhnm,bhmd->bhnd", p, vd).reshape(-1, D)
    lse_ref = scipy.special.logsumexp(logits, axis=-1).reshape(-1)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12
    # and the mask matters: the noncausal rows differ
    o_nc, _ = oracle.exact_rows(qb, kb, vb, ss, rows)
    assert np.max(np.abs(o - o_nc)) > 1e-2


@pytest.mark.parametrize("N,D", [(200, 64), (256, 128)])
def test_causal_last_row_equals_noncausal(N, D):
    q, k, v = wl.make_custom(1, 2, N, D, seed=40 + N, scale=1.5)
    qq, kq, vq = _quant(*(wl.bf16_bits(t) for t in (q, k, v)))
    ss = 1.0 / math.sqrt(D)
    rows = np.array([N - 1, 2 * N - 1], dtype=np.int64)
    a = oracle.directp_rows(qq, kq, vq, (1, 2, N, D), ss, rows, want_codes=True, causal=True)
    b = oracle.directp_rows(qq, kq, vq, (1, 2, N, D), ss, rows, want_codes=True)
    for key in ("o", "lse", "codes", "kshift", "m"):
        assert np.array_equal(a[key], b[key]), key


@pytest.mark.parametrize("D", [64, 128])
def test_causal_row0_returns_vhat0(D):
    N = 150
    q, k, v = wl.make_custom(1, 2, N, D, seed=50 + D, scale=3.0)
    qq, kq, vq = _quant(*(wl.bf16_bits(t) for t in (q, k, v)))
    rows = np.array([0, N], dtype=np.int64)
    r = oracle.directp_rows(qq, kq, vq, (1, 2, N, D), 0.125, rows, want_codes=True, causal=True)
    npad = (N + 127) // 128 * 128
    for u, bh in enumerate((0, 1)):
        assert np.all(r["codes"][u][1:] == 0) and np.all(r["kshift"][u][1:] == 0)
        # one key: its probability is the whole row, O is that key's value
        assert np.array_equal(r["o"][u], _decode_v_row0(vq, N, D, bh))
        code0 = int(r["codes"][u][0])
        assert code0 in (5, 6, 7)  # 2^(X - K_0) lies in (3, 6]
        l = _dec_codes(code0) * 2.0 ** max(int(r["kshift"][u][0]) - int(r["m"][u]), -127)
        assert r["lse"][u] == pytest.approx(math.log(2) * (int(r["m"][u]) + math.log2(l)), abs=1e-12)
    assert npad == 256


@pytest.mark.parametrize("D", [64, 128])
def test_causal_row_equals_last_row_of_cut_sequence(D):
    N, H = 200, 2
    q, k, v = wl.make_custom(1, H, N, D, seed=60 + D, scale=1.0)
    # the tensor-wide maxima of Q and K sit in row 0 of head 0, so a cut
    # sequence keeps the same tensor scales
    q[0, 0, 0, 0] = 40.0
    k[0, 0, 0, 1] = -40.0
    qb, kb, vb = (wl.bf16_bits(t) for t in (q, k, v))
    ss = 1.0 / math.sqrt(D)
    full_q, full_k, full_v = _quant(qb, kb, vb)
    for cut in (32, 96, 160):  # multiples of the 32-key V block
        cq, ck, cv = _quant(*(np.ascontiguousarray(t[:, :, :cut]) for t in (qb, kb, vb)))
        assert cq[2] == full_q[2] and ck[2] == full_k[2]
        rows_full = np.array([h * N + i for h in range(H) for i in range(cut)], dtype=np.int64)
        rows_cut = np.array([h * cut + i for h in range(H) for i in range(cut)], dtype=np.int64)
        a = oracle.directp_rows(full_q, full_k, full_v, (1, H, N, D), ss, rows_full, want_codes=True,
                                causal=True)
        b = oracle.directp_rows(cq, ck, cv, (1, H, cut, D), ss, rows_cut, want_codes=True, causal=True)
        assert np.array_equal(a["o"], b["o"]) and np.array_equal(a["lse"], b["lse"])
        assert np.array_equal(a["m"], b["m"])
        assert np.array_equal(a["codes"][:, :cut], b["codes"][:, :cut])
        assert np.all(a["codes"][:, cut:] == 0)
        assert np.array_equal(a["kshift"][:, :cut // 32], b["kshift"][:, :cut // 32])
        # the last row of the cut sequence sees all its keys: the noncausal row
        last = np.array([h * cut + cut - 1 for h in range(H)], dtype=np.int64)
        c = oracle.directp_rows(cq, ck, cv, (1, H, cut, D), ss, last, want_codes=True)
        sel = [h * cut + cut - 1 for h in range(H)]
        assert np.array_equal(a["o"][sel], c["o"]) and np.array_equal(a["lse"][sel], c["lse"])


def test_causal_rows_normalised_and_masked():
    N, D = 170, 64
    q, k, v = wl.make_custom(1, 1, N, D, seed=71, scale=2.0)
    qq, kq, vq = _quant(*(wl.bf16_bits(t) for t in (q, k, v)))
    r = oracle.directp_rows(qq, kq, vq, (1, 1, N, D), 0.125, np.arange(N), want_codes=True, causal=True)
    for i in range(N):
        codes = r["codes"][i]
        assert np.all(codes[i + 1:] == 0)
        assert np.all(r["kshift"][i][(i // 32) + 1:] == 0)
        e = np.maximum(r["kshift"][i] - r["m"][i], -127)
        p = _dec_codes(codes[:i + 1]) * np.repeat(2.0 ** e, 32)[:i + 1]
        assert abs(r["lse"][i] - math.log(2) * (r["m"][i] + math.log2(p.sum()))) < 1e-12
        assert p.max() <= 1.0 + 1e-12 and p.max() > 0.4
