"""Pins for the oracle's Direct-P attention rows.

Checked against: hand-worked score rows (tests/golden/directp_rows.json); a
library softmax-attention (scipy) for the unquantized pass (Stage A); a numpy
P-hat @ V-hat recomputation from the oracle's own codes and the decoded
quantized operands (Stage B); the invariants the method states or implies
(rows of p/l sum to 1, codes invariant under an integer shift of all scores,
all-equal scores give the mean of V and LSE = ln N).
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from blackwell_nvfp4_quantize_gb300 import workloads as wl

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _dec_codes(codes):
    codes = np.asarray(codes)
    v = E2M1[codes & 7]
    return np.where(codes & 8, -v, v)


def _unpack(payload_row, n):
    b = np.asarray(payload_row)
    out = np.empty(b.size * 2, dtype=np.uint8)
    out[0::2] = b & 0xF
    out[1::2] = b >> 4
    return out[:n]


def test_map_row_hand_worked(golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "directp_rows.json")))
    for row in gold["rows"]:
        codes, ks, m, l = oracle.directp_map_row(np.array(row["s"], dtype=np.float32), row["c"])
        assert codes.tolist() == row["codes"], row["name"]
        assert ks.tolist() == row["kshift"], row["name"]
        assert m == row["M"], row["name"]
        assert l == row["l"], row["name"]


def test_map_row_integer_shift_invariance():
    rng = np.random.default_rng(3)
    s = (rng.standard_normal(96) * 3).astype(np.float32)
    c0, k0, m0, l0 = oracle.directp_map_row(s, 1.0)
    for shift in (-7, 1, 5, 40):
        c1, k1, m1, l1 = oracle.directp_map_row(s + np.float32(shift), 1.0)
        assert np.array_equal(c0, c1)
        assert np.array_equal(k1, k0 + shift)
        assert m1 == m0 + shift and l1 == l0


def test_map_row_properties():
    rng = np.random.default_rng(4)
    for trial in range(50):
        n = int(rng.integers(1, 200))
        s = (rng.standard_normal(n) * rng.uniform(0.1, 20)).astype(np.float32)
        c = float(rng.uniform(0.05, 2.0))
        codes, ks, m, l = oracle.directp_map_row(s, c)
        x = (np.float32(c) * s).astype(np.float32)
        assert m == math.ceil(float(x.max()))
        for b in range((n + 31) // 32):
            blk = slice(b * 32, min(n, b * 32 + 32))
            # no-clip block shift: largest probability of the block within 6, and > 3
            top = 2.0 ** (float(x[blk].max()) - ks[b])
            assert 3.0 - 1e-5 < top <= 6.0 + 1e-5
            # codes are monotone in the score within a block
            order = np.argsort(x[blk], kind="stable")
            assert np.all(np.diff(codes[blk][order].astype(int)) >= 0)
            assert codes[blk].max() >= 5  # block max maps to 3, 4 or 6
        # the row maximum has probability in (1/2, 1]: p = dec*2^(K-M)
        p = _dec_codes(codes) * np.repeat(2.0 ** np.maximum(ks - m, -127), 32)[:n]
        assert abs(p.sum() - l) <= 1e-12 * l
        assert 0.4 < p.max() <= 1.0 + 1e-12


def _small_problem(seed, B=1, H=2, N=160, D=64, kind="normal", scale=1.0):
    q, k, v = wl.make_custom(B, H, N, D, seed=seed, kind=kind, scale=scale)
    qb, kb, vb = (wl.bf16_bits(t) for t in (q, k, v))
    return (q, k, v), (qb, kb, vb)


def test_stage_a_exact_equals_library_softmax_attention():
    (q, k, v), (qb, kb, vb) = _small_problem(11, B=2, H=2, N=96, D=64, scale=2.0)
    B, H, N, D = q.shape
    ss = 1.0 / math.sqrt(D)
    rows = np.arange(B * H * N, dtype=np.int64)
    o, lse = oracle.exact_rows(qb, kb, vb, ss, rows)
    qd, kd, vd = (t.double().numpy() for t in (q, k, v))
    logits = ss * np.einsum("bhnd,bhmd->bhnm", qd, kd)
    p = scipy.special.softmax(logits, axis=-1)
    o_ref = np.einsum("bhnm,bhmd->bhnd", p, vd).reshape(-1, D)
    lse_ref = scipy.special.logsumexp(logits, axis=-1).reshape(-1)
    assert np.max(np.abs(o - o_ref)) < 1e-12
    assert np.max(np.abs(lse - lse_ref)) < 1e-12


def _decode_nvfp4(payload, sf, N, D, bh, n):
    codes = _unpack(payload.reshape(-1, D // 2)[bh * N + n], D)
    scales = np.array([oracle.e4m3_decode(int(sf[oracle.sf_index(bh, (N + 127) // 128, n, kb, D // 16)]))
                       for kb in range(D // 16)])
    return _dec_codes(codes) * np.repeat(scales, 16)


def _decode_v(payload_t, sf, N, D, bh):
    npad = (N + 127) // 128 * 128
    out = np.zeros((N, D))
    for d in range(D):
        codes = _unpack(payload_t.reshape(-1, npad // 2)[bh * D + d], npad)[:N]
        sc = np.array([2.0 ** (int(sf[(bh * (npad // 128) + n // 128) * 512 + (d % 32) * 16 + (d // 32) * 4
                                      + (n % 128) // 32]) - 127) for n in range(N)])
        out[:, d] = _dec_codes(codes) * sc
    return out


@pytest.mark.parametrize("N,D", [(160, 64), (256, 128), (77, 64)])
def test_stage_b_phat_vhat_recomputation(N, D):
    (q, k, v), (qb, kb, vb) = _small_problem(21 + N, B=1, H=2, N=N, D=D, scale=1.5)
    B, H = 1, 2
    qq = oracle.quant_nvfp4(qb)
    kq = oracle.quant_nvfp4(kb)
    vq = oracle.quant_mxfp4_v(vb)
    ss = 1.0 / math.sqrt(D)
    rows = np.arange(B * H * N, dtype=np.int64)
    res = oracle.directp_rows(qq, kq, vq, (B, H, N, D), ss, rows, want_codes=True)
    npad = (N + 127) // 128 * 128
    for bh in range(B * H):
        vhat = _decode_v(vq[0], vq[1], N, D, bh)
        khat = np.stack([_decode_nvfp4(kq[0], kq[1], N, D, bh, n) for n in range(N)])
        for i in range(N):
            r = bh * N + i
            qhat = _decode_nvfp4(qq[0], qq[1], N, D, bh, i)
            codes = res["codes"][r][:N]
            assert np.all(res["codes"][r][N:] == 0)
            e = np.maximum(res["kshift"][r] - res["m"][r], -127)
            p = _dec_codes(codes) * np.repeat(2.0 ** e, 32)[:N]
            l = p.sum()
            assert abs(res["lse"][r] - math.log(2) * (res["m"][r] + math.log2(l))) < 1e-12
            o_ref = p @ vhat / l
            assert np.max(np.abs(res["o"][r] - o_ref)) < 1e-12
            # rows of p / l sum to one
            assert abs((p / l).sum() - 1.0) < 1e-12
            # the scores behind the codes: M is the ceiling of the largest scaled score
            c = np.float32(ss * 1.4426950408889634 * float(qq[2]) * float(kq[2]))
            s32 = (khat @ qhat).astype(np.float32)
            assert res["m"][r] == math.ceil(float((c * s32).astype(np.float32).max()))
        assert npad % 128 == 0


def test_all_equal_scores_give_mean_of_v():
    # Q = 0 makes every score 0: M = 0, K_b = -2, every code is 6 (4.0) at scale 2^-2, p = 1.
    (q, k, v), (qb, kb, vb) = _small_problem(5, B=1, H=1, N=200, D=64, kind="zero_q")
    N, D = 200, 64
    qq, kq, vq = oracle.quant_nvfp4(qb), oracle.quant_nvfp4(kb), oracle.quant_mxfp4_v(vb)
    res = oracle.directp_rows(qq, kq, vq, (1, 1, N, D), 0.125, np.arange(N), want_codes=True)
    vhat = _decode_v(vq[0], vq[1], N, D, 0)
    assert np.all(res["codes"][:, :N] == 6)
    assert np.all(res["m"] == 0) and np.all(res["kshift"][:, :7] == -2)
    assert np.max(np.abs(res["o"] - vhat.mean(axis=0)[None, :])) < 1e-12
    assert np.max(np.abs(res["lse"] - math.log(N))) < 1e-12


def test_quantized_close_to_exact_attention():
    # report-style sanity: FP4 attention stays near fp64 softmax attention
    (q, k, v), (qb, kb, vb) = _small_problem(8, B=1, H=2, N=256, D=64)
    B, H, N, D = 1, 2, 256, 64
    qq, kq, vq = oracle.quant_nvfp4(qb), oracle.quant_nvfp4(kb), oracle.quant_mxfp4_v(vb)
    rows = np.arange(B * H * N, dtype=np.int64)
    res = oracle.directp_rows(qq, kq, vq, (B, H, N, D), 0.125, rows)
    o_ex, lse_ex = oracle.exact_rows(qb, kb, vb, 0.125, rows)
    cos = np.sum(res["o"] * o_ex) / (np.linalg.norm(res["o"]) * np.linalg.norm(o_ex))
    assert cos > 0.95
    assert np.max(np.abs(res["lse"] - lse_ex)) < 0.5
