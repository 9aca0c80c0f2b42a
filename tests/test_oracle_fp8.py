"""Pins for the oracle's FP8 P/V variant ("Hardware-Aware FP4 FlashAttention-4",
"What the paper found": training keeps FP8 probabilities and values): MXFP8
(E4M3) V along keys and Direct-P with E4M3 probability codes.

Checked against: hand-worked blocks and rows (tests/golden/mxfp8_block.json,
tests/golden/directp_rows_fp8.json); the scale rule's invariant
amax <= 448 * 2^e < 2 * amax and the E4M3 half-step error bound; a numpy
P-hat @ V-hat recomputation that decodes the payload independently; the
row invariants (p/l sums to one, integer-shift invariance, all-equal scores
give the mean of V-hat and LSE = ln N); and closeness to fp64 softmax
attention, which FP8 operands must meet more tightly than FP4.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from blackwell_nvfp4_quantize_gb300 import workloads as wl


def _e4m3(code):
    code = int(code)
    e, m = (code >> 3) & 15, code & 7
    v = m * 2.0 ** -9 if e == 0 else (8 + m) * 2.0 ** (e - 10)
    return -v if code & 0x80 else v


def _e4m3_vec(codes):
    return np.array([_e4m3(c) for c in np.asarray(codes).reshape(-1)]).reshape(np.asarray(codes).shape)


def _hex(xs):
    return [int(x, 16) if isinstance(x, str) and x.startswith("0x") else int(x) for x in xs]


def test_mxfp8_block_hand_worked(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "mxfp8_block.json")))
    B, H, N, D = g["shape"]
    v = np.array(_hex(g["v_bf16_bits"]), dtype=np.uint16).reshape(B, H, N, D)
    payload, sf = oracle.quant_mxfp8_v(v)
    assert payload.shape == (1, 1, 1, 128)
    assert payload[0, 0, 0, :64].tolist() == _hex(g["codes_first_64"])
    assert np.all(payload[0, 0, 0, 64:] == 0)
    assert sf[:4].tolist() == g["scale_bytes_row0"]
    assert np.all(sf[4:] == 0)


def test_mxfp8_scale_rule_and_error_bound():
    q, k, v = wl.make_custom(1, 2, 200, 64, seed=81, scale=3.0)
    vb = wl.bf16_bits(v)
    payload, sf = oracle.quant_mxfp8_v(vb)
    vf = v.float().numpy()
    npad = 256
    for bh in range(2):
        for d in range(0, 64, 7):
            for kb in range(npad // 32):
                atom = bh * (npad // 128) + kb // 4
                e = int(sf[atom * 512 + (d % 32) * 16 + (d // 32) * 4 + kb % 4]) - 127
                blk = vf.reshape(2, 200, 64)[bh, kb * 32:min(200, kb * 32 + 32), d]
                codes = payload.reshape(2, 64, npad)[bh, d, kb * 32:kb * 32 + 32]
                if blk.size == 0:
                    assert e == -127 and np.all(codes == 0)
                    continue
                amax = float(np.abs(blk).max())
                if amax > 0:
                    assert amax <= 448.0 * 2.0 ** e < 2 * amax
                vhat = _e4m3_vec(codes[:blk.size]) * 2.0 ** e
                # round to nearest: within half a step of E4M3 at the value's binade
                step = np.where(np.abs(blk) >= 2.0 ** (e - 6), 2.0 ** (np.floor(np.log2(np.maximum(np.abs(blk), 1e-30))) - 3),
                                2.0 ** (e - 9))
                assert np.all(np.abs(vhat - blk) <= 0.5 * step + 1e-12)


def test_fp8_map_row_hand_worked(golden_dir):
    g = json.load(open(os.path.join(golden_dir, "directp_rows_fp8.json")))
    for row in g["rows"]:
        codes, ks, m, l = oracle.directp_map_row(np.array(row["s"], dtype=np.float32), row["c"],
                                                 pv_fmt=oracle.PV_MXFP8)
        assert codes.tolist() == row["codes"], row["name"]
        assert ks.tolist() == row["kshift"], row["name"]
        assert m == row["M"], row["name"]
        assert l == pytest.approx(row["l"], rel=1e-15, abs=0), row["name"]


def test_fp8_map_row_properties():
    rng = np.random.default_rng(5)
    for _ in range(40):
        n = int(rng.integers(1, 160))
        s = (rng.standard_normal(n) * rng.uniform(0.1, 20)).astype(np.float32)
        c = float(rng.uniform(0.05, 2.0))
        codes, ks, m, l = oracle.directp_map_row(s, c, pv_fmt=oracle.PV_MXFP8)
        x = (np.float32(c) * s).astype(np.float32)
        for b in range((n + 31) // 32):
            blk = slice(b * 32, min(n, b * 32 + 32))
            top = 2.0 ** (float(x[blk].max()) - ks[b])
            assert 224.0 * (1 - 1e-6) < top <= 448.0 * (1 + 1e-6)
            order = np.argsort(x[blk], kind="stable")
            assert np.all(np.diff(codes[blk][order].astype(int)) >= 0)
        p = _e4m3_vec(codes) * np.repeat(2.0 ** np.maximum(ks - m, -127), 32)[:n]
        assert abs(p.sum() - l) <= 1e-12 * l
        assert 0.45 < p.max() <= 1.0 + 1e-12
    s = (rng.standard_normal(70) * 4).astype(np.float32)
    c0, k0, m0, l0 = oracle.directp_map_row(s, 1.0, pv_fmt=oracle.PV_MXFP8)
    for shift in (-5, 2, 30):
        c1, k1, m1, l1 = oracle.directp_map_row(s + np.float32(shift), 1.0, pv_fmt=oracle.PV_MXFP8)
        assert np.array_equal(c0, c1) and np.array_equal(k1, k0 + shift) and m1 == m0 + shift and l1 == l0


def _quant8(q, k, v):
    qb, kb, vb = (wl.bf16_bits(t) for t in (q, k, v))
    return oracle.quant_nvfp4(qb), oracle.quant_nvfp4(kb), oracle.quant_mxfp8_v(vb)


def _decode_nvfp4_rows(payload, sf, N, D, bh):
    e2m1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    rows = payload.reshape(-1, D // 2)[bh * N:(bh + 1) * N]
    codes = np.empty((N, D), dtype=np.uint8)
    codes[:, 0::2] = rows & 0xF
    codes[:, 1::2] = rows >> 4
    vals = np.where(codes & 8, -1.0, 1.0) * e2m1[codes & 7]
    out = np.empty((N, D))
    for n in range(N):
        sc = [_e4m3(sf[oracle.sf_index(bh, (N + 127) // 128, n, kb, D // 16)]) for kb in range(D // 16)]
        out[n] = vals[n] * np.repeat(sc, 16)
    return out


@pytest.mark.parametrize("causal", [False, True])
def test_fp8_stage_b_recomputation(causal):
    N, D = 150, 64
    q, k, v = wl.make_custom(1, 1, N, D, seed=91, scale=1.5)
    qq, kq, vq = _quant8(q, k, v)
    res = oracle.directp_rows(qq, kq, vq, (1, 1, N, D), 0.125, np.arange(N), want_codes=True, causal=causal,
                              pv_fmt=oracle.PV_MXFP8)
    npad = 256
    vcodes = vq[0].reshape(D, npad)[:, :N]
    vsc = np.array([[2.0 ** (int(vq[1][(n // 128) * 512 + (d % 32) * 16 + (d // 32) * 4 + (n % 128) // 32]) - 127)
                     for n in range(N)] for d in range(D)])
    vhat = (_e4m3_vec(vcodes) * vsc).T  # [N, D]
    qhat = _decode_nvfp4_rows(qq[0], qq[1], N, D, 0)
    khat = _decode_nvfp4_rows(kq[0], kq[1], N, D, 0)
    c = np.float32(0.125 * 1.4426950408889634 * float(qq[2]) * float(kq[2]))
    for i in range(0, N, 7):
        nk = i + 1 if causal else N
        e = np.maximum(res["kshift"][i] - res["m"][i], -127)
        p = _e4m3_vec(res["codes"][i][:nk]) * np.repeat(2.0 ** e, 32)[:nk]
        assert np.all(res["codes"][i][nk:] == 0)
        l = p.sum()
        assert np.max(np.abs(res["o"][i] - p @ vhat[:nk] / l)) < 1e-12
        assert abs(res["lse"][i] - math.log(2) * (res["m"][i] + math.log2(l))) < 1e-12
        s32 = (khat[:nk] @ qhat[i]).astype(np.float32)
        assert res["m"][i] == math.ceil(float((c * s32).astype(np.float32).max()))


def test_fp8_all_equal_scores_give_mean_of_v():
    # Q = 0: every score 0, M = 0, K_b = ceil(-log2 448) = -8, code E4M3(256) = 0x78, p = 1
    N, D = 200, 64
    q, k, v = wl.make_custom(1, 1, N, D, seed=5, kind="zero_q")
    qq, kq, vq = _quant8(q, k, v)
    res = oracle.directp_rows(qq, kq, vq, (1, 1, N, D), 0.125, np.arange(N), want_codes=True,
                              pv_fmt=oracle.PV_MXFP8)
    assert np.all(res["codes"][:, :N] == 0x78) and np.all(res["m"] == 0)
    assert np.all(res["kshift"][:, :7] == -8)
    npad = 256
    vcodes = vq[0].reshape(D, npad)[:, :N]
    vsc = np.array([[2.0 ** (int(vq[1][(n // 128) * 512 + (d % 32) * 16 + (d // 32) * 4 + (n % 128) // 32]) - 127)
                     for n in range(N)] for d in range(D)])
    vhat = (_e4m3_vec(vcodes) * vsc).T
    assert np.max(np.abs(res["o"] - vhat.mean(axis=0)[None, :])) < 1e-12
    assert np.max(np.abs(res["lse"] - math.log(N))) < 1e-12


def test_fp8_closer_to_exact_attention_than_fp4():
    B, H, N, D = 1, 2, 256, 64
    q, k, v = wl.make_custom(B, H, N, D, seed=8)
    qb, kb, vb = (wl.bf16_bits(t) for t in (q, k, v))
    qq, kq = oracle.quant_nvfp4(qb), oracle.quant_nvfp4(kb)
    rows = np.arange(B * H * N, dtype=np.int64)
    r8 = oracle.directp_rows(qq, kq, oracle.quant_mxfp8_v(vb), (B, H, N, D), 0.125, rows, pv_fmt=oracle.PV_MXFP8)
    r4 = oracle.directp_rows(qq, kq, oracle.quant_mxfp4_v(vb), (B, H, N, D), 0.125, rows)
    o_ex, _ = oracle.exact_rows(qb, kb, vb, 0.125, rows)
    err8 = np.linalg.norm(r8["o"] - o_ex) / np.linalg.norm(o_ex)
    err4 = np.linalg.norm(r4["o"] - o_ex) / np.linalg.norm(o_ex)
    # the NVFP4 scores dominate both errors; FP8 P and V still remove a good part
    assert err8 < 0.8 * err4 and err8 < 0.2
