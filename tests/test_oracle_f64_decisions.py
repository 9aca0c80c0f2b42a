"""The oracle's two readings of the Direct-P decisions.

The fp32-decision reading (orc_directp_map_row) rounds S, c, X = c*S and
t = X - K_b to fp32, as the forward kernel computes them; the fp64-decision
reading (orc_directp_map_row_f64) keeps them in fp64 -- the plain reading of
"What the paper found" (log-softmax scores mapped directly to E2M1 codes).
Both are pinned here against each other through what the mathematics fixes:
they may differ only where fp32 rounding moves a value across a decision
threshold, so every difference must sit within a few fp32 roundings of one:
  * a block shift K_b = ceil(X_b - log2 6): X_b - log2 6 next to an integer;
  * the row maximum M = ceil(max X): max X next to an integer;
  * a code E2M1(2^t): t next to log2 of a rounding boundary of E2M1
    (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5), when both readings used the same K_b.
"""
import math

import numpy as np
import pytest

import oracle

LOG2_6 = math.log2(6.0)
BOUNDS = np.log2(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]))
U32 = 2.0 ** -24  # unit roundoff of fp32


def _near_int(x, tol):
    return abs(x - round(x)) <= tol


def _check_row(s32, c32):
    codes32, ks32, m32, _ = oracle.directp_map_row(s32, c32)
    s64 = s32.astype(np.float64)
    c64 = float(c32)
    codes64, ks64, m64, _ = oracle.directp_map_row_f64(s64, c64)
    x = c64 * s64
    n = s32.shape[0]
    ndiff = 0
    if m32 != m64:
        assert _near_int(x.max(), 4 * U32 * (abs(x.max()) + 1)), (m32, m64, x.max())
    for b in range((n + 31) // 32):
        j0, j1 = 32 * b, min(n, 32 * b + 32)
        xb = x[j0:j1].max()
        if ks32[b] != ks64[b]:
            assert _near_int(xb - LOG2_6, 4 * U32 * (abs(xb) + 4)), (b, ks32[b], ks64[b], xb)
            ndiff += int(np.sum(codes32[j0:j1] != codes64[j0:j1]))
            continue
        t = x[j0:j1] - ks64[b]
        d = codes32[j0:j1] != codes64[j0:j1]
        if np.any(d):
            dist = np.min(np.abs(t[d, None] - BOUNDS[None, :]), axis=1)
            tol = 4 * U32 * (np.abs(x[j0:j1][d]) + abs(ks64[b]) + 4)
            assert np.all(dist <= tol), (b, t[d], dist, tol)
            ndiff += int(np.sum(d))
    return ndiff


@pytest.mark.parametrize("sigma", [0.5, 3.0, 20.0, 300.0])
def test_fp32_and_fp64_decisions_differ_only_at_thresholds(sigma):
    rng = np.random.default_rng(int(sigma * 10))
    total = diff = 0
    for _ in range(40):
        n = int(rng.integers(1, 1025))
        s32 = (rng.standard_normal(n) * sigma).astype(np.float32)
        c32 = np.float32(rng.uniform(0.05, 0.5))
        diff += _check_row(s32, c32)
        total += n
    # differences are confined to rounding neighbourhoods of the thresholds: rare
    assert diff <= max(2, total // 10000), (diff, total)


def test_decisions_equal_on_exactly_representable_rows():
    # c a power of two and small-integer scores: every product and difference
    # is exact in fp32, so the two readings must agree on everything
    rng = np.random.default_rng(5)
    for _ in range(20):
        s32 = rng.integers(-200, 200, size=300).astype(np.float32)
        c32 = np.float32(0.125)
        codes32, ks32, m32, l32 = oracle.directp_map_row(s32, c32)
        codes64, ks64, m64, l64 = oracle.directp_map_row_f64(s32.astype(np.float64), float(c32))
        assert np.array_equal(codes32, codes64) and np.array_equal(ks32, ks64) and m32 == m64 and l32 == l64


def test_fp64_reading_decides_by_the_fp64_value_at_a_boundary():
    # block maximum 2.0 (c = 1): K_b = ceil(2 - log2 6) = 0, so t = s.  Scores
    # a hair above / below log2(1.25) -- closer than fp32 can resolve -- map to
    # 1.5 (code 3) / 1.0 (code 2) under the fp64 reading.
    a = math.log2(1.25)
    for eps, code in ((1e-12, 3), (-1e-12, 2)):
        codes, ks, m, _ = oracle.directp_map_row_f64(np.array([2.0, a + eps]), 1.0)
        assert ks[0] == 0 and m == 2
        assert codes[1] == code, (eps, codes)
    # the fp32 reading sees the same two scores as one fp32 value
    assert np.float32(a + 1e-12) == np.float32(a - 1e-12)


def test_full_rows_two_readings_agree_on_quantized_operands():
    # the whole row pass (quantized Q, K, V of a small workload) under both
    # readings: codes and block shifts agree almost everywhere, O and LSE agree
    # to within the effect of the few flipped codes
    from blackwell_nvfp4_quantize_gb300 import workloads as wl

    q, k, v = wl.make_custom(1, 2, 700, 128, seed=31, kind="normal", scale=1.5)
    qq = oracle.quant_nvfp4(wl.bf16_bits(q))
    kq = oracle.quant_nvfp4(wl.bf16_bits(k))
    vq = oracle.quant_mxfp4_v(wl.bf16_bits(v))
    rows = np.arange(2 * 700, dtype=np.int64)
    shape = (1, 2, 700, 128)
    r32 = oracle.directp_rows(qq, kq, vq, shape, 1 / math.sqrt(128), rows, want_codes=True)
    r64 = oracle.directp_rows(qq, kq, vq, shape, 1 / math.sqrt(128), rows, want_codes=True, f64_decisions=True)
    agree = np.mean(r32["codes"][:, :700] == r64["codes"][:, :700])
    kagree = np.mean(r32["kshift"] == r64["kshift"])
    print("fp32 vs fp64 decisions: codes agree %.7f, kshift agree %.7f" % (agree, kagree))
    assert agree >= 0.9999 and kagree >= 0.9999
    assert np.max(np.abs(r32["lse"] - r64["lse"])) < 1e-3
    assert np.max(np.abs(r32["o"] - r64["o"])) < 2e-2
