"""Pins of the backward oracle (CPU): FP8 formats, MX block scaling, the
backward operands' quantizers and layouts, and the backward itself against
automatic differentiation.

The method: "Hardware-Aware FP4 FlashAttention-4", summary page, "What the
paper found" -- for causal training the backward reconstructs the
probabilities from the saved quantized Q/K and LSE and uses FP8 gradient
operands, including E5M2 output gradients.
"""
import json
import os

import numpy as np
import pytest
import torch

import oracle
import oracle.bwd as ob

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


# ---- formats ---------------------------------------------------------------

def test_e5m2_hand_worked_cases():
    d = json.load(open(os.path.join(GOLDEN, "e5m2_cases.json")))
    for c in d["cases"]:
        y = np.float32(c["y"])
        assert int(ob.fp8_encode(y, ob.E5M2)) == c["code"], c
        if c["code"] not in (123, 251) or abs(c["y"]) == 57344.0:
            # away from saturation the decoded value is the nearest one
            assert ob.fp8_decode(c["code"], ob.E5M2) == ob.fp8_round(y, ob.E5M2)


def test_e4m3_encoder_matches_the_c_oracle():
    # the C oracle's E4M3 encoder is pinned by its own hand-worked cases;
    # this numpy restatement must agree with it on a dense grid
    rng = np.random.default_rng(5)
    ys = np.concatenate([rng.standard_normal(4000) * s for s in (1e-3, 1e-1, 1, 30, 300, 1000)])
    ys = np.concatenate([ys, [0.0, -0.0, 448.0, 464.0, 480.0, -1e6, 2.0 ** -9, 2.0 ** -10, 1.5 * 2.0 ** -10]])
    ys = ys.astype(np.float32)
    got = ob.fp8_encode(ys, ob.E4M3)
    want = np.array([oracle.e4m3_encode(float(y)) for y in ys], dtype=np.uint8)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt,tdtype,vmax", [(0, torch.float8_e4m3fn, 448.0), (1, torch.float8_e5m2, 57344.0)])
def test_fp8_round_matches_torch_casts(fmt, tdtype, vmax):
    # torch's float8 casts round to nearest even inside the finite range
    rng = np.random.default_rng(11 + fmt)
    ys = np.concatenate([rng.standard_normal(20000) * s for s in (2.0 ** -20, 2.0 ** -12, 2.0 ** -6, 1, 64, vmax / 8)])
    # every midpoint between neighbouring codes, where ties decide
    codes = np.arange(256, dtype=np.uint8)
    vals = ob.fp8_decode(codes, fmt)
    fin = np.isfinite(vals) & (np.abs(vals) <= vmax)
    pos = np.unique(vals[fin & (vals >= 0)])
    mids = (pos[1:] + pos[:-1]) / 2
    ys = np.concatenate([ys, mids, -mids]).astype(np.float32)
    ys = ys[np.abs(ys) <= vmax]
    want = torch.from_numpy(ys).to(tdtype).to(torch.float64).numpy()
    got = ob.fp8_round(ys, fmt)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", [ob.E4M3, ob.E5M2])
def test_fp8_code_round_trip(fmt):
    codes = np.arange(256, dtype=np.uint8)
    vals = ob.fp8_decode(codes, fmt)
    ok = np.isfinite(vals) & (np.abs(vals) <= (448.0 if fmt == ob.E4M3 else 57344.0))
    if fmt == ob.E4M3:
        ok &= (codes & 0x7F) != 0x7F  # E4M3FN NaN codes
    else:
        ok &= ((codes >> 2) & 31) != 31  # E5M2 infinities / NaN
    assert np.array_equal(ob.fp8_encode(vals[ok], fmt), codes[ok])


@pytest.mark.parametrize("fmt,vmax", [(ob.E4M3, 448.0), (ob.E5M2, 57344.0)])
def test_mx_exponent_is_the_smallest_no_clip_scale(fmt, vmax):
    rng = np.random.default_rng(3)
    a = np.exp(rng.uniform(-80, 80, 50000))
    a = np.concatenate([a, vmax * 2.0 ** np.arange(-20, 20), np.nextafter(vmax * 2.0 ** np.arange(-20, 20), np.inf)])
    e = ob.mx_exponent(a, fmt)
    assert np.all(a <= vmax * np.ldexp(1.0, e))
    inner = e > -127
    assert np.all(a[inner] > vmax * np.ldexp(1.0, e[inner] - 1))
    assert ob.mx_exponent(0.0, fmt) == -127


# ---- quantizers and layouts -----------------------------------------------

@pytest.mark.parametrize("N", [128, 200, 384])
def test_transposed_e4m3_quantizer_matches_the_c_oracle(N):
    rng = np.random.default_rng(N)
    x = rng.standard_normal((2, 2, N, 64)).astype(np.float32) * np.exp(rng.uniform(-3, 3, (2, 2, 1, 64)))
    bits = _bf16_bits(x)
    codes, sf, vals = ob.quant_mxfp8_t(bits, ob.E4M3)
    c_codes, c_sf = oracle.quant_mxfp8_v(bits)
    assert np.array_equal(codes, c_codes)
    assert np.array_equal(sf, c_sf)


@pytest.mark.parametrize("fmt,vmax,half_step", [(ob.E4M3, 448.0, 2.0 ** -4), (ob.E5M2, 57344.0, 2.0 ** -3)])
def test_row_quantizer_bounds_and_layout(fmt, vmax, half_step):
    rng = np.random.default_rng(7 + fmt)
    N, D = 300, 128
    x = (rng.standard_normal((N, D)) * np.exp(rng.uniform(-8, 8, (N, 1)))).astype(np.float32)
    bits = _bf16_bits(x)
    xf = ob.bf16_to_f32(bits).astype(np.float64)
    codes, sf, vals = ob.quant_mxfp8_rows_head(bits, fmt)
    # scale bytes sit where the atom layout says, and give the no-clip exponent
    for n in (0, 37, 127, 128, 299):
        for kb in range(D // 32):
            e = int(sf[(n // 128) * 512 + ob.atom_index(n, kb)]) - 127
            amax = np.max(np.abs(xf[n, 32 * kb:32 * kb + 32]))
            assert e == ob.mx_exponent(amax, fmt)
            # normal elements: relative error within half a step; all: absolute
            # error within half the subnormal step of the block's scale
            blk = xf[n, 32 * kb:32 * kb + 32]
            err = np.abs(vals[n, 32 * kb:32 * kb + 32] - blk)
            sub = 2.0 ** (e + (-6 if fmt == ob.E4M3 else -14) - (3 if fmt == ob.E4M3 else 2))
            assert np.all(err <= np.maximum(half_step * np.abs(blk), sub / 2) * (1 + 1e-12))
    # the decoded codes times the block scale are the values
    e_of = np.zeros((N, D // 32), dtype=np.int64)
    for kb in range(D // 32):
        e_of[:, kb] = sf[(np.arange(N) // 128) * 512 + ob.atom_index(np.arange(N), kb)].astype(np.int64) - 127
    assert np.array_equal(ob.fp8_decode(codes, fmt) * np.ldexp(1.0, np.repeat(e_of, 32, axis=1)), vals)
    # quantizing along D equals quantizing the transpose along the sequence
    codes_t, _, vals_t = ob.quant_mxfp8_t_head(_bf16_bits(x.T.copy()), fmt)
    assert np.array_equal(vals_t.T, vals)


def test_nvfp4_decode_uses_the_c_scale_index():
    B, H, N, D = 1, 3, 200, 128
    for bh in (0, 2):
        off = ob.nvfp4_sf_offsets(bh, N, D)
        for r, k in [(0, 0), (31, 7), (32, 3), (127, 4), (128, 5), (199, 7)]:
            assert off[r, k] == oracle.sf_index(bh, (N + 127) // 128, r, k, D // 16)


def test_nvfp4_decode_reconstructs_the_inputs():
    rng = np.random.default_rng(9)
    B, H, N, D = 1, 2, 256, 64
    x = rng.standard_normal((B, H, N, D)).astype(np.float32)
    bits = _bf16_bits(x)
    payload, sf, g = oracle.quant_nvfp4(bits)
    xf = ob.bf16_to_f32(bits).astype(np.float64)
    for bh in range(B * H):
        vals = ob.decode_nvfp4_head(payload.reshape(B * H, N, D // 2)[bh], sf, bh, N, D) * float(g)
        # E2M1 with an E4M3 block scale: within half a step of the largest code
        # (1 of 6) of each 16-block plus the scale's own rounding
        blk = xf.reshape(B * H, N, D // 16, 16)[bh]
        amax = np.max(np.abs(blk), axis=-1, keepdims=True)
        err = np.abs(vals.reshape(N, D // 16, 16) - blk)
        assert np.all(err <= amax * (1.0 / 6.0) * 1.07 + 1e-30)
    # exactly representable inputs come back exactly: with every 16-block's
    # maximum at 6 x 7/64 the tensor scale g = amax / 2688 = 2^-12 and every
    # block scale is E4M3(448), so each value is its code times 448 g = 7/64
    codes = rng.integers(0, 16, (1, 1, 128, 64))
    lut = np.array([oracle.e2m1_decode(int(c)) for c in range(16)])
    y = lut[codes] * (7.0 / 64.0)
    for c0 in (0, 16, 32, 48):
        y[..., c0] = (6.0 if c0 != 32 else -6.0) * (7.0 / 64.0)
    p, s, g = oracle.quant_nvfp4(_bf16_bits(y))
    assert float(g) == 2.0 ** -12
    v = ob.decode_nvfp4_head(p.reshape(128, 32), s, 0, 128, 64) * float(g)
    assert np.array_equal(v, y[0, 0])


# ---- the backward ----------------------------------------------------------

def _autograd(q, k, v, do, scale):
    qt, kt, vt = (torch.tensor(a, dtype=torch.float64, requires_grad=True) for a in (q, k, v))
    z = scale * (qt @ kt.T)
    N = q.shape[0]
    z = z.masked_fill(torch.ones(N, N, dtype=torch.bool).triu(1), float("-inf"))
    lse = torch.logsumexp(z, dim=1)
    o = torch.softmax(z, dim=1) @ vt
    (o * torch.tensor(do)).sum().backward()
    return o.detach().numpy(), lse.detach().numpy(), qt.grad.numpy(), kt.grad.numpy(), vt.grad.numpy()


def _unquantized_case(N, D, seed, spread=1.0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((N, D)) * spread
    k = rng.standard_normal((N, D)) * spread
    v = rng.standard_normal((N, D))
    do = rng.standard_normal((N, D))
    scale = 1.0 / np.sqrt(D)
    o, lse, dq, dk, dv = _autograd(q, k, v, do, scale)
    c32 = ob.score_multiplier(scale, 1.0, 1.0)
    l2 = (lse.astype(np.float32) * ob.LOG2E_F32).astype(np.float32)
    delta = np.sum(do * o, axis=1).astype(np.float32)
    return q, k, v, do, scale, c32, l2, delta, (dq, dk, dv)


@pytest.mark.parametrize("N,D,spread", [(128, 64, 1.0), (200, 64, 2.0), (256, 128, 1.0), (130, 128, 0.5)])
def test_unquantized_backward_equals_autograd(N, D, spread):
    q, k, v, do, scale, c32, l2, delta, (dq, dk, dv) = _unquantized_case(N, D, N + D, spread)
    out = ob.bwd_head(q, k, c32, scale, l2, delta, do, v, do, q, k, fp8=False)
    # only fp32 roundings (S, the exponent, P, dP, dP - Delta, dS) separate the two
    for name, want in (("dq", dq), ("dk", dk), ("dv", dv)):
        err = np.max(np.abs(out[name] - want)) / np.max(np.abs(want))
        assert err < 2e-5, (name, err)
    # row subsets are the same rows
    sub = ob.bwd_head(q, k, c32, scale, l2, delta, do, v, do, q, k, qrows=[0, 5, N - 1], krows=[1, N - 2], fp8=False)
    assert np.allclose(sub["dq"], out["dq"][[0, 5, N - 1]], rtol=0, atol=0)
    assert np.allclose(sub["dk"], out["dk"][[1, N - 2]], rtol=0, atol=0)
    assert np.allclose(sub["dv"], out["dv"][[1, N - 2]], rtol=0, atol=0)


def test_reconstructed_probabilities_are_the_softmax():
    q, k, v, do, scale, c32, l2, delta, _ = _unquantized_case(192, 64, 21)
    out = ob.bwd_head(q, k, c32, scale, l2, delta, do, v, do, q, k, fp8=False)
    p = out["p_q"].astype(np.float64)
    z = scale * (q @ k.T)
    z[np.triu_indices(192, 1)] = -np.inf
    want = np.exp(z - np.max(z, axis=1, keepdims=True))
    want /= np.sum(want, axis=1, keepdims=True)
    assert np.max(np.abs(p - want)) < 1e-6
    assert np.all(np.abs(np.sum(p, axis=1) - 1) < 1e-5)
    assert np.all(p[np.triu_indices(192, 1)] == 0)


def test_fp8_backward_is_close_to_autograd_and_further_than_fp32():
    N, D = 256, 64
    q, k, v, do, scale, c32, l2, delta, (dq, dk, dv) = _unquantized_case(N, D, 77)
    # the FP8 operands the kernels use, from the bf16-rounded inputs
    qb, kb, vb, dob = (_bf16_bits(a.astype(np.float32)) for a in (q, k, v, do))
    _, _, v_rows = ob.quant_mxfp8_rows_head(vb, ob.E4M3)
    _, _, do_rows = ob.quant_mxfp8_rows_head(dob, ob.E5M2)
    _, _, do_t = ob.quant_mxfp8_t_head(dob, ob.E5M2)
    _, _, q_t = ob.quant_mxfp8_t_head(qb, ob.E4M3)
    _, _, k_t = ob.quant_mxfp8_t_head(kb, ob.E4M3)
    out8 = ob.bwd_head(q, k, c32, scale, l2, delta, do_rows, v_rows, do_t, q_t, k_t)
    out32 = ob.bwd_head(q, k, c32, scale, l2, delta, do, v, do, q, k, fp8=False)
    for name, want in (("dq", dq), ("dk", dk), ("dv", dv)):
        rel8 = np.linalg.norm(out8[name] - want) / np.linalg.norm(want)
        rel32 = np.linalg.norm(out32[name] - want) / np.linalg.norm(want)
        # E5M2 keeps 3 significant bits (relative step 2^-2), E4M3 4 bits
        assert rel8 < 0.15, (name, rel8)
        assert rel32 < rel8, (name, rel32, rel8)


def test_causal_dependencies():
    # dK/dV of key j depend on the queries i >= j only; dQ of query i on the keys j <= i only
    N, D = 160, 64
    q, k, v, do, scale, c32, l2, delta, _ = _unquantized_case(N, D, 5)
    base = ob.bwd_head(q, k, c32, scale, l2, delta, do, v, do, q, k, fp8=False)
    j = 70
    do2 = do.copy()
    do2[:j] += 1.0
    q2 = q.copy()
    q2[:j] *= -1
    d2 = delta.copy()
    d2[:j] += 3.0
    pert = ob.bwd_head(q2, k, c32, scale, l2, d2, do2, v, do2, q2, k, krows=[j, N - 1], qrows=[], fp8=False)
    assert np.array_equal(pert["dk"], base["dk"][[j, N - 1]])
    assert np.array_equal(pert["dv"], base["dv"][[j, N - 1]])
    i = 60
    k2 = k.copy()
    k2[i + 1:] *= 3
    v2 = v.copy()
    v2[i + 1:] += 1
    pert = ob.bwd_head(q, k2, c32, scale, l2, delta, do, v2, do, q, k2, qrows=[0, i], krows=[], fp8=False)
    assert np.array_equal(pert["dq"], base["dq"][[0, i]])
