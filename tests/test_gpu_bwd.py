"""GPU parity of the causal backward (dQ, dK, dV) and of its FP8 operand
quantizers against the oracle (oracle/bwd.py).

Method: "Hardware-Aware FP4 FlashAttention-4", summary page, "What the paper
found": the backward reconstructs the probabilities from the saved quantized
Q/K and LSE and uses FP8 gradient operands, including E5M2 output gradients.

Every input of both sides comes from the seeded generators and the oracle:
the saved NVFP4 Q/K are the oracle's quantization, O and LSE the oracle's
causal forward; the GPU quantizes its FP8 operands itself (checked bit for
bit against the oracle's here).

Tolerance.  Both sides round the same quantities to the same FP8 codes except
where a value sits at a rounding boundary and the two fp32 computations of it
(the kernel's ex2 approximation and MMA accumulation order against the
oracle's exact exponential and sums) fall on different sides: then one term
of a sum moves by one FP8 step, at most 2^-2 of that term (E5M2; 2^-3 for
E4M3).  Each output element is therefore held to
    |gpu - oracle| <= 0.3 * (largest |term| of its sum) + 1e-4 * max|oracle|
(one flipped code of its largest term, plus fp32 accumulation), and at most
0.5% of the elements may exceed 1e-3 * max|oracle| at all.
"""
import numpy as np
import pytest
import torch

import oracle
import oracle.bwd as ob

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def _rand(shape, seed, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    return (torch.randn(shape, generator=g) * scale).to(torch.bfloat16)


def _oracle_forward(qb, kb, vb, shape, scale, heads):
    """Oracle quantization of Q, K (NVFP4) and V (MXFP4) and its causal
    forward over every row of the given heads: (q_np, k_np, o [heads,N,D],
    lse [heads,N])."""
    B, H, N, D = shape
    q_np = oracle.quant_nvfp4(qb)
    k_np = oracle.quant_nvfp4(kb)
    v_np = oracle.quant_mxfp4_v(vb)
    rows = np.concatenate([np.arange(N, dtype=np.int64) + bh * N for bh in heads])
    out = oracle.directp_rows(q_np, k_np, v_np, shape, scale, rows, causal=True)
    return q_np, k_np, out["o"].reshape(len(heads), N, D), out["lse"].reshape(len(heads), N)


def _nvfp4_to_gpu(t_np, shape):
    import blackwell_nvfp4_quantize_gb300 as fa
    B, H, N, D = shape
    p, s, g = t_np
    return fa.NVFP4Tensor(torch.from_numpy(p).reshape(B, H, N, D // 2).cuda(), torch.from_numpy(s).cuda(),
                          torch.tensor([float(g)], dtype=torch.float32).cuda(), tuple(shape))


def _term_bound(coef, op):
    """Largest |coef[r, i] * op[i, d]| over i for every (r, d)."""
    a = np.abs(coef)
    b = np.abs(op)
    out = np.zeros((a.shape[0], b.shape[1]))
    for r in range(a.shape[0]):
        out[r] = np.max(a[r][:, None] * b, axis=0)
    return out


def _compare(name, got, want, bound, label):
    err = np.abs(got - want)
    top = float(np.max(np.abs(want)))
    allow = 0.3 * bound + 1e-4 * top
    frac_big = float(np.mean(err > 1e-3 * top))
    worst = float(np.max(err / np.maximum(allow, 1e-300)))
    rel_fro = float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))
    print("%s %s: max|err|/max|ref| %.2e  rel_fro %.2e  >1e-3: %.4f%%  worst err/allow %.3f"
          % (label, name, float(np.max(err)) / top, rel_fro, 100 * frac_big, worst))
    assert np.all(err <= allow), (label, name, worst)
    assert frac_big <= 0.005, (label, name, frac_big)


def run_bwd_case(q, k, v, dout, heads, qrows_per_head, krows_per_head, label, seed=0):
    """Runs the GPU backward on the whole tensor and compares dQ (rows qrows)
    and dK, dV (keys krows) of the given heads with the oracle."""
    import blackwell_nvfp4_quantize_gb300 as fa

    B, H, N, D = q.shape
    scale = 1.0 / np.sqrt(D)
    qb, kb, vb, db = _bits(q), _bits(k), _bits(v), _bits(dout)
    q_np, k_np, o_h, lse_h = _oracle_forward(qb, kb, vb, q.shape, scale, heads)
    q_saved, k_saved = _nvfp4_to_gpu(q_np, q.shape), _nvfp4_to_gpu(k_np, q.shape)
    # O and LSE of the other heads: the library's causal forward (those heads
    # are not compared); the compared heads carry the oracle's
    o_gpu, lse_gpu = fa.fwd_directp_causal(q_saved, k_saved, fa.quant_v_mxfp4(v.cuda()), scale)
    for n, bh in enumerate(heads):
        b, h = divmod(int(bh), H)
        o_gpu[b, h] = torch.from_numpy(o_h[n]).to(torch.bfloat16).cuda()
        lse_gpu[b, h] = torch.from_numpy(lse_h[n].astype(np.float32)).cuda()
    dq, dk, dv = fa.attention_backward_causal(q.cuda(), k.cuda(), v.cuda(), o_gpu, lse_gpu, dout.cuda(),
                                              q_saved, k_saved, scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    dq, dk, dv = (t.cpu().numpy().reshape(B * H, N, D) for t in (dq, dk, dv))
    o_bits = _bits(o_gpu.cpu()).reshape(B * H, N, D)
    lse_all = lse_gpu.cpu().numpy().reshape(B * H, N)
    rng = np.random.default_rng(seed)
    c32 = ob.score_multiplier(scale, q_np[2], k_np[2])
    for n, bh in enumerate(heads):
        bh = int(bh)
        qhat = ob.decode_nvfp4_head(q_np[0].reshape(B * H, N, D // 2)[bh], q_np[1], bh, N, D)
        khat = ob.decode_nvfp4_head(k_np[0].reshape(B * H, N, D // 2)[bh], k_np[1], bh, N, D)
        delta, l2 = ob.prep(o_bits[bh], db.reshape(B * H, N, D)[bh], lse_all[bh])
        hb = lambda x: x.reshape(B * H, N, D)[bh]
        v_rows = ob.quant_mxfp8_rows_head(hb(vb), ob.E4M3)[2]
        do_rows = ob.quant_mxfp8_rows_head(hb(db), ob.E5M2)[2]
        do_t = ob.quant_mxfp8_t_head(hb(db), ob.E5M2)[2]
        q_t = ob.quant_mxfp8_t_head(hb(qb), ob.E4M3)[2]
        k_t = ob.quant_mxfp8_t_head(hb(kb), ob.E4M3)[2]

        def pick(count):
            if count >= N or N <= 2:
                return np.arange(N)
            mid = rng.choice(np.arange(1, N - 1), size=max(count - 2, 0), replace=False)
            return np.unique(np.concatenate([[0, N - 1], mid]))

        qr, kr = pick(qrows_per_head), pick(krows_per_head)
        ref = ob.bwd_head(qhat, khat, c32, scale, l2, delta, do_rows, v_rows, do_t, q_t, k_t, qrows=qr, krows=kr)
        tag = "%s head %d" % (label, bh)
        _compare("dV", dv[bh][kr], ref["dv"], _term_bound(ref["p_kv"].T, do_t), tag)
        _compare("dK", dk[bh][kr], ref["dk"], scale * _term_bound(ref["ds_kv"].T, q_t), tag)
        _compare("dQ", dq[bh][qr], ref["dq"], scale * _term_bound(ref["ds_q"], k_t), tag)


# ---- FP8 operand quantizers and the prep pass ------------------------------

@pytest.mark.parametrize("shape", [(1, 1, 128, 64), (1, 2, 200, 128), (2, 2, 333, 64)])
@pytest.mark.parametrize("fmt", [0, 1])
def test_fp8_quantizers_bit_exact(shape, fmt):
    import blackwell_nvfp4_quantize_gb300 as fa
    x = _rand(shape, 11 + fmt + shape[2], 3.0)
    # a wide range of magnitudes per row and channel, zero rows, tiny values
    x = (x.float() * torch.exp(torch.linspace(-20, 20, shape[2])).view(1, 1, -1, 1)).to(torch.bfloat16)
    x[..., 0, :] = 0
    xb = _bits(x)
    rows = fa.quant_mxfp8_rows(x.cuda(), fmt)
    t = fa.quant_mxfp8_t(x.cuda(), fmt)
    c_rows, sf_rows, _ = ob.quant_mxfp8_rows(xb, fmt)
    c_t, sf_t, _ = ob.quant_mxfp8_t(xb, fmt)
    assert np.array_equal(rows.payload.cpu().numpy(), c_rows)
    assert np.array_equal(rows.sf.cpu().numpy(), sf_rows)
    assert np.array_equal(t.payload.cpu().numpy(), c_t)
    assert np.array_equal(t.sf.cpu().numpy(), sf_t)


@pytest.mark.parametrize("idx", [1, 2, 3])
def test_fp8_quantizers_workloads(idx):
    import blackwell_nvfp4_quantize_gb300 as fa
    from blackwell_nvfp4_quantize_gb300 import workloads as wl
    w = wl.WORKLOADS[idx]
    q, k, v = wl.make_inputs(w)
    for x, fmt in ((v, 0), (q, 0), (k, 0), (v, 1)):
        xb = _bits(x)
        rows = fa.quant_mxfp8_rows(x.cuda(), fmt)
        t = fa.quant_mxfp8_t(x.cuda(), fmt)
        c_rows, sf_rows, _ = ob.quant_mxfp8_rows(xb, fmt)
        c_t, sf_t, _ = ob.quant_mxfp8_t(xb, fmt)
        assert np.array_equal(rows.payload.cpu().numpy(), c_rows)
        assert np.array_equal(rows.sf.cpu().numpy(), sf_rows)
        assert np.array_equal(t.payload.cpu().numpy(), c_t)
        assert np.array_equal(t.sf.cpu().numpy(), sf_t)


@pytest.mark.parametrize("shape", [(1, 1, 128, 64), (2, 3, 200, 128)])
def test_prep(shape):
    import blackwell_nvfp4_quantize_gb300 as fa
    B, H, N, D = shape
    o, do = _rand(shape, 1), _rand(shape, 2)
    lse = torch.randn((B, H, N), generator=torch.Generator().manual_seed(3)) * 5
    nl2, delta = fa.bwd_prep(o.cuda(), do.cuda(), lse.cuda())
    want_delta, want_l2 = ob.prep(_bits(o), _bits(do), lse.numpy())
    npad = (N + 127) // 128 * 128
    nl2, delta = nl2.cpu().numpy(), delta.cpu().numpy()
    assert np.array_equal(nl2[..., :N], -want_l2)
    assert np.all(np.isinf(nl2[..., N:])) and np.all(nl2[..., N:] < 0)
    assert np.all(delta[..., N:] == 0)
    # fp32 accumulation of D products: within D 2^-24 of the sum of |terms|
    mag = np.sum(np.abs(ob.bf16_to_f32(_bits(o)).astype(np.float64) * ob.bf16_to_f32(_bits(do))), axis=-1)
    assert np.all(np.abs(delta[..., :N] - want_delta) <= D * 2.0 ** -24 * mag + 1e-30)
    assert nl2.shape == (B, H, npad)


# ---- the backward ------------------------------------------------------------

@pytest.mark.parametrize("shape", [(1, 1, 1, 64), (1, 1, 1, 128), (1, 2, 37, 128), (1, 1, 128, 64), (1, 1, 256, 128),
                                   (1, 2, 200, 64), (2, 1, 384, 128), (1, 1, 1000, 64)])
def test_bwd_small_full(shape):
    B, H, N, D = shape
    q, k, v, do = (_rand(shape, 100 + i + N) for i in range(4))
    run_bwd_case(q, k, v, do, heads=list(range(B * H)), qrows_per_head=N, krows_per_head=N,
                 label="bwd %s" % (shape,))


def test_bwd_large_magnitudes():
    # wide score range (sharp softmax) and large output gradients
    shape = (1, 1, 384, 128)
    q, k = _rand(shape, 7, 3.0), _rand(shape, 8, 3.0)
    v, do = _rand(shape, 9, 10.0), _rand(shape, 10, 1e3)
    run_bwd_case(q, k, v, do, heads=[0], qrows_per_head=384, krows_per_head=384, label="bwd sharp")


def test_bwd_workload1_full():
    from blackwell_nvfp4_quantize_gb300 import workloads as wl
    w = wl.WORKLOADS[1]
    q, k, v = wl.make_inputs(w)
    do = _rand(w.shape, 4001)
    run_bwd_case(q, k, v, do, heads=[0], qrows_per_head=w.shape[2], krows_per_head=w.shape[2], label="w1")


@pytest.mark.parametrize("idx,heads", [(2, [0, 3, 7]), (3, [0, 17, 31]), (4, [0, 7, 19, 23, 31, 39]),
                                       (5, [0, 13, 29, 37, 50, 63])])
def test_bwd_workloads_sampled(idx, heads):
    # heads spread over the tensor (first, last and between), 16 dQ rows
    # and 16 dK/dV keys each (rows 0 and N-1 always), in the full-size launch
    from blackwell_nvfp4_quantize_gb300 import workloads as wl
    w = wl.WORKLOADS[idx]
    q, k, v = wl.make_inputs(w)
    do = _rand(w.shape, 4000 + idx)
    run_bwd_case(q, k, v, do, heads=heads, qrows_per_head=16, krows_per_head=16, label=w.name, seed=idx)
