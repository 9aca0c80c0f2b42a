"""Helpers shared by the GPU parity tests: move GPU-quantized buffers to the
oracle's numpy form, run the forward and compare it with the oracle.

Parity bar: probability codes agree on >= 99.9% of entries (ties may flip
with fp32 accumulation order), block shifts likewise, O within max-abs 2e-2
and LSE within 1e-3.  Codes and block shifts are compared with both readings
of the oracle's decisions: in fp32 (the kernel's precision) and in fp64 (S,
c, X and X - K_b unrounded, the plain reading of the method); both must agree
on >= 99.9%."""
import numpy as np
import torch

import oracle


def nv_to_np(t):
    return (t.payload.cpu().numpy(), t.sf.cpu().numpy(), np.float32(t.g.cpu().item()))


def mx_to_np(t):
    return (t.payload_t.cpu().numpy(), t.sf.cpu().numpy())


def unpack_codes(packed: np.ndarray) -> np.ndarray:
    packed = np.asarray(packed, dtype=np.uint8)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.uint8)
    out[..., 0::2] = packed & 0xF
    out[..., 1::2] = packed >> 4
    return out


def sample_rows(B, H, N, heads, rows_per_head, seed):
    """Flat row ids (b*H+h)*N+i: for each chosen head, rows 0 and N-1 and one
    random row in each of rows_per_head equal strata of [0, N)."""
    rng = np.random.default_rng(seed)
    n = min(N, rows_per_head)
    edges = np.linspace(0, N, n + 1).astype(np.int64)
    out = []
    for bh in heads:
        r = [rng.integers(lo, hi) for lo, hi in zip(edges[:-1], edges[1:]) if hi > lo]
        r = np.unique(np.concatenate([[0, N - 1], np.array(r, dtype=np.int64)]))
        out.extend(int(bh) * N + int(i) for i in r)
    return np.array(sorted(set(out)), dtype=np.int64)


def cosine(a, b):
    a = np.asarray(a, dtype=np.float64).reshape(-1)
    b = np.asarray(b, dtype=np.float64).reshape(-1)
    return float(a @ b / (np.linalg.norm(a) * np.linalg.norm(b)))


O_TOL = 2e-2
LSE_TOL = 1e-3
CODE_AGREE = 0.999
# O is stored in bf16: an 8-bit significand, so round to nearest even has a
# relative error up to 2^-8 (1 + 2^-8 rounds to 1.0).  The 2e-2 absolute bound
# applies to O as computed (fp32, before that store, read through the dump
# entry point); the stored bf16 O is checked against 2e-2 plus its own
# rounding, and to be exactly the rounding of the fp32 value.
BF16_REL = 2.0 ** -8


def quantize(q, k, v, fp8pv=False):
    import blackwell_nvfp4_quantize_gb300 as fa

    vq = fa.quant_v_mxfp8(v.cuda()) if fp8pv else fa.quant_v_mxfp4(v.cuda())
    return fa.quant_qk_nvfp4(q.cuda()), fa.quant_qk_nvfp4(k.cuda()), vq


def run_and_check(q, k, v, scale, dump_slices, sample, label, causal=False, fp8pv=False):
    """Runs the forward (causal: query i sees keys 0..i; fp8pv: E4M3
    probability codes and MXFP8 V) and compares it with the oracle.
    dump_slices: list of (b, h, row0, nrows) compared in full (codes, block
    shifts, fp32 O before its bf16 store, LSE); sample: flat row ids whose
    stored bf16 O and LSE are compared."""
    import blackwell_nvfp4_quantize_gb300 as fa

    B, H, N, D = q.shape
    qq, kq, vq = quantize(q, k, v, fp8pv)
    pv_fmt = oracle.PV_MXFP8 if fp8pv else oracle.PV_MXFP4
    if fp8pv:
        o, lse = fa.fwd_directp_fp8pv(qq, kq, vq, scale, causal=causal)
    else:
        fwd = fa.fwd_directp_causal if causal else fa.fwd_directp
        o, lse = fwd(qq, kq, vq, scale)
    torch.cuda.synchronize()
    assert fa.device_status() == fa.FP4ATTN_OK
    qn, kn, vn = nv_to_np(qq), nv_to_np(kq), mx_to_np(vq)
    o_np = o.float().cpu().numpy().reshape(-1, D)
    lse_np = lse.cpu().numpy().reshape(-1)
    assert np.all(np.isfinite(o_np)) and np.all(np.isfinite(lse_np))
    # stored bf16 O / LSE on sampled rows: 2e-2 plus the bf16 rounding of the output
    ref = oracle.directp_rows(qn, kn, vn, (B, H, N, D), scale, sample, causal=causal, pv_fmt=pv_fmt)
    err_o16 = float(np.max(np.abs(o_np[sample] - ref["o"]) - BF16_REL * np.abs(ref["o"])))
    err_l = float(np.max(np.abs(lse_np[sample] - ref["lse"])))
    # codes, block shifts and fp32 O through the dump entry point (same kernel and launch shape)
    agree = total = kagree = ktotal = agree64 = kagree64 = 0
    err_o32 = 0.0
    for (b, h, row0, nrows) in dump_slices:
        o2, lse2, codes, kshift, o32 = fa.debug_dump_p(qq, kq, vq, b, h, row0, nrows, scale, causal=causal)
        torch.cuda.synchronize()
        # the dump variant computes the same O / LSE, and O is the bf16 rounding of its fp32 value
        assert torch.equal(o2, o) and torch.equal(lse2, lse)
        assert torch.equal(o32.to(torch.bfloat16), o2.reshape(-1, D)[(b * H + h) * N + row0:][:nrows])
        rows = np.arange(nrows, dtype=np.int64) + (b * H + h) * N + row0
        r = oracle.directp_rows(qn, kn, vn, (B, H, N, D), scale, rows, want_codes=True, causal=causal,
                                pv_fmt=pv_fmt)
        err_o32 = max(err_o32, float(np.max(np.abs(o32.cpu().numpy() - r["o"]))))
        err_l = max(err_l, float(np.max(np.abs(lse_np[rows] - r["lse"]))))
        gc = codes.cpu().numpy() if fp8pv else unpack_codes(codes.cpu().numpy())
        agree += int(np.sum(gc[:, :N] == r["codes"][:, :N]))
        total += nrows * N
        nblk = (N + 31) // 32
        gk = kshift.cpu().numpy()[:, :nblk]
        kagree += int(np.sum(gk == r["kshift"][:, :nblk]))
        ktotal += gk.size
        r64 = oracle.directp_rows(qn, kn, vn, (B, H, N, D), scale, rows, want_codes=True, causal=causal,
                                  pv_fmt=pv_fmt, f64_decisions=True)
        agree64 += int(np.sum(gc[:, :N] == r64["codes"][:, :N]))
        kagree64 += int(np.sum(gk == r64["kshift"][:, :nblk]))
        assert np.all(gc[:, N:] == 0)
    frac = agree / max(total, 1)
    kfrac = kagree / max(ktotal, 1)
    frac64 = agree64 / max(total, 1)
    kfrac64 = kagree64 / max(ktotal, 1)
    print("%s: max|dO32|=%.3g max|dO16|-bf16=%.3g max|dLSE|=%.3g codes agree %.6f (fp64 reading %.6f) "
          "kshift agree %.6f (fp64 reading %.6f)" % (label, err_o32, err_o16, err_l, frac, frac64, kfrac, kfrac64))
    assert err_o32 <= O_TOL, err_o32
    assert err_o16 <= O_TOL, err_o16
    assert err_l <= LSE_TOL, err_l
    if total:
        assert frac >= CODE_AGREE, frac
        assert kfrac >= CODE_AGREE, kfrac
        assert frac64 >= CODE_AGREE, frac64
        assert kfrac64 >= CODE_AGREE, kfrac64
    return o_np, lse_np
