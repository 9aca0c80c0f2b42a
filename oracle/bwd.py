"""CPU oracle for the causal backward -- TEST INFRASTRUCTURE ONLY.

Plain numpy (fp64, with fp32 exactly where the kernel takes a format decision
in fp32).  Only the test-suite and the benchmark's CPU legs may import it; the
CUDA library never does and shares no code with it.

Source: "Hardware-Aware FP4 FlashAttention-4", neuraltrendhub.com summary
page, section "What the paper found" (for causal training the forward saves
the quantized Q/K payloads, scales and LSE; the backward reconstructs the
probabilities from them and uses FP8 gradient operands, including E5M2 output
gradients), and the paper's abstract (the causal path reconstructs
probabilities from the saved quantized queries and keys and uses FP8 gradient
operands).  The pages give no formula; the readings taken here:

* Probabilities are reconstructed from the saved NVFP4 Q/K (the same block-
  scaled product as the forward) and the saved LSE:
  P_ij = 2^(c S_ij - LSE_i log2 e), c = fp32(softmax_scale log2 e g_Q g_K),
  for keys j <= i, else 0.  The exponent is one fp32 FMA (c S - L_i) with
  L_i = fp32(LSE_i * fp32(log2 e)); P_ij is fp32, values below 2^-126 flushed
  to zero (the kernel's exponential flushes subnormal results).
* Delta_i = sum_d dO_id O_id (fp32); dP = dO V^T; dS_ij = P_ij (dP_ij - Delta_i),
  the plain FlashAttention backward with P recomputed.
* Every product runs on FP8 operands with MX block scaling (E8M0 scale per
  32 consecutive elements along the product's contraction axis; e the
  smallest integer >= -127 with amax <= fmt_max 2^e; codes RNE-satfinite of
  x 2^-e): gradients (dO, dS) in E5M2, everything else (V, Q, K, P) in E4M3.
  Hence dO is quantized twice (blocks along D for dP, along the sequence for
  dV), dS twice (along the queries for dK, along the keys for dQ), V along D,
  Q and K along the sequence (taken from the bf16 training inputs; the saved
  NVFP4 Q/K serve the probability reconstruction).
* dV_j = sum_i P~_ij dO~_i;  dK_j = softmax_scale sum_i dS~_ij Q~_i;
  dQ_i = softmax_scale sum_j dS~_ij K~_j  (fp32 outputs).
"""
from __future__ import annotations

import numpy as np

E4M3, E5M2 = 0, 1
# (mantissa bits, minimum normal exponent, exponent bias, largest finite value)
_FMT = {E4M3: (3, -6, 7, 448.0), E5M2: (2, -14, 15, 57344.0)}
LOG2E_F32 = np.float32(1.4426950408889634)


# ---- formats -------------------------------------------------------------

def fp8_round(y, fmt):
    """Nearest FP8 value (ties to even, saturating at +-max, sign kept) of
    each fp32/fp64 value: the value of cvt.rn.satfinite.{e4m3,e5m2}."""
    m, emin, _, vmax = _FMT[fmt]
    y = np.asarray(y, dtype=np.float64)
    a = np.abs(y)
    _, ex = np.frexp(a)                         # a = f 2^ex, f in [0.5, 1)
    e = np.maximum(ex - 1, emin)                # exponent of the binade (normals), emin for subnormals
    ulp = np.ldexp(1.0, e - m)
    q = np.rint(a / ulp) * ulp                  # a / ulp is exact; rint is ties-to-even
    q = np.minimum(q, vmax)
    return np.copysign(q, y)


def fp8_encode(y, fmt):
    """FP8 code bytes of fp8_round(y) (E4M3: s eeee mmm, E5M2: s eeeee mm)."""
    m, emin, bias, _ = _FMT[fmt]
    q = fp8_round(y, fmt)
    a = np.abs(q)
    sign = np.signbit(q).astype(np.uint32)
    _, ex = np.frexp(a)
    e = ex - 1
    normal = a >= np.ldexp(1.0, emin)
    efield = np.where(normal, e + bias, 0)
    mant = np.where(normal, np.ldexp(a, -e) - 1.0, np.ldexp(a, -(emin - m)) / (1 << m))
    mfield = np.rint(mant * (1 << m)).astype(np.int64)
    code = (sign << 7) | (efield.astype(np.uint32) << m) | mfield.astype(np.uint32)
    return code.astype(np.uint8)


def fp8_decode(code, fmt):
    m, emin, bias, _ = _FMT[fmt]
    c = np.asarray(code, dtype=np.uint32)
    s = (c >> 7) & 1
    ef = (c >> m) & ((1 << (7 - m)) - 1)
    mf = c & ((1 << m) - 1)
    mag = np.where(ef == 0, np.ldexp(mf.astype(np.float64), emin - m),
                   np.ldexp(1.0 + mf / float(1 << m), ef.astype(np.int64) - bias))
    return np.where(s == 1, -mag, mag)


def mx_exponent(amax, fmt):
    """Smallest integer e >= -127 with amax <= fmt_max 2^e (-127 for amax = 0),
    taken exactly from amax = f 2^k, f in [1, 2), and fmt_max = 1.75 2^p."""
    p = 8 if fmt == E4M3 else 15
    a = np.asarray(amax, dtype=np.float64)
    f, ex = np.frexp(a)
    k = ex - 1
    e = np.where(2.0 * f <= 1.75, k - p, k - p + 1)
    e = np.where(a > 0, e, -127)
    return np.clip(e, -127, 127).astype(np.int64)


def mx_quant_blocks(x32, fmt):
    """MX block quantization along the last axis of an fp32 array whose last
    axis is a multiple of 32.  Returns (values f64 same shape, codes u8, e i64
    [..., n/32]).  The scaled value is one fp32 multiply by 2^-e."""
    x32 = np.asarray(x32, dtype=np.float32)
    shp = x32.shape
    blk = x32.reshape(shp[:-1] + (shp[-1] // 32, 32))
    e = mx_exponent(np.max(np.abs(blk), axis=-1).astype(np.float64), fmt)
    inv = np.ldexp(np.float32(1.0), (-e)[..., None]).astype(np.float32)
    y = (blk * inv).astype(np.float32)
    q = fp8_round(y, fmt)
    codes = fp8_encode(y, fmt)
    vals = np.ldexp(q, e[..., None])
    return vals.reshape(shp), codes.reshape(shp), e


def bf16_to_f32(bits):
    return (np.asarray(bits, dtype=np.uint32) << 16).view(np.float32)


def atom_index(row, kblock):
    """Byte of (row, 32-element block) inside a 512-byte scale atom of 128 rows."""
    r = np.asarray(row) % 128
    return (r % 32) * 16 + (r // 32) * 4 + np.asarray(kblock)


# ---- quantizers of the backward operands ----------------------------------

def quant_mxfp8_rows_head(x_bits, fmt):
    """One head's bf16 [N,D] -> MXFP8 along D: codes [N,D] u8, scale atoms
    [T*512] u8 (one 512-byte atom per 128-row tile; row n%128, block d/32),
    decoded values [N,D] f64."""
    x = bf16_to_f32(x_bits)
    N, D = x.shape
    T = (N + 127) // 128
    vals, codes, e = mx_quant_blocks(x, fmt)
    sf = np.zeros((T, 512), dtype=np.uint8)
    n = np.arange(N)
    for kb in range(D // 32):
        sf[n // 128, atom_index(n, kb)] = (e[:, kb] + 127).astype(np.uint8)
    return codes, sf.reshape(-1), vals


def quant_mxfp8_t_head(x_bits, fmt):
    """One head's bf16 [N,D] -> MXFP8 along the sequence, transposed: codes
    [D,Npad] u8 (padded tokens code 0), scale atoms [T*512] u8 (one per
    128-token tile; row d, block (n%128)/32), decoded values [N,D] f64."""
    x = bf16_to_f32(x_bits)
    N, D = x.shape
    T = (N + 127) // 128
    xt = np.zeros((D, T * 128), dtype=np.float32)
    xt[:, :N] = x.T
    vals, codes, e = mx_quant_blocks(xt, fmt)
    sf = np.zeros((T, 512), dtype=np.uint8)
    d = np.arange(D)
    eb = e.reshape(D, T, 4)
    for kb in range(4):
        sf[:, atom_index(d, kb)] = (eb[:, :, kb].T + 127).astype(np.uint8)
    return codes, sf.reshape(-1), vals[:, :N].T.copy()


def _per_head(fn, x_bits, fmt):
    B, H = x_bits.shape[:2]
    parts = [fn(x_bits[b, h], fmt) for b in range(B) for h in range(H)]
    codes = np.stack([p[0] for p in parts]).reshape((B, H) + parts[0][0].shape)
    sf = np.concatenate([p[1] for p in parts])
    vals = np.stack([p[2] for p in parts]).reshape((B, H) + parts[0][2].shape)
    return codes, sf, vals


def quant_mxfp8_rows(x_bits, fmt):
    """bf16 [B,H,N,D] -> (codes [B,H,N,D], atoms ordered by (b, h, tile), values)."""
    return _per_head(quant_mxfp8_rows_head, np.asarray(x_bits, dtype=np.uint16), fmt)


def quant_mxfp8_t(x_bits, fmt):
    """bf16 [B,H,N,D] -> (codes [B,H,D,Npad], atoms ordered by (b, h, tile), values [B,H,N,D])."""
    return _per_head(quant_mxfp8_t_head, np.asarray(x_bits, dtype=np.uint16), fmt)


def nvfp4_sf_offsets(bh, N, D):
    """Byte offsets [N, D/16] of the NVFP4 block scales of head bh: 128-row
    tiles of D/64 atoms, row r, 16-element block k at atom k/4, byte
    (r%32)*16 + (r/32)*4 + k%4."""
    T = (N + 127) // 128
    apt = D // 64
    r = np.arange(N)[:, None]
    k = np.arange(D // 16)[None, :]
    atom = (bh * T + r // 128) * apt + k // 4
    return atom * 512 + (r % 128 % 32) * 16 + (r % 128 // 32) * 4 + k % 4


def decode_nvfp4_head(payload_head, sf, bh, N, D):
    """Saved NVFP4 Q or K of head bh -> the block-scaled values without the
    tensor scale g (code value x E4M3 block scale), f64 [N,D]: the operand of
    the S = Q K^T product, whose g's are folded into c."""
    from . import e2m1_decode, e4m3_decode
    lut2 = np.array([e2m1_decode(c) for c in range(16)])
    lut3 = np.array([e4m3_decode(c) if (c & 0x7F) != 0x7F else np.nan for c in range(256)])  # 0x7F/0xFF: NaN
    p = np.asarray(payload_head, dtype=np.uint8).reshape(N, D // 2)
    codes = np.empty((N, D), dtype=np.uint8)
    codes[:, 0::2] = p & 15
    codes[:, 1::2] = p >> 4
    scales = lut3[np.asarray(sf, dtype=np.uint8)[nvfp4_sf_offsets(bh, N, D)]]  # [N, D/16]
    return lut2[codes] * np.repeat(scales, 16, axis=1)


# ---- the backward ----------------------------------------------------------

def prep(o_bits, do_bits, lse):
    """Delta_i = sum_d dO_id O_id (fp32 result of an fp64 sum) and the
    log2-domain LSE L_i = fp32(LSE_i * fp32(log2 e)), each [B,H,N]."""
    o = bf16_to_f32(o_bits).astype(np.float64)
    do = bf16_to_f32(do_bits).astype(np.float64)
    delta = np.sum(o * do, axis=-1).astype(np.float32)
    l2 = (np.asarray(lse, dtype=np.float32) * LOG2E_F32).astype(np.float32)
    return delta, l2


def probabilities(s_raw, c32, l2, qi, kj):
    """P (fp32) for score block s_raw [len(qi), len(kj)] (exact block-scaled
    sums), query ids qi, key ids kj: 2^fp32(c S - L_i), 0 where key > query."""
    s32 = s_raw.astype(np.float32).astype(np.float64)
    arg = (np.float64(c32) * s32 - l2[qi].astype(np.float64)[:, None]).astype(np.float32)
    p = np.exp2(arg.astype(np.float64)).astype(np.float32)
    p[p < np.float32(2.0 ** -126)] = 0.0  # the kernel's ex2 flushes subnormal results
    p[kj[None, :] > qi[:, None]] = 0.0
    return p


def bwd_head(qhat, khat, c32, softmax_scale, l2, delta, do_rows, v_rows, do_t, q_t, k_t,
             qrows=None, krows=None, fp8=True):
    """Causal backward of one (b, h).

    qhat, khat: [N,D] f64 block-scaled NVFP4 values (decode_nvfp4); c32: the
    forward's fp32 score multiplier; l2, delta: [N] fp32 (prep); do_rows,
    v_rows: [N,D] decoded MXFP8 values along D (E5M2 dO, E4M3 V); do_t, q_t,
    k_t: [N,D] decoded MXFP8 values along the sequence (E5M2 dO, E4M3 Q, K).
    qrows / krows: the query rows of dQ and the key rows of dK, dV to compute
    (default all).  fp8=False skips the FP8 quantization of P and dS (the
    other operands are whatever the caller passes): the same algorithm with
    exact operands, which the tests hold against automatic differentiation.
    Returns dict dq [len(qrows),D], dk, dv [len(krows),D] f64 and the fp32
    P and dS blocks behind them.
    """
    def mx(x, fmt):
        return mx_quant_blocks(x, fmt)[0] if fp8 else x.astype(np.float64)

    N, D = qhat.shape
    npad = (N + 127) // 128 * 128
    qrows = np.arange(N) if qrows is None else np.asarray(qrows)
    krows = np.arange(N) if krows is None else np.asarray(krows)
    out = {}
    # dK, dV for key rows j: all queries i (0 .. Npad-1; padded ones have P = 0)
    if len(krows):
        qi = np.arange(N)
        s_raw = qhat @ khat[krows].T                         # [N, K]
        p = probabilities(s_raw, c32, l2, qi, krows)         # [N, K] fp32
        dp = (do_rows @ v_rows[krows].T).astype(np.float32)  # [N, K]
        t = (dp - delta[:, None]).astype(np.float32)
        ds = (p * t).astype(np.float32)
        # blocks along the queries: the key row is the MMA's M row
        pt = np.zeros((len(krows), npad), dtype=np.float32)
        dst = np.zeros((len(krows), npad), dtype=np.float32)
        pt[:, :N] = p.T
        dst[:, :N] = ds.T
        p_q = mx(pt, E4M3)
        ds_q = mx(dst, E5M2)
        out["dv"] = p_q[:, :N] @ do_t
        out["dk"] = softmax_scale * (ds_q[:, :N] @ q_t)
        out["p_kv"], out["ds_kv"] = p, ds
    if len(qrows):
        kj = np.arange(N)
        s_raw = qhat[qrows] @ khat.T                         # [Q, N]
        p = probabilities(s_raw, c32, l2, qrows, kj)
        dp = (do_rows[qrows] @ v_rows.T).astype(np.float32)
        t = (dp - delta[qrows][:, None]).astype(np.float32)
        ds = (p * t).astype(np.float32)
        dsp = np.zeros((len(qrows), npad), dtype=np.float32)
        dsp[:, :N] = ds
        ds_q = mx(dsp, E5M2)
        out["dq"] = softmax_scale * (ds_q[:, :N] @ k_t)
        out["p_q"], out["ds_q"] = p, ds
    return out


def score_multiplier(softmax_scale, g_q, g_k):
    """c = fp32(softmax_scale log2 e g_Q g_K), the products in fp64 rounded once
    (the forward's score multiplier)."""
    return np.float32(float(softmax_scale) * 1.4426950408889634074 * float(g_q) * float(g_k))


def exact_bwd_head(q, k, v, do, softmax_scale):
    """Unquantized causal attention backward in fp64 for one head (q, k, v, do
    [N,D] f64): returns (o, lse, dq, dk, dv) by the textbook formulas -- the
    reference the quantized backward approaches as the formats widen."""
    N = q.shape[0]
    z = softmax_scale * (q @ k.T)
    z[np.triu_indices(N, 1)] = -np.inf
    m = np.max(z, axis=1, keepdims=True)
    e = np.exp(z - m)
    l = np.sum(e, axis=1, keepdims=True)
    p = e / l
    o = p @ v
    lse = (m + np.log(l))[:, 0]
    dp = do @ v.T
    delta = np.sum(do * o, axis=1, keepdims=True)
    ds = p * (dp - delta)
    return o, lse, softmax_scale * (ds @ k), softmax_scale * (ds.T @ q), p.T @ do
