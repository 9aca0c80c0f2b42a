/*
 * fp4attn oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-purpose CPU restatement of what the Direct-P FP4
 * attention forward computes, used to check the CUDA library.  Only the
 * test-suite, the smoke check and the benchmark's CPU-baseline leg may load
 * it.  It shares no code, header, table or constant with the CUDA library.
 *
 * Source of the method: "Hardware-Aware FP4 FlashAttention-4" (arXiv
 * 2609.04105), as summarised on its neuraltrendhub.com page, section "What the
 * paper found", and in its abstract:
 *   - Q and K are kept in NVFP4,
 *   - log-softmax (max-shifted log2) scores are mapped directly to MXFP4 E2M1
 *     probability codes,
 *   - the row denominator is summed from the same rounded probabilities that
 *     the PV product consumes,
 *   - the forward pass emits O together with the LSE.
 * The pages give no formulas for scale selection or for the mapping; the
 * readings this file implements are listed next to each function.
 *
 * Precision: fp64 wherever the pages fix nothing, except where a floating
 * point value decides an integer (a quantised code or a block exponent); those
 * decisions are taken in fp32, the precision of the kernel that is checked.
 *
 * Parity status per function is stated next to each declaration.
 */
#ifndef FP4ATTN_ORACLE_H
#define FP4ATTN_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- number formats (OCP microscaling formats referenced by the pages) ---- */

/* E2M1 code -> value.  Magnitudes 0, .5, 1, 1.5, 2, 3, 4, 6; bit 3 is the
 * sign.  Pinned: round trip over all 16 codes, hand-worked ties. */
double orc_e2m1_decode(uint8_t code);

/* value -> E2M1 code: round to nearest, ties to the even code, saturate to
 * +-6, keep the sign bit (negative values that round to zero give 0x8).
 * Pinned: hand-worked ties, monotonicity, round trip; exhaustive agreement
 * with the hardware conversion (GPU test). */
uint8_t orc_e2m1_encode(double y);

/* E4M3 (OCP "E4M3FN": bias 7, no infinities, 0x7F/0xFF are NaN) */
double orc_e4m3_decode(uint8_t code);
/* value -> E4M3: nearest, ties to even code, saturate to +-448. Pinned as
 * E2M1. */
uint8_t orc_e4m3_encode(double y);

/* E8M0: byte b is 2^(b-127); 0xFF is NaN. */
double orc_e8m0_decode(uint8_t code);

/* ---- scale-factor atom addressing ----
 * Scale factors are stored in 512-byte atoms covering 128 rows x 4
 * consecutive scale blocks; row r, block k of an atom sits at byte
 * (r%32)*16 + (r/32)*4 + k.  Atoms are ordered [b*H+h][row tile][k/4]. */
size_t orc_sf_index(size_t bh, int n_row_tiles, int row, int kblock, int kblocks_per_row);

/* ---- quantizers ---- */

/* NVFP4 for Q or K, input bf16 bits [B,H,N,D] row-major.
 *   g       = amax(|x|) / 2688 (fp32), or 1 when the tensor is all zero
 *   per 16-element block along D:
 *     sb    = E4M3( amax_b / (6*g) )           (fp32 multiply then divide)
 *     s     = dec(sb) * g                      (fp32)
 *     code  = E2M1( x * (1/s) )                (fp32 reciprocal, fp32 multiply)
 *             or 0 for the whole block when s == 0
 * payload: [B,H,N,D/2] bytes, element 2i in the low nibble of byte i.
 * sf     : atoms, rows padded to a multiple of 128 (size orc_nvfp4_sf_bytes).
 * Pinned: hand-worked blocks, error bound, scale invariants. */
size_t orc_nvfp4_sf_bytes(int B, int H, int N, int D);
void orc_quant_nvfp4(const uint16_t *x, int B, int H, int N, int D,
                     uint8_t *payload, uint8_t *sf, float *g_out, int nthreads);

/* MXFP4 for V along the key axis, written transposed.
 *   per (b,h,d) and 32-key block:  e = the smallest integer >= -127 with
 *   amax <= 6 * 2^e;  scale byte e+127;  code = E2M1( v * 2^-e ) (exact).
 * payload: [B,H,D,Npad/2], Npad = N rounded up to 128; padded keys are 0.
 * sf     : atoms over (row = d, block = key block), one atom per 128 keys
 *          (size orc_mxfp4_sf_bytes).
 * Pinned: hand-worked blocks, amax <= 6*2^e < 2*amax, error bound. */
size_t orc_mxfp4_sf_bytes(int B, int H, int N, int D);
void orc_quant_mxfp4_v(const uint16_t *v, int B, int H, int N, int D,
                       uint8_t *payload_t, uint8_t *sf, int nthreads);

/* MXFP8 for V along the key axis, written transposed (the FP8 P/V variant:
 * "What the paper found", training keeps FP8 probabilities and values).
 *   per (b,h,d) and 32-key block:  e = the smallest integer >= -127 with
 *   amax <= 448 * 2^e;  scale byte e+127;  code = E4M3( v * 2^-e ).
 * payload: [B,H,D,Npad] bytes (one code per key), padded keys 0.
 * sf     : atoms exactly as for MXFP4 V (size orc_mxfp4_sf_bytes).
 * Pinned: hand-worked block, amax <= 448*2^e < 2*amax, error bound. */
void orc_quant_mxfp8_v(const uint16_t *v, int B, int H, int N, int D,
                       uint8_t *payload_t, uint8_t *sf, int nthreads);

/* P/V operand formats of the PV product. */
enum { ORC_PV_MXFP4 = 0, ORC_PV_MXFP8 = 1 };

/* ---- Direct-P attention, two-pass restatement ----
 * For each requested row i of head bh (rows[r] = bh*N + i), over the keys j
 * the row sees -- all N, or with causal != 0 ("What the paper found": the
 * causal training forward) keys 0..i only:
 *   S_ij   = sum_d qhat_id * khat_jd                    (fp64, exact here)
 *   c      = fp32( softmax_scale * log2(e) * g_Q * g_K ) (fp64 products)
 *   X_ij   = fp32( c * fp32(S_ij) )
 *   X_b    = max of X over each 32-key block,  K_b = ceil(X_b - log2 R)
 *            with R the largest finite code value: 6 (E2M1, pv_fmt
 *            ORC_PV_MXFP4) or 448 (E4M3, pv_fmt ORC_PV_MXFP8)
 *   M_i    = ceil(max_j X_ij)                      (an integer row max)
 *   t_ij   = fmaf(c, fp32(S_ij), -K_b)
 *   code   = E2M1 or E4M3 ( 2^t_ij )                (exact exponential)
 *   e_b    = max(K_b - M_i, -127),  p_ij = dec(code) * 2^e_b
 *   l_i    = sum_j p_ij,  O_i = sum_j p_ij vhat_j / l_i,
 *   LSE_i  = ln2 * (M_i + log2 l_i)
 * Outputs per requested row: O (D doubles), lse, and optionally the codes
 * (Npad bytes, one code per byte, padded and unseen keys 0), K_b (Npad/32
 * int32, 0 for blocks the row does not see) and M.
 * Pinned: rows of p/l sum to 1, all-equal scores, integer-shift invariance,
 * hand-worked rows (golden), and P-hat @ V-hat recomputation; causal: the
 * last row equals the noncausal row, row 0 returns v-hat_0 exactly, and a
 * row equals the noncausal last row of the sequence cut after it. */
void orc_directp_rows(const uint8_t *q_payload, const uint8_t *q_sf, float g_q,
                      const uint8_t *k_payload, const uint8_t *k_sf, float g_k,
                      const uint8_t *v_payload_t, const uint8_t *v_sf,
                      int B, int H, int N, int D, float softmax_scale, int causal, int pv_fmt,
                      const int64_t *rows, int nrows,
                      double *o, double *lse,
                      uint8_t *codes, int32_t *kshift, int32_t *mrow,
                      int nthreads);

/* orc_directp_rows with a choice of the precision the mapping's decisions
 * are taken in.  f64_decisions = 0: as above (S, c, X and t rounded to fp32,
 * as the forward kernel computes them).  f64_decisions = 1: the plain fp64
 * reading -- X = c*S with S and c in fp64, K_b = ceil(X_b - log2 R) and the
 * code of the exact 2^(X - K_b) all in fp64 (orc_directp_map_row_f64).
 * Pinned: the two readings differ only where fp32 rounding moves a value
 * across a decision threshold (a code boundary of 2^t or an integer of
 * X_b - log2 R), checked against the fp64 distance to that threshold. */
void orc_directp_rows_ex(const uint8_t *q_payload, const uint8_t *q_sf, float g_q,
                         const uint8_t *k_payload, const uint8_t *k_sf, float g_k,
                         const uint8_t *v_payload_t, const uint8_t *v_sf,
                         int B, int H, int N, int D, float softmax_scale, int causal, int pv_fmt,
                         int f64_decisions, const int64_t *rows, int nrows,
                         double *o, double *lse,
                         uint8_t *codes, int32_t *kshift, int32_t *mrow,
                         int nthreads);

/* One row of fp64 scores mapped with fp64 decisions (see above). */
void orc_directp_map_row_f64(const double *s, int n, double c, int fmt,
                             uint8_t *codes, int32_t *kshift, int32_t *m_out,
                             double *l_out);

/* The same row pass on explicit scores: for one row of n fp32 scores S,
 * multiplier c and code format fmt, returns the codes (n bytes), K_b per
 * 32-key block, M and l (with p = dec(code)*2^e_b as above).  Used to pin the
 * mapping on hand-worked rows. */
void orc_directp_map_row(const float *s, int n, float c, int fmt,
                         uint8_t *codes, int32_t *kshift, int32_t *m_out,
                         double *l_out);

/* Unquantized softmax attention for the same rows (causal as above), fp64
 * throughout, on the bf16 inputs: X = softmax_scale*log2(e)*q.k, M = max X,
 * p = 2^(X-M).  Pinned: equals a library softmax-attention to 1e-12
 * (Stage A), with and without the causal mask. */
void orc_exact_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    int B, int H, int N, int D, double softmax_scale, int causal,
                    const int64_t *rows, int nrows, double *o, double *lse,
                    int nthreads);

#ifdef __cplusplus
}
#endif
#endif
