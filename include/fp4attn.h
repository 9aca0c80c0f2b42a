/*
 * fp4attn -- Direct-P FP4 attention forward for GB300 (sm_103a).
 *
 * C ABI of the CUDA library libfp4attn.so.  Every call takes plain device
 * pointers (fp4attn_fwd_host_batch also host buffers) and sizes, is
 * asynchronous on the given CUDA stream (a cudaStream_t passed as void*,
 * NULL = legacy default stream), validates its
 * arguments on the host before launching anything, and returns an
 * FP4ATTN_STATUS code.  The caller owns all input and output memory.  No call
 * allocates device memory, except that the first call on a device sets up a
 * 256-byte status word for that device (cudaMalloc once; see
 * fp4attn_device_status).
 *
 * The operation follows "Hardware-Aware FP4 FlashAttention-4" (arXiv
 * 2609.04105); sections cited are those of its neuraltrendhub.com summary
 * page ("What the paper found") and of the abstract.  The method keeps Q and
 * K in NVFP4, maps max-shifted log2 scores directly to MXFP4 E2M1
 * probability codes, sums the softmax denominator from the same rounded
 * probabilities that the PV product consumes, and emits O together with the
 * LSE.  Where the pages fix no formula the library implements these readings:
 *   NVFP4 (Q, K): 16-element blocks along D; g = amax(|x|)/2688 per tensor
 *     (1 when all zero); block scale byte = E4M3(amax_b / (6 g)) (RNE,
 *     saturating); codes = E2M1(x * fp32(1 / (dec(byte) * g))), RNE,
 *     saturating, sign kept; a block whose scale decodes to 0 is all zero.
 *   MXFP4 (V, along keys): 32-key blocks per (b, h, d); scale 2^e with e the
 *     smallest integer >= -127 such that amax <= 6 * 2^e; codes = E2M1(v*2^-e).
 *   Direct-P: c = fp32(softmax_scale * log2(e) * g_Q * g_K);
 *     X = c * S (S the block-scaled FP4 product of the codes);
 *     per 32-key block K_b = ceil(X_b - log2 6) with X_b the block maximum;
 *     code = E2M1(2^(X - K_b)); the block's E8M0 scale is 2^(K_b - M) for an
 *     integer reference maximum M (>= ceil of every score seen so far);
 *     l = sum of the decoded probabilities; O = (P V) / l;
 *     LSE = ln 2 * (M + log2 l), the natural-log log-sum-exp of
 *     softmax_scale * (q . k) as seen through the quantized operands.
 *
 * Data layouts (all row-major, byte addressed):
 *   bf16 inputs/outputs:  [B, H, N, D]
 *   E2M1 packing:         element 2i in bits 0-3 of byte i, 2i+1 in bits 4-7
 *   Q/K payload:          [B, H, N, D/2] bytes
 *   V payload (keys inner, "transposed"): [B, H, D, Npad/2] bytes,
 *                         Npad = N rounded up to a multiple of 128; keys >= N
 *                         hold code 0
 *   scale-factor atoms:   512 bytes cover 128 rows x 4 consecutive scale
 *                         blocks; row r, block k of an atom is the byte at
 *                         (r % 32) * 16 + (r / 32) * 4 + k
 *     Q/K scales: atom [b*H + h][n / 128][block / 4], rows = tokens n,
 *                 blocks = 16-element groups along D   (D/16 per token)
 *     V scales:   atom [b*H + h][n / 128], rows = channels d (D <= 128,
 *                 rows >= D are 0), blocks = 32-key groups of that tile
 *   LSE:                  fp32 [B, H, N]
 *   FP8 P/V variant (MXFP8 V, E4M3 probability codes; "What the paper
 *   found": training keeps FP8 probabilities and values):
 *     V payload: [B, H, D, Npad] bytes, one E4M3 code per key (keys >= N: 0);
 *     V scales:  exactly the MXFP4 V atoms; e is the smallest integer >= -127
 *                with amax <= 448 * 2^e, code = E4M3(v * 2^-e);
 *     P codes:   E4M3(2^(X - K_b)) with K_b = ceil(X_b - log2 448); the rest
 *                of the Direct-P definition is unchanged.
 *
 * Supported shapes: D in {64, 128}; B, H, N >= 1; B*H*N < 2^31.  The
 * quantizers accept any N; fp4attn_fwd_directp accepts any N >= 1 (a partial
 * last key tile is masked, a partial last query tile is not stored).
 * All pointers must be 16-byte aligned.
 */
#ifndef FP4ATTN_H
#define FP4ATTN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum {
    FP4ATTN_OK = 0,
    FP4ATTN_ERR_INVALID_ARG = 1, /* null or misaligned pointer, bad size, non-finite scale */
    FP4ATTN_ERR_UNSUPPORTED = 2, /* D not in {64, 128}, sizes beyond the supported range */
    FP4ATTN_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    FP4ATTN_ERR_TIMEOUT = 4      /* a bounded device-side wait gave up (see fp4attn_device_status) */
};

/* Quantized NVFP4 tensor (Q or K) as written by fp4attn_quant_qk_nvfp4. */
typedef struct {
    const uint8_t *payload; /* [B,H,N,D/2] */
    const uint8_t *sf;      /* scale atoms, fp4attn_nvfp4_bytes(...).sf bytes */
    const float *g;         /* one fp32 tensor scale, in device memory */
} fp4attn_nvfp4_t;

/* Quantized MXFP4 V as written by fp4attn_quant_v_mxfp4. */
typedef struct {
    const uint8_t *payload_t; /* [B,H,D,Npad/2] */
    const uint8_t *sf;        /* scale atoms, fp4attn_mxfp4_v_bytes(...).sf bytes */
} fp4attn_mxfp4_t;

/* Quantized MXFP8 V as written by fp4attn_quant_v_mxfp8. */
typedef struct {
    const uint8_t *payload_t; /* [B,H,D,Npad] */
    const uint8_t *sf;        /* scale atoms, fp4attn_mxfp8_v_bytes(...).sf bytes */
} fp4attn_mxfp8_t;

/* An MXFP8 operand of the backward: FP8 codes and their E8M0 scale atoms,
 * either row-major (fp4attn_quant_mxfp8_rows: [B,H,N,D] bytes, blocks along
 * D) or sequence-blocked and transposed (fp4attn_quant_mxfp8_t: [B,H,D,Npad]
 * bytes, blocks along the sequence). */
typedef struct {
    const uint8_t *payload;
    const uint8_t *sf;
} fp4attn_fp8_t;

/* FP8 code formats of the backward's operands. */
enum {
    FP4ATTN_FP8_E4M3 = 0, /* 4 exponent, 3 mantissa bits, largest 448 (OCP E4M3FN) */
    FP4ATTN_FP8_E5M2 = 1  /* 5 exponent, 2 mantissa bits, largest 57344 */
};

/* Writable buffers of a quantized NVFP4 tensor (outputs of a call). */
typedef struct {
    uint8_t *payload; /* [B,H,N,D/2] */
    uint8_t *sf;      /* scale atoms, fp4attn_nvfp4_bytes(...).sf bytes */
    float *g;         /* one fp32 tensor scale, in device memory */
} fp4attn_nvfp4_buf_t;

/* Writable buffers of a quantized MXFP4 V (outputs of a call). */
typedef struct {
    uint8_t *payload_t; /* [B,H,D,Npad/2] */
    uint8_t *sf;        /* scale atoms, fp4attn_mxfp4_v_bytes(...).sf bytes */
} fp4attn_mxfp4_buf_t;

/* Message for a status code (static string, never NULL). */
const char *fp4attn_status_string(int status);

/* Sizes in bytes of the NVFP4 buffers for a [B,H,N,D] tensor.
 * Returns FP4ATTN_ERR_INVALID_ARG / _UNSUPPORTED for bad shapes. */
int fp4attn_nvfp4_bytes(int B, int H, int N, int D, size_t *payload_bytes, size_t *sf_bytes);

/* Sizes in bytes of the MXFP4 V buffers for a [B,H,N,D] tensor. */
int fp4attn_mxfp4_v_bytes(int B, int H, int N, int D, size_t *payload_bytes, size_t *sf_bytes);

/* Sizes in bytes of the MXFP8 V buffers for a [B,H,N,D] tensor. */
int fp4attn_mxfp8_v_bytes(int B, int H, int N, int D, size_t *payload_bytes, size_t *sf_bytes);

/* NVFP4-quantize Q or K ("What the paper found": NVFP4 for Q and K).
 * x: bf16 [B,H,N,D] (device, read only).  Writes payload, sf (every byte of
 * the padded atoms) and *g (device, 4 bytes; used as the amax accumulator
 * while the call runs).  Launches a memset and three kernels on stream;
 * inputs must be finite. */
int fp4attn_quant_qk_nvfp4(const void *x, uint8_t *payload, uint8_t *sf, float *g,
                           int B, int H, int N, int D, void *stream);

/* MXFP4-quantize V along the key axis, writing it key-inner
 * ("What the paper found": MXFP4 E2M1 P/V operands of the PV product).
 * v: bf16 [B,H,N,D].  Writes payload_t and sf (all bytes, padding included).
 * One kernel; inputs must be finite. */
int fp4attn_quant_v_mxfp4(const void *v, uint8_t *payload_t, uint8_t *sf,
                          int B, int H, int N, int D, void *stream);

/* MXFP8-quantize V along the key axis, written key-inner (the FP8 P/V
 * variant: "What the paper found", training keeps FP8 probabilities and
 * values).  v: bf16 [B,H,N,D].  Writes payload_t and sf (all bytes, padding
 * included).  One kernel; inputs must be finite. */
int fp4attn_quant_v_mxfp8(const void *v, uint8_t *payload_t, uint8_t *sf,
                          int B, int H, int N, int D, void *stream);

/* MXFP8-quantize a bf16 [B,H,N,D] tensor along the sequence, written
 * token-inner: payload_t [B,H,D,Npad] bytes (tokens >= N: code 0) and the
 * scale atoms of fp4attn_mxfp8_v_bytes, laid out as the V atoms (rows =
 * channels, blocks = 32-token groups of each 128-token tile).  e is the
 * smallest integer >= -127 with amax <= fmt_max * 2^e (fmt_max 448 for E4M3,
 * 57344 for E5M2) and code = FP8(x * 2^-e), nearest, ties to even,
 * saturating.  fmt: FP4ATTN_FP8_E4M3 or FP4ATTN_FP8_E5M2 (the backward's
 * E4M3 Q and K and E5M2 output gradient dO; "What the paper found": the
 * backward uses FP8 gradient operands, including E5M2 output gradients).
 * fp4attn_quant_v_mxfp8 is this call with E4M3.  One kernel. */
int fp4attn_quant_mxfp8_t(const void *x, uint8_t *payload_t, uint8_t *sf, int fmt,
                          int B, int H, int N, int D, void *stream);

/* Sizes of the row-major MXFP8 buffers: payload B*H*N*D bytes, scale atoms
 * as fp4attn_mxfp8_v_bytes. */
int fp4attn_mxfp8_rows_bytes(int B, int H, int N, int D, size_t *payload_bytes, size_t *sf_bytes);

/* MXFP8-quantize a bf16 [B,H,N,D] tensor along D, row-major: payload
 * [B,H,N,D] bytes; scale atom [b*H + h][n / 128], row n % 128, block d / 32
 * (blocks d >= D and rows n >= N hold 0).  Same scale rule and codes as
 * fp4attn_quant_mxfp8_t.  The backward's E4M3 V and E5M2 dO for the
 * dP = dO V^T product.  A memset of sf and one kernel. */
int fp4attn_quant_mxfp8_rows(const void *x, uint8_t *payload, uint8_t *sf, int fmt,
                             int B, int H, int N, int D, void *stream);

/* Sizes of the backward's two per-row fp32 arrays (nl2, delta):
 * B*H*Npad floats each, Npad = N rounded up to a multiple of 128. */
int fp4attn_bwd_workspace_bytes(int B, int H, int N, int D, size_t *nl2_bytes, size_t *delta_bytes);

/* First step of the causal backward: delta[b,h,n] = sum_d dO * O (fp32
 * accumulation of the bf16 products) and nl2[b,h,n] = -fp32(lse * fp32(log2 e))
 * (the negated log2-domain LSE) into [B,H,Npad] arrays, with nl2 = -inf and
 * delta = 0 for n >= N.  o, dout: bf16 [B,H,N,D]; lse: fp32 [B,H,N] as the
 * causal forward wrote it.  One kernel. */
int fp4attn_bwd_prep(const void *o, const void *dout, const float *lse, float *nl2, float *delta,
                     int B, int H, int N, int D, void *stream);

/* Causal Direct-P backward ("What the paper found": the backward
 * reconstructs the probabilities from the saved quantized Q/K payloads,
 * scales and LSE values and uses FP8 gradient operands, including E5M2
 * output gradients).  Computes, for query i and key j <= i,
 *   P_ij  = 2^(fp32(c S_ij + nl2_i))  (c, S: the forward's score multiplier
 *                                      and block-scaled NVFP4 product of q, k;
 *                                      ex2 flushes results below 2^-126)
 *   dP_ij = dO~_i . V~_j              (E5M2 dO and E4M3 V, blocks along D)
 *   dS_ij = P_ij (dP_ij - delta_i)    (fp32)
 *   dV_j  = sum_i P~_ij dO~_i                  P~ E4M3, blocks of 32 queries
 *   dK_j  = softmax_scale sum_i dS~_ij Q~_i     dS~ E5M2, blocks of 32 queries
 *   dQ_i  = softmax_scale sum_j dS~_ij K~_j     dS~ E5M2, blocks of 32 keys
 * where X~ is MX block quantization (E8M0 scale per 32 elements along each
 * product's contraction axis, the rule of fp4attn_quant_mxfp8_t).
 * q, k: the NVFP4 tensors the causal forward consumed (saved);
 * v_rows: E4M3 fp4attn_quant_mxfp8_rows of V; do_rows: E5M2 rows of dO;
 * do_t: E5M2 fp4attn_quant_mxfp8_t of dO; q_t, k_t: E4M3
 * fp4attn_quant_mxfp8_t of Q and K; nl2, delta: from fp4attn_bwd_prep;
 * dq, dk, dv: fp32 [B,H,N,D] outputs (every element written).
 * softmax_scale: the forward's (finite, > 0).  Two kernel launches (keys
 * stationary for dK and dV, queries stationary for dQ); errors as
 * fp4attn_fwd_directp. */
int fp4attn_bwd_directp_causal(const fp4attn_nvfp4_t *q, const fp4attn_nvfp4_t *k,
                               const fp4attn_fp8_t *v_rows, const fp4attn_fp8_t *do_rows,
                               const fp4attn_fp8_t *do_t, const fp4attn_fp8_t *q_t, const fp4attn_fp8_t *k_t,
                               const float *nl2, const float *delta, float *dq, float *dk, float *dv,
                               int B, int H, int N, int D, float softmax_scale, void *stream);

/* Noncausal Direct-P forward (abstract: "Direct-P for noncausal inference";
 * "What the paper found": E2M1 probability codes from log-softmax scores,
 * denominator from the same rounded probabilities, LSE).
 * q, k: quantized NVFP4 tensors; v: quantized MXFP4 V; o: bf16 [B,H,N,D];
 * lse: fp32 [B,H,N].  softmax_scale must be finite and > 0.  Block shifts
 * and reference maxima are 32-bit integers, so every scaled score
 * c*S = softmax_scale*log2(e)*q.k must stay below 2^30 in magnitude (for
 * D = 128, amax(q)*amax(k) below about 7e7); larger scores are outside the
 * supported range.  One kernel launch on stream.  Returns
 * FP4ATTN_ERR_TIMEOUT only from fp4attn_device_status; a launch returns OK
 * or an argument/CUDA error. */
int fp4attn_fwd_directp(const fp4attn_nvfp4_t *q, const fp4attn_nvfp4_t *k, const fp4attn_mxfp4_t *v,
                        void *o, float *lse, int B, int H, int N, int D, float softmax_scale,
                        void *stream);

/* Causal Direct-P forward ("What the paper found": for causal training the
 * forward saves the quantized Q/K payloads, scales and LSE for the
 * backward; abstract: the causal path passes the forward quantization into
 * backward).  Query row i attends to keys 0 .. i only; otherwise it computes
 * exactly what fp4attn_fwd_directp computes (same scale rules, mapping,
 * denominator and LSE definition over the keys a row sees), with the same
 * arguments, layouts and errors.  Key tiles wholly above the diagonal are
 * skipped.  One kernel launch on stream. */
int fp4attn_fwd_directp_causal(const fp4attn_nvfp4_t *q, const fp4attn_nvfp4_t *k, const fp4attn_mxfp4_t *v,
                               void *o, float *lse, int B, int H, int N, int D, float softmax_scale,
                               void *stream);

/* Direct-P forward with FP8 P/V operands ("What the paper found": FP8
 * probabilities and values are kept for training; abstract: matched
 * training retains FP8 probabilities and values).  Q and K stay NVFP4; V is
 * MXFP8 (fp4attn_quant_v_mxfp8); the probability codes are E4M3 with the
 * block shift K_b = ceil(X_b - log2 448) and the PV product runs on E4M3
 * operands with UE8M0 block scales.  causal != 0: query row i attends to keys
 * 0 .. i (as fp4attn_fwd_directp_causal), otherwise to all keys.  Other
 * arguments, layouts and errors as fp4attn_fwd_directp.  One kernel launch. */
int fp4attn_fwd_directp_fp8pv(const fp4attn_nvfp4_t *q, const fp4attn_nvfp4_t *k, const fp4attn_mxfp8_t *v,
                              void *o, float *lse, int B, int H, int N, int D, float softmax_scale, int causal,
                              void *stream);

/* The causal training forward in one call: NVFP4-quantizes q and k (bf16
 * [B,H,N,D], device) into the caller's q_saved and k_saved buffers,
 * MXFP4-quantizes v into v_quant, and runs fp4attn_fwd_directp_causal on
 * them.  q_saved, k_saved (payloads, scale atoms, tensor scales) and lse are
 * the state a backward pass reconstructs the probabilities from; the caller
 * owns and keeps them.  Sizes as returned by fp4attn_nvfp4_bytes and
 * fp4attn_mxfp4_v_bytes.  All arguments are checked before anything is
 * launched; launches the two quantizer sequences, the V quantizer and the
 * forward on stream. */
int fp4attn_fwd_directp_causal_save(const void *q, const void *k, const void *v,
                                    const fp4attn_nvfp4_buf_t *q_saved, const fp4attn_nvfp4_buf_t *k_saved,
                                    const fp4attn_mxfp4_buf_t *v_quant, void *o, float *lse,
                                    int B, int H, int N, int D, float softmax_scale, void *stream);

/* Allocation-free variant of fp4attn_fwd_directp (the paper has no
 * counterpart; this is an interface convenience).  Some callers cannot let a
 * library call cudaMalloc: processes that have reserved almost all device
 * memory up front for their own pool (a late allocation fails or fragments
 * it), frameworks that route every device allocation through their own
 * allocator and forbid side allocations, and latency-critical loops where an
 * allocation's implicit device synchronisation is unacceptable.  This entry
 * point computes exactly what fp4attn_fwd_directp computes, with the same
 * arguments, layouts and errors, and never calls cudaMalloc, cudaFree or any
 * allocating routine.  The only memory the forward needs besides the caller's
 * inputs and outputs is its status word (8 bytes, for any problem size); here
 * it lives in a static 256-byte device array that every GPU loading the
 * library holds until the process exits.
 *   - The first call on each device looks up that array's device address
 *     (cudaGetSymbolAddress, with the device current) and caches it; make that
 *     first call before any stream capture begins.
 *   - Every call clears the word on `stream` before launching.  All calls share
 *     the one array, so calls whose work overlaps on the GPU (for example on
 *     two streams) race on it.
 *   - There is no status word to read back: if a bounded device-side wait
 *     gives up, every LSE entry of that call is set to NaN (O is incomplete).
 * Launches a memset, the forward kernel and a small check kernel on stream. */
int fp4attn_fwd_directp_noalloc(const fp4attn_nvfp4_t *q, const fp4attn_nvfp4_t *k, const fp4attn_mxfp4_t *v,
                                void *o, float *lse, int B, int H, int N, int D, float softmax_scale,
                                void *stream);

/* Test support for fp4attn_fwd_directp_noalloc (no counterpart in the paper):
 * drives its failure report without a fault.  Clears the allocation-free
 * entry point's static status word, runs one warp whose bounded wait on an
 * mbarrier that nothing completes gives up after limit_us microseconds
 * (1 .. 10^6) and records the timeout in that word, then runs the same report
 * kernel the entry point runs: every entry of lse[0 .. n) becomes NaN.  lse is
 * a caller-owned fp32 device buffer, 16-byte aligned.  Allocates nothing;
 * FP4ATTN_ERR_INVALID_ARG for a null/misaligned buffer or bad n / limit. */
int fp4attn_debug_noalloc_timeout(float *lse, long long n, int limit_us, void *stream);

/* Test support: *exists = 1 if the library has created its per-device status
 * block (the one cudaMalloc of the library; see fp4attn_device_status) on the
 * current device, 0 if not.  Lets a test show that a sequence of calls --
 * the allocation-free forward above, the quantizers -- never created it.
 * FP4ATTN_ERR_INVALID_ARG for a null pointer. */
int fp4attn_debug_status_word_exists(int *exists);

/* Same computation as fp4attn_fwd_directp (same kernel, same launch shape),
 * and in addition writes the probability codes, block shifts and fp32 output
 * of query rows row0 .. row0+nrows-1 of head (b, h):
 *   codes:  [nrows, Npad/2] bytes, packed like the payloads (keys >= N are 0)
 *   kshift: [nrows, Npad/32] int32 block shifts K_b (0 for blocks past N)
 *   o_f32:  [nrows, D] fp32, the normalised output before its bf16 rounding
 * For parity tests; O and LSE are written exactly as by the forward call. */
int fp4attn_debug_dump_p(const fp4attn_nvfp4_t *q, const fp4attn_nvfp4_t *k, const fp4attn_mxfp4_t *v,
                         void *o, float *lse, int B, int H, int N, int D, float softmax_scale,
                         int b, int h, int row0, int nrows, uint8_t *codes, int32_t *kshift,
                         float *o_f32, void *stream);

/* fp4attn_debug_dump_p for the causal forward: the same outputs, where the
 * codes and shifts of keys past a row's diagonal are 0.  Clears codes and
 * kshift on stream first (the kernel never visits key tiles past the
 * diagonal). */
int fp4attn_debug_dump_p_causal(const fp4attn_nvfp4_t *q, const fp4attn_nvfp4_t *k, const fp4attn_mxfp4_t *v,
                                void *o, float *lse, int B, int H, int N, int D, float softmax_scale,
                                int b, int h, int row0, int nrows, uint8_t *codes, int32_t *kshift,
                                float *o_f32, void *stream);

/* fp4attn_debug_dump_p for the FP8 P/V forward: codes are E4M3 bytes,
 * [nrows, Npad] (one byte per key); kshift and o_f32 as there.  Clears codes
 * and kshift on stream first. */
int fp4attn_debug_dump_p_fp8pv(const fp4attn_nvfp4_t *q, const fp4attn_nvfp4_t *k, const fp4attn_mxfp8_t *v,
                               void *o, float *lse, int B, int H, int N, int D, float softmax_scale, int causal,
                               int b, int h, int row0, int nrows, uint8_t *codes, int32_t *kshift,
                               float *o_f32, void *stream);

/* Test support (no counterpart in the method): for format 0 (E2M1), 1
 * (E4M3) or 2 (E5M2), converts every fp32 bit pattern u in [lo, hi] with the hardware
 * round-to-nearest-even saturating conversion the library uses, and records
 * into pairs[2i], pairs[2i+1] (device, capacity pairs) each pattern u > lo
 * whose code differs from that of u-1, plus the pair (lo, code(lo)); *count
 * (device int) receives the number of pairs found (may exceed capacity; the
 * order of pairs is unspecified). */
int fp4attn_debug_cvt_transitions(int format, uint32_t lo, uint32_t hi, uint32_t *pairs, int capacity,
                                  int *count, void *stream);

/* Test support (no counterpart in the method): exercises the failure path of
 * the bounded device-side waits without any fault.  One warp waits on an
 * mbarrier that nothing arrives at, through the same bounded wait the forward
 * uses but limited to limit_us microseconds (1 .. 1000000); the wait gives up,
 * sets the status word (read it with fp4attn_device_status, which then reports
 * FP4ATTN_ERR_TIMEOUT once) and the kernel returns normally. */
int fp4attn_debug_wait_timeout(int limit_us, void *stream);

/* Measurement support (no counterpart on the pages): the dense tensor-core
 * rate of the block-scaled products the forward issues, the denominator of
 * its roofline.  Launches one CTA per SM; one thread per CTA issues `iters`
 * rounds of M = 128, N = 128, K = 128 products (2*128^3 FLOP per round) from
 * shared-memory operands into a TMEM accumulator:
 *   kind 0  kind::mxf4nvf4, E2M1 x E2M1, 16-element UE4M3 scales (QK^T form)
 *   kind 1  kind::mxf4,     E2M1 x E2M1, 32-element UE8M0 scales (PV form)
 *   kind 2  kind::mxf8f6f4, E4M3 x E4M3, 32-element UE8M0 scales (FP8 PV form)
 * The caller times the launch on `stream` (FLOP = SMs * iters * 2 * 128^3).
 * Errors: FP4ATTN_ERR_INVALID_ARG for kind outside 0..2 or iters outside
 * 1..2^26; a wait that gives up shows in fp4attn_device_status. */
int fp4attn_debug_mma_peak(int kind, int iters, void *stream);

/* Flags of fp4attn_fwd_host_batch: which forward each step runs. */
enum {
    FP4ATTN_HB_CAUSAL = 1, /* fp4attn_fwd_directp_causal (with FP8PV: causal FP8 P/V) */
    FP4ATTN_HB_FP8PV = 2   /* MXFP8 V and fp4attn_fwd_directp_fp8pv */
};

/* Workspace size (bytes) of fp4attn_fwd_host_batch for one problem shape and
 * flags: two slots of bf16 Q, K, V, O and fp32 LSE, plus one set of quantized
 * Q, K (NVFP4) and V (MXFP4, or MXFP8 with FP4ATTN_HB_FP8PV), each region
 * 256-byte aligned.  Errors: bad shape, null bytes or unknown flags. */
int fp4attn_fwd_host_batch_workspace_bytes(int B, int H, int N, int D, int flags, size_t *bytes);

/* The forward of nsteps independent problems of one shape, from HOST memory
 * to HOST memory (the paper has no counterpart; this is the serving-loop form
 * of the calls above: the abstract's forward, run on data that lives on the
 * host).  Step i reads bf16 [B,H,N,D] q_h[i], k_h[i], v_h[i] and writes bf16
 * o_h[i] and fp32 [B,H,N] lse_h[i]; it computes exactly what
 * fp4attn_quant_qk_nvfp4 (Q, K), fp4attn_quant_v_mxfp4 or _mxfp8 (V) and the
 * forward chosen by flags compute on device copies of those buffers.
 * Pointer arrays and host buffers are the caller's; the host buffers must
 * stay valid and untouched until the work completes (synchronise `stream`),
 * and should be pinned (cudaHostAlloc / cudaHostRegister), or the copies
 * do not overlap the kernels.  workspace: a device buffer of at least
 * fp4attn_fwd_host_batch_workspace_bytes bytes, 256-byte aligned, owned by
 * the caller and used by no other work until the call's work completes; it,
 * `stream` and the call's own streams belong to the current device.
 * Pipelining: an upload and a download stream of the call's own run beside
 * `stream`, ordered by events, so step i+1's upload and step i-1's download
 * overlap step i's kernels; the kernels run on `stream`, which is made to
 * wait for the last download before the call returns, so events recorded on
 * `stream` before and after the call span every copy.  All arguments are
 * checked before anything is queued (FP4ATTN_ERR_INVALID_ARG / _UNSUPPORTED);
 * a CUDA error while queueing stops the queueing and returns
 * FP4ATTN_ERR_CUDA, with the work already queued still ordered before
 * `stream`.  Bounded device-side waits that give up show in
 * fp4attn_device_status.  Allocates no device memory; creates and releases
 * two streams and eight events per call. */
int fp4attn_fwd_host_batch(int nsteps, const void *const *q_h, const void *const *k_h, const void *const *v_h,
                           void *const *o_h, float *const *lse_h, int B, int H, int N, int D,
                           float softmax_scale, int flags, void *workspace, size_t workspace_bytes,
                           void *stream);

/* Reads and clears the status word the kernels of this library set when a
 * bounded device-side wait gives up (they then stop early and leave their
 * outputs incomplete).  Synchronises the given stream first.  Returns
 * FP4ATTN_OK or FP4ATTN_ERR_TIMEOUT (or _CUDA if the readback fails). */
int fp4attn_device_status(void *stream);

#ifdef __cplusplus
}
#endif
#endif
