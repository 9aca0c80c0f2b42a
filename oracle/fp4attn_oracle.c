/*
 * fp4attn oracle -- TEST INFRASTRUCTURE ONLY (see fp4attn_oracle.h).
 *
 * Plain C11, compiled with -ffp-contract=off so that every fp32 expression
 * rounds exactly as written; fused multiply-adds appear only where fmaf() is
 * called by name.  Nothing here is shared with the CUDA library.
 *
 * Method source: "Hardware-Aware FP4 FlashAttention-4", neuraltrendhub.com
 * summary page, "What the paper found" (NVFP4 Q/K, E2M1 probability codes
 * mapped from max-shifted log2 scores, denominator from the rounded
 * probabilities, LSE saved by the forward pass).
 */
#include "fp4attn_oracle.h"

#include <assert.h>
#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* small helpers                                                            */
/* ------------------------------------------------------------------------ */

static float bf16_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

typedef struct {
    void (*fn)(void *ctx, long lo, long hi);
    void *ctx;
    long lo, hi;
} range_job;

static void *range_job_run(void *p) {
    range_job *j = (range_job *)p;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

/* Runs fn over [0, n) split into nthreads contiguous chunks. */
static void parallel_for(long n, int nthreads, void (*fn)(void *, long, long), void *ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < nthreads) nthreads = n > 0 ? (int)n : 1;
    if (nthreads == 1) {
        fn(ctx, 0, n);
        return;
    }
    pthread_t tid[256];
    range_job jobs[256];
    long chunk = (n + nthreads - 1) / nthreads;
    int started = 0;
    for (int t = 0; t < nthreads; t++) {
        long lo = t * chunk, hi = lo + chunk < n ? lo + chunk : n;
        if (lo >= hi) break;
        jobs[t].fn = fn;
        jobs[t].ctx = ctx;
        jobs[t].lo = lo;
        jobs[t].hi = hi;
        if (pthread_create(&tid[t], NULL, range_job_run, &jobs[t]) != 0) {
            range_job_run(&jobs[t]); /* run inline if a thread cannot start */
            tid[t] = 0;
        }
        started = t + 1;
    }
    for (int t = 0; t < started; t++)
        if (tid[t]) pthread_join(tid[t], NULL);
}

/* ------------------------------------------------------------------------ */
/* number formats                                                           */
/* ------------------------------------------------------------------------ */

/* E2M1 magnitudes by code: exponent bits 2..1, mantissa bit 0, bias 1;
 * exponent field 0 is the subnormal 0.5*m. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1_decode(uint8_t code) {
    double m = E2M1_MAG[code & 7];
    return (code & 8) ? -m : m;
}

uint8_t orc_e2m1_encode(double y) {
    assert(!isnan(y));
    uint8_t sign = signbit(y) ? 8 : 0;
    double a = fabs(y);
    if (a >= 6.0) return sign | 7; /* saturate to the largest finite value */
    int best = 0;
    double bestd = a;
    for (int k = 1; k < 8; k++) {
        double d = fabs(a - E2M1_MAG[k]);
        /* strictly nearer wins; on a tie the even code wins */
        if (d < bestd || (d == bestd && (k % 2) == 0)) {
            best = k;
            bestd = d;
        }
    }
    return (uint8_t)(sign | best);
}

double orc_e4m3_decode(uint8_t code) {
    int e = (code >> 3) & 15, m = code & 7;
    assert((code & 0x7F) != 0x7F); /* NaN has no value */
    double v = (e == 0) ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return (code & 0x80) ? -v : v;
}

uint8_t orc_e4m3_encode(double y) {
    assert(!isnan(y));
    uint8_t sign = signbit(y) ? 0x80 : 0;
    double a = fabs(y);
    if (a >= 448.0) return sign | 0x7E; /* saturate to the largest finite value */
    int best = 0;
    double bestd = a;
    for (int c = 1; c <= 0x7E; c++) {
        double d = fabs(a - orc_e4m3_decode((uint8_t)c));
        if (d < bestd || (d == bestd && (c % 2) == 0)) {
            best = c;
            bestd = d;
        }
    }
    return (uint8_t)(sign | best);
}

double orc_e8m0_decode(uint8_t code) {
    assert(code != 0xFF);
    return ldexp(1.0, (int)code - 127);
}

/* ------------------------------------------------------------------------ */
/* scale-factor atoms                                                       */
/* ------------------------------------------------------------------------ */

size_t orc_sf_index(size_t bh, int n_row_tiles, int row, int kblock, int kblocks_per_row) {
    int tile = row / 128, r = row % 128;
    int atom = kblock / 4, k = kblock % 4;
    int atoms_per_tile = kblocks_per_row / 4;
    size_t a = ((bh * (size_t)n_row_tiles + (size_t)tile) * (size_t)atoms_per_tile + (size_t)atom);
    return a * 512 + (size_t)((r % 32) * 16 + (r / 32) * 4 + k);
}

static int row_tiles(int N) { return (N + 127) / 128; }

/* ------------------------------------------------------------------------ */
/* NVFP4 quantizer (Q, K)                                                   */
/* ------------------------------------------------------------------------ */

size_t orc_nvfp4_sf_bytes(int B, int H, int N, int D) {
    return (size_t)B * H * row_tiles(N) * (size_t)(D / 64) * 512;
}

typedef struct {
    const uint16_t *x;
    int B, H, N, D;
    uint8_t *payload, *sf;
    float g;
} nvfp4_ctx;

static void nvfp4_rows_chunk(void *p, long lo, long hi) {
    nvfp4_ctx *c = (nvfp4_ctx *)p;
    const int D = c->D, KB = D / 16;
    const float g = c->g;
    for (long row = lo; row < hi; row++) {
        long bh = row / c->N;
        int n = (int)(row % c->N);
        const uint16_t *xr = c->x + row * D;
        for (int kb = 0; kb < KB; kb++) {
            float amax_b = 0.0f;
            for (int e = 0; e < 16; e++) {
                float a = fabsf(bf16_to_float(xr[kb * 16 + e]));
                if (a > amax_b) amax_b = a;
            }
            float denom = 6.0f * g;
            float t = amax_b / denom;
            uint8_t sb = orc_e4m3_encode((double)t);
            float s = (float)orc_e4m3_decode(sb) * g;
            c->sf[orc_sf_index((size_t)bh, row_tiles(c->N), n, kb, KB)] = sb;
            float inv = (s != 0.0f) ? 1.0f / s : 0.0f;
            for (int e = 0; e < 16; e += 2) {
                uint8_t lo4 = 0, hi4 = 0;
                if (s != 0.0f) {
                    float y0 = bf16_to_float(xr[kb * 16 + e]) * inv;
                    float y1 = bf16_to_float(xr[kb * 16 + e + 1]) * inv;
                    lo4 = orc_e2m1_encode((double)y0);
                    hi4 = orc_e2m1_encode((double)y1);
                }
                c->payload[row * (D / 2) + (kb * 16 + e) / 2] = (uint8_t)(lo4 | (hi4 << 4));
            }
        }
    }
}

void orc_quant_nvfp4(const uint16_t *x, int B, int H, int N, int D,
                     uint8_t *payload, uint8_t *sf, float *g_out, int nthreads) {
    assert(D % 64 == 0);
    long total = (long)B * H * N * D;
    nvfp4_ctx c = {x, B, H, N, D, payload, sf, 1.0f};

    /* tensor amax (exact: a maximum of magnitudes) */
    float amax = 0.0f;
    for (long i = 0; i < total; i++) {
        float a = fabsf(bf16_to_float(x[i]));
        if (a > amax) amax = a;
    }
    c.g = (amax > 0.0f) ? amax / 2688.0f : 1.0f;
    *g_out = c.g;

    memset(sf, 0, orc_nvfp4_sf_bytes(B, H, N, D));
    parallel_for((long)B * H * N, nthreads, nvfp4_rows_chunk, &c);
}

/* ------------------------------------------------------------------------ */
/* MXFP4 quantizer (V, along keys, transposed)                              */
/* ------------------------------------------------------------------------ */

size_t orc_mxfp4_sf_bytes(int B, int H, int N, int D) {
    (void)D;
    return (size_t)B * H * row_tiles(N) * 512;
}

typedef struct {
    const uint16_t *v;
    int B, H, N, D;
    uint8_t *payload_t, *sf;
} mxfp4_ctx;

static void mxfp4_chunk(void *p, long lo, long hi) {
    mxfp4_ctx *c = (mxfp4_ctx *)p;
    const int N = c->N, D = c->D, Npad = row_tiles(N) * 128;
    for (long unit = lo; unit < hi; unit++) { /* unit = bh*D + d */
        long bh = unit / D;
        int d = (int)(unit % D);
        uint8_t *prow = c->payload_t + unit * (Npad / 2);
        for (int kb = 0; kb < Npad / 32; kb++) {
            float amax = 0.0f;
            for (int j = 0; j < 32; j++) {
                int n = kb * 32 + j;
                if (n >= N) break;
                float a = fabsf(bf16_to_float(c->v[(bh * N + n) * D + d]));
                if (a > amax) amax = a;
            }
            int e = -127;
            while (e < 127 && (double)amax > ldexp(6.0, e)) e++;
            /* atom row = d (padded to 128), block = key block within the tile */
            size_t atom = (size_t)bh * row_tiles(N) + (size_t)(kb / 4);
            c->sf[atom * 512 + (size_t)((d % 32) * 16 + (d / 32) * 4 + (kb % 4))] = (uint8_t)(e + 127);
            for (int j = 0; j < 32; j += 2) {
                uint8_t nib[2] = {0, 0};
                for (int u = 0; u < 2; u++) {
                    int n = kb * 32 + j + u;
                    if (n < N) {
                        double y = ldexp((double)bf16_to_float(c->v[(bh * N + n) * D + d]), -e);
                        nib[u] = orc_e2m1_encode(y);
                    }
                }
                prow[(kb * 32 + j) / 2] = (uint8_t)(nib[0] | (nib[1] << 4));
            }
        }
    }
}

void orc_quant_mxfp4_v(const uint16_t *v, int B, int H, int N, int D,
                       uint8_t *payload_t, uint8_t *sf, int nthreads) {
    assert(D <= 128);
    mxfp4_ctx c = {v, B, H, N, D, payload_t, sf};
    memset(sf, 0, orc_mxfp4_sf_bytes(B, H, N, D));
    parallel_for((long)B * H * D, nthreads, mxfp4_chunk, &c);
}

/* ------------------------------------------------------------------------ */
/* MXFP8 quantizer (V, along keys, transposed)                              */
/* ------------------------------------------------------------------------ */

/* The same 32-key blocks and E8M0 scale atoms as MXFP4 V; the scale is the
 * smallest power of two 2^e (e >= -127) with amax <= 448 * 2^e, and each code
 * is E4M3(v * 2^-e), one byte per key. */
static void mxfp8_chunk(void *p, long lo, long hi) {
    mxfp4_ctx *c = (mxfp4_ctx *)p;
    const int N = c->N, D = c->D, Npad = row_tiles(N) * 128;
    for (long unit = lo; unit < hi; unit++) { /* unit = bh*D + d */
        long bh = unit / D;
        int d = (int)(unit % D);
        uint8_t *prow = c->payload_t + unit * Npad;
        for (int kb = 0; kb < Npad / 32; kb++) {
            float amax = 0.0f;
            for (int j = 0; j < 32; j++) {
                int n = kb * 32 + j;
                if (n >= N) break;
                float a = fabsf(bf16_to_float(c->v[(bh * N + n) * D + d]));
                if (a > amax) amax = a;
            }
            int e = -127;
            while (e < 127 && (double)amax > ldexp(448.0, e)) e++;
            size_t atom = (size_t)bh * row_tiles(N) + (size_t)(kb / 4);
            c->sf[atom * 512 + (size_t)((d % 32) * 16 + (d / 32) * 4 + (kb % 4))] = (uint8_t)(e + 127);
            for (int j = 0; j < 32; j++) {
                int n = kb * 32 + j;
                uint8_t code = 0;
                if (n < N) code = orc_e4m3_encode(ldexp((double)bf16_to_float(c->v[(bh * N + n) * D + d]), -e));
                prow[kb * 32 + j] = code;
            }
        }
    }
}

void orc_quant_mxfp8_v(const uint16_t *v, int B, int H, int N, int D,
                       uint8_t *payload_t, uint8_t *sf, int nthreads) {
    assert(D <= 128);
    mxfp4_ctx c = {v, B, H, N, D, payload_t, sf};
    memset(sf, 0, orc_mxfp4_sf_bytes(B, H, N, D));
    parallel_for((long)B * H * D, nthreads, mxfp8_chunk, &c);
}

/* ------------------------------------------------------------------------ */
/* Direct-P row mapping                                                     */
/* ------------------------------------------------------------------------ */

/* log2(6) rounded to fp32; the block shift K_b = ceil(X_b - log2 6) is the
 * smallest integer with X_b - K_b <= log2 6, i.e. with the block's largest
 * probability 2^(X_b - K_b) within E2M1's largest finite value 6. */
static const float LOG2_6_F32 = 2.5849625007211561f;
/* log2(448) rounded to fp32: the same rule for E4M3 probability codes, whose
 * largest finite value is 448. */
static const float LOG2_448_F32 = 8.8073549220576041f;

/* 2^t for an fp32 t, in fp64: exact for integers, correctly rounded libm
 * otherwise (the decision it feeds is taken against irrational thresholds). */
static double exp2_exact(float t) {
    if (t == floorf(t)) return ldexp(1.0, (int)t);
    return exp2((double)t);
}

/* One row: scores s[0..n), multiplier c, code format fmt (ORC_PV_MXFP4:
 * E2M1, ORC_PV_MXFP8: E4M3).  Returns codes, K_b, M and l. */
void orc_directp_map_row(const float *s, int n, float c, int fmt,
                         uint8_t *codes, int32_t *kshift, int32_t *m_out,
                         double *l_out) {
    const float log2_max = (fmt == ORC_PV_MXFP8) ? LOG2_448_F32 : LOG2_6_F32;
    int nblk = (n + 31) / 32;
    float xmax = -INFINITY;
    for (int j = 0; j < n; j++) {
        float x = c * s[j];
        if (x > xmax) xmax = x;
    }
    int32_t M = (int32_t)ceilf(xmax);
    double l = 0.0;
    for (int b = 0; b < nblk; b++) {
        int j0 = b * 32, j1 = j0 + 32 < n ? j0 + 32 : n;
        float xb = -INFINITY;
        for (int j = j0; j < j1; j++) {
            float x = c * s[j];
            if (x > xb) xb = x;
        }
        int32_t K = (int32_t)ceilf(xb - log2_max);
        kshift[b] = K;
        int e = K - M;
        if (e < -127) e = -127;
        double scale = ldexp(1.0, e);
        for (int j = j0; j < j1; j++) {
            float t = fmaf(c, s[j], (float)(-K));
            double p = exp2_exact(t);
            uint8_t code = (fmt == ORC_PV_MXFP8) ? orc_e4m3_encode(p) : orc_e2m1_encode(p);
            codes[j] = code;
            l += ((fmt == ORC_PV_MXFP8) ? orc_e4m3_decode(code) : orc_e2m1_decode(code)) * scale;
        }
    }
    *m_out = M;
    *l_out = l;
}

/* The same row mapping with every decision taken in fp64: X = c*S in fp64
 * (S and c not rounded to fp32), K_b = ceil(X_b - log2 R) with the fp64
 * log2 R, code = E2M1/E4M3 of the exact 2^(X - K_b).  This is the plainest
 * reading of the mapping ("What the paper found": scores mapped directly to
 * codes); orc_directp_map_row takes the same decisions in fp32, the
 * precision the forward kernel computes in. */
void orc_directp_map_row_f64(const double *s, int n, double c, int fmt,
                             uint8_t *codes, int32_t *kshift, int32_t *m_out,
                             double *l_out) {
    const double log2_max = log2((fmt == ORC_PV_MXFP8) ? 448.0 : 6.0);
    int nblk = (n + 31) / 32;
    double xmax = -INFINITY;
    for (int j = 0; j < n; j++) {
        double x = c * s[j];
        if (x > xmax) xmax = x;
    }
    int32_t M = (int32_t)ceil(xmax);
    double l = 0.0;
    for (int b = 0; b < nblk; b++) {
        int j0 = b * 32, j1 = j0 + 32 < n ? j0 + 32 : n;
        double xb = -INFINITY;
        for (int j = j0; j < j1; j++) {
            double x = c * s[j];
            if (x > xb) xb = x;
        }
        int32_t K = (int32_t)ceil(xb - log2_max);
        kshift[b] = K;
        int e = K - M;
        if (e < -127) e = -127;
        double scale = ldexp(1.0, e);
        for (int j = j0; j < j1; j++) {
            double p = exp2(c * s[j] - (double)K);
            uint8_t code = (fmt == ORC_PV_MXFP8) ? orc_e4m3_encode(p) : orc_e2m1_encode(p);
            codes[j] = code;
            l += ((fmt == ORC_PV_MXFP8) ? orc_e4m3_decode(code) : orc_e2m1_decode(code)) * scale;
        }
    }
    *m_out = M;
    *l_out = l;
}

/* ------------------------------------------------------------------------ */
/* Direct-P attention rows                                                  */
/* ------------------------------------------------------------------------ */

static const double LOG2E = 1.4426950408889634074;
static const double LN2 = 0.69314718055994530942;

typedef struct {
    /* inputs */
    const uint8_t *qp, *qsf, *kp, *ksf, *vp, *vsf;
    float gq, gk, c;
    int B, H, N, D;
    int causal; /* row i sees keys 0..i only */
    int pv_fmt; /* ORC_PV_MXFP4 or ORC_PV_MXFP8 */
    int f64_decisions; /* map with orc_directp_map_row_f64 (fp64 S, c, X) */
    double c64; /* the multiplier in fp64 */
    /* per-head decoded operands */
    long bh;
    double *khat; /* [N][D] */
    double *vhat; /* [N][D] (un-transposed for the row pass) */
    /* rows of this head: indices into the caller's arrays */
    const int64_t *rows;
    const int *sel;
    /* outputs */
    double *o, *lse;
    uint8_t *codes;
    int32_t *kshift, *mrow;
} attn_ctx;

static void decode_head_chunk(void *p, long lo, long hi) {
    attn_ctx *a = (attn_ctx *)p;
    const int N = a->N, D = a->D, KB = D / 16, Npad = row_tiles(N) * 128;
    for (long n = lo; n < hi; n++) {
        const uint8_t *kr = a->kp + ((size_t)a->bh * N + (size_t)n) * (D / 2);
        for (int d = 0; d < D; d++) {
            uint8_t byte = kr[d / 2];
            uint8_t code = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            uint8_t sfb = a->ksf[orc_sf_index((size_t)a->bh, row_tiles(N), (int)n, d / 16, KB)];
            a->khat[n * D + d] = orc_e2m1_decode(code) * orc_e4m3_decode(sfb);
        }
        for (int d = 0; d < D; d++) {
            size_t atom = (size_t)a->bh * row_tiles(N) + (size_t)(n / 128);
            int kb = (int)((n % 128) / 32);
            uint8_t sfb = a->vsf[atom * 512 + (size_t)((d % 32) * 16 + (d / 32) * 4 + kb)];
            if (a->pv_fmt == ORC_PV_MXFP8) {
                const uint8_t *vr = a->vp + ((size_t)a->bh * D + (size_t)d) * Npad;
                a->vhat[n * D + d] = orc_e4m3_decode(vr[n]) * orc_e8m0_decode(sfb);
            } else {
                const uint8_t *vr = a->vp + ((size_t)a->bh * D + (size_t)d) * (Npad / 2);
                uint8_t byte = vr[n / 2];
                uint8_t code = (n % 2 == 0) ? (byte & 0xF) : (byte >> 4);
                a->vhat[n * D + d] = orc_e2m1_decode(code) * orc_e8m0_decode(sfb);
            }
        }
    }
}

static void attn_rows_chunk(void *p, long lo, long hi) {
    attn_ctx *a = (attn_ctx *)p;
    const int N = a->N, D = a->D, KB = D / 16, Npad = row_tiles(N) * 128;
    double *qhat = (double *)malloc(sizeof(double) * (size_t)D);
    float *s32 = (float *)malloc(sizeof(float) * (size_t)N);
    double *s64 = (double *)malloc(sizeof(double) * (size_t)N);
    uint8_t *codes = (uint8_t *)malloc((size_t)Npad);
    int32_t *ks = (int32_t *)malloc(sizeof(int32_t) * (size_t)(Npad / 32));
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    for (long u = lo; u < hi; u++) {
        int r = a->sel[u];
        long flat = (long)a->rows[r];
        int i = (int)(flat % N);
        const uint8_t *qr = a->qp + (size_t)flat * (D / 2);
        for (int d = 0; d < D; d++) {
            uint8_t byte = qr[d / 2];
            uint8_t code = (d % 2 == 0) ? (byte & 0xF) : (byte >> 4);
            uint8_t sfb = a->qsf[orc_sf_index((size_t)a->bh, row_tiles(N), i, d / 16, KB)];
            qhat[d] = orc_e2m1_decode(code) * orc_e4m3_decode(sfb);
        }
        /* the keys this row sees: all of them, or (causal) keys 0..i */
        const int nk = a->causal ? i + 1 : N;
        for (int j = 0; j < nk; j++) {
            double s = 0.0;
            for (int d = 0; d < D; d++) s += qhat[d] * a->khat[(size_t)j * D + d];
            s32[j] = (float)s;
            s64[j] = s;
        }
        memset(codes, 0, (size_t)Npad);
        memset(ks, 0, sizeof(int32_t) * (size_t)(Npad / 32));
        int32_t M;
        double l;
        if (a->f64_decisions)
            orc_directp_map_row_f64(s64, nk, a->c64, a->pv_fmt, codes, ks, &M, &l);
        else
            orc_directp_map_row(s32, nk, a->c, a->pv_fmt, codes, ks, &M, &l);
        for (int d = 0; d < D; d++) acc[d] = 0.0;
        for (int j = 0; j < nk; j++) {
            int e = ks[j / 32] - M;
            if (e < -127) e = -127;
            double dec = (a->pv_fmt == ORC_PV_MXFP8) ? orc_e4m3_decode(codes[j]) : orc_e2m1_decode(codes[j]);
            double pj = dec * ldexp(1.0, e);
            if (pj == 0.0) continue;
            for (int d = 0; d < D; d++) acc[d] += pj * a->vhat[(size_t)j * D + d];
        }
        for (int d = 0; d < D; d++) a->o[(size_t)r * D + d] = acc[d] / l;
        a->lse[r] = LN2 * ((double)M + log2(l));
        if (a->codes) memcpy(a->codes + (size_t)r * Npad, codes, (size_t)Npad);
        if (a->kshift) memcpy(a->kshift + (size_t)r * (Npad / 32), ks, sizeof(int32_t) * (size_t)(Npad / 32));
        if (a->mrow) a->mrow[r] = M;
    }
    free(qhat);
    free(s32);
    free(s64);
    free(codes);
    free(ks);
    free(acc);
}

void orc_directp_rows(const uint8_t *q_payload, const uint8_t *q_sf, float g_q,
                      const uint8_t *k_payload, const uint8_t *k_sf, float g_k,
                      const uint8_t *v_payload_t, const uint8_t *v_sf,
                      int B, int H, int N, int D, float softmax_scale, int causal, int pv_fmt,
                      const int64_t *rows, int nrows,
                      double *o, double *lse,
                      uint8_t *codes, int32_t *kshift, int32_t *mrow,
                      int nthreads) {
    orc_directp_rows_ex(q_payload, q_sf, g_q, k_payload, k_sf, g_k, v_payload_t, v_sf, B, H, N, D,
                        softmax_scale, causal, pv_fmt, 0, rows, nrows, o, lse, codes, kshift, mrow, nthreads);
}

void orc_directp_rows_ex(const uint8_t *q_payload, const uint8_t *q_sf, float g_q,
                         const uint8_t *k_payload, const uint8_t *k_sf, float g_k,
                         const uint8_t *v_payload_t, const uint8_t *v_sf,
                         int B, int H, int N, int D, float softmax_scale, int causal, int pv_fmt,
                         int f64_decisions, const int64_t *rows, int nrows,
                         double *o, double *lse,
                         uint8_t *codes, int32_t *kshift, int32_t *mrow,
                         int nthreads) {
    attn_ctx a;
    memset(&a, 0, sizeof a);
    a.qp = q_payload;
    a.qsf = q_sf;
    a.kp = k_payload;
    a.ksf = k_sf;
    a.vp = v_payload_t;
    a.vsf = v_sf;
    a.gq = g_q;
    a.gk = g_k;
    a.B = B;
    a.H = H;
    a.N = N;
    a.D = D;
    a.causal = causal;
    a.pv_fmt = pv_fmt;
    /* the log2-domain score multiplier, rounded once to fp32 (and kept in
     * fp64 for the fp64-decision reading) */
    a.c64 = (((double)softmax_scale * LOG2E) * (double)g_q) * (double)g_k;
    a.c = (float)a.c64;
    a.f64_decisions = f64_decisions;
    a.rows = rows;
    a.o = o;
    a.lse = lse;
    a.codes = codes;
    a.kshift = kshift;
    a.mrow = mrow;
    a.khat = (double *)malloc(sizeof(double) * (size_t)N * D);
    a.vhat = (double *)malloc(sizeof(double) * (size_t)N * D);
    int *sel = (int *)malloc(sizeof(int) * (size_t)(nrows > 0 ? nrows : 1));
    char *done = (char *)calloc((size_t)(nrows > 0 ? nrows : 1), 1);
    a.sel = sel;
    for (int r0 = 0; r0 < nrows; r0++) {
        if (done[r0]) continue;
        long bh = (long)(rows[r0] / N);
        int cnt = 0;
        for (int r = r0; r < nrows; r++)
            if (!done[r] && (long)(rows[r] / N) == bh) {
                sel[cnt++] = r;
                done[r] = 1;
            }
        a.bh = bh;
        parallel_for(N, nthreads, decode_head_chunk, &a);
        parallel_for(cnt, nthreads, attn_rows_chunk, &a);
    }
    free(a.khat);
    free(a.vhat);
    free(sel);
    free(done);
}

/* ------------------------------------------------------------------------ */
/* unquantized attention                                                    */
/* ------------------------------------------------------------------------ */

typedef struct {
    const uint16_t *q, *k, *v;
    int N, D;
    double scale;
    int causal;
    const int64_t *rows;
    double *o, *lse;
} exact_ctx;

static void exact_chunk(void *p, long lo, long hi) {
    exact_ctx *a = (exact_ctx *)p;
    const int N = a->N, D = a->D;
    double *x = (double *)malloc(sizeof(double) * (size_t)N);
    for (long r = lo; r < hi; r++) {
        long flat = (long)a->rows[r];
        long bh = flat / N;
        const uint16_t *qr = a->q + (size_t)flat * D;
        const int nk = a->causal ? (int)(flat % N) + 1 : N; /* keys the row sees */
        double M = -INFINITY;
        for (int j = 0; j < nk; j++) {
            const uint16_t *kr = a->k + ((size_t)bh * N + (size_t)j) * D;
            double s = 0.0;
            for (int d = 0; d < D; d++) s += (double)bf16_to_float(qr[d]) * (double)bf16_to_float(kr[d]);
            x[j] = a->scale * LOG2E * s;
            if (x[j] > M) M = x[j];
        }
        double l = 0.0;
        for (int j = 0; j < nk; j++) {
            x[j] = exp2(x[j] - M);
            l += x[j];
        }
        for (int d = 0; d < D; d++) {
            double acc = 0.0;
            for (int j = 0; j < nk; j++)
                acc += x[j] * (double)bf16_to_float(a->v[((size_t)bh * N + (size_t)j) * D + d]);
            a->o[(size_t)r * D + d] = acc / l;
        }
        a->lse[r] = LN2 * (M + log2(l));
    }
    free(x);
}

void orc_exact_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    int B, int H, int N, int D, double softmax_scale, int causal,
                    const int64_t *rows, int nrows, double *o, double *lse,
                    int nthreads) {
    (void)B;
    (void)H;
    exact_ctx a = {q, k, v, N, D, softmax_scale, causal, rows, o, lse};
    parallel_for(nrows, nthreads, exact_chunk, &a);
}
