/*
 * The CPU oracle for Q4_K / Q8_0 dequantize-and-multiply.
 *
 * TEST INFRASTRUCTURE ONLY: called by the tests, the smoke check and the
 * bench's CPU-baseline leg, never by the product path, and sharing no code
 * with it.  Built with -O2 -ffp-contract=off -fno-fast-math: every f32
 * operation below is a single IEEE-rounded operation, no fused multiply-add.
 * The only parallelism is OpenMP over independent output rows; each row's
 * accumulation order is fixed (k ascending), so results do not depend on the
 * thread count.
 *
 * What it computes follows the pages' CPU reference for the Metal kernels
 * ("Mac Qwen3.6-27B Metal Q4_K perf diagnosis", TL;DR: the GEMV is checked
 * against a CPU f32 reference; "Qwen3.6-27B on Apple M3 Pro", reconciliation
 * table: raw q4_k blocks with a scalar f32 GEMV): dequantize to f32, then dot.
 * Here the dot accumulates in f64.  See oracle.h for the byte layouts.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ f16 */

float orc_f16_decode(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    float v;
    if (e == 0)
        v = ldexpf((float)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexpf((float)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* Split a positive finite v into binary16 (exponent field, scaled significand)
 * for the chosen rounding of the significand.  mode 0: round up, 1: RNE. */
static uint16_t f16_from_positive(float v, int mode) {
    if (v == 0.0f) return 0;
    if (v < ldexpf(1.0f, -14)) {                   /* binary16 subnormal range */
        float s = ldexpf(v, 24);                   /* exact: power-of-two scaling */
        float m = mode == 0 ? ceilf(s) : rintf(s);
        return (uint16_t)m;                        /* m == 1024 is the smallest normal, 0x0400 */
    }
    int ex;
    frexpf(v, &ex);                                /* v in [2^(ex-1), 2^ex) */
    int E = ex - 1;
    float s = ldexpf(v, 10 - E);                   /* in [1024, 2048), exact */
    float m = mode == 0 ? ceilf(s) : rintf(s);
    int mant = (int)m - 1024;
    if (mant == 1024) { mant = 0; E += 1; }
    if (E > 15) return 0x7BFF;                     /* saturate at 65504 */
    return (uint16_t)(((E + 15) << 10) | mant);
}

uint16_t orc_f16_round_up(float v) {
    if (!(v > 0.0f)) return 0;
    if (v > 65504.0f) return 0x7BFF;
    return f16_from_positive(v, 0);
}

uint16_t orc_f16_rne(float v) {
    uint16_t sign = v < 0.0f ? 0x8000 : 0;
    float a = fabsf(v);
    if (a >= 65520.0f) return sign | 0x7BFF;       /* would round to inf: saturate */
    return sign | f16_from_positive(a, 1);
}

float orc_bf16_decode(uint16_t b) {
    union { uint32_t u; float f; } c;
    c.u = (uint32_t)b << 16;
    return c.f;
}

/* ----------------------------------------------------------------- Q4_K */

static int imin(int a, int b) { return a < b ? a : b; }
static int imax(int a, int b) { return a > b ? a : b; }

/* Covering min/max quantizer for one 256-weight super-block (the pinned
 * reading; the pages only name the format). */
void orc_q4k_quantize_superblock(const float* x, uint8_t* out) {
    float lo[8], hi[8], mn[8], r[8];
    int sc[8], m[8];
    float max_mn = 0.0f, max_r = 0.0f;
    for (int j = 0; j < 8; j++) {
        float l = 0.0f, h = x[32 * j];
        for (int i = 0; i < 32; i++) {
            float v = x[32 * j + i];
            if (v < l) l = v;
            if (v > h) h = v;
        }
        lo[j] = l;
        hi[j] = h;
        mn[j] = -l;
        if (mn[j] > max_mn) max_mn = mn[j];
    }
    uint16_t dmin_h = orc_f16_round_up(max_mn / 63.0f);
    float dmin = orc_f16_decode(dmin_h);
    for (int j = 0; j < 8; j++) {
        m[j] = dmin > 0.0f ? imin(63, (int)ceilf(mn[j] / dmin)) : 0;
        r[j] = hi[j] + dmin * (float)m[j];
        if (r[j] > max_r) max_r = r[j];
    }
    uint16_t d_h = orc_f16_round_up(max_r / (15.0f * 63.0f));
    float d = orc_f16_decode(d_h);
    for (int j = 0; j < 8; j++)
        sc[j] = d > 0.0f ? imax(0, imin(63, (int)ceilf(r[j] / (15.0f * d)))) : 0;

    uint8_t q[256];
    for (int j = 0; j < 8; j++) {
        float off = dmin * (float)m[j];
        float step = d * (float)sc[j];
        for (int i = 0; i < 32; i++) {
            int qi = 0;
            if (sc[j] > 0) qi = imax(0, imin(15, (int)rintf((x[32 * j + i] + off) / step)));
            q[32 * j + i] = (uint8_t)qi;
        }
    }
    (void)lo;

    out[0] = (uint8_t)(d_h & 0xFF);
    out[1] = (uint8_t)(d_h >> 8);
    out[2] = (uint8_t)(dmin_h & 0xFF);
    out[3] = (uint8_t)(dmin_h >> 8);
    uint8_t* s = out + 4;
    for (int j = 0; j < 4; j++) {
        s[j] = (uint8_t)(sc[j] | ((sc[j + 4] >> 4) << 6));
        s[j + 4] = (uint8_t)(m[j] | ((m[j + 4] >> 4) << 6));
        s[j + 8] = (uint8_t)((sc[j + 4] & 15) | ((m[j + 4] & 15) << 4));
    }
    uint8_t* qs = out + 16;
    for (int g = 0; g < 4; g++)
        for (int l = 0; l < 32; l++)
            qs[32 * g + l] = (uint8_t)(q[64 * g + l] | (q[64 * g + 32 + l] << 4));
}

int orc_q4k_pack(const float* w, int64_t N, int64_t K, uint8_t* out) {
    if (N < 0 || K < 0 || K % 256 != 0) return -1;
    int64_t nb = K / 256;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++)
            orc_q4k_quantize_superblock(w + n * K + 256 * b, out + (n * nb + b) * 144);
    return 0;
}

void orc_q4k_fields(const uint8_t* blk, uint16_t* d, uint16_t* dmin, uint8_t sc[8], uint8_t m[8],
                    uint8_t q[256]) {
    *d = (uint16_t)(blk[0] | (blk[1] << 8));
    *dmin = (uint16_t)(blk[2] | (blk[3] << 8));
    const uint8_t* s = blk + 4;
    for (int j = 0; j < 4; j++) {
        sc[j] = s[j] & 63;
        m[j] = s[j + 4] & 63;
        sc[j + 4] = (uint8_t)((s[j + 8] & 15) | ((s[j] >> 6) << 4));
        m[j + 4] = (uint8_t)((s[j + 8] >> 4) | ((s[j + 4] >> 6) << 4));
    }
    const uint8_t* qs = blk + 16;
    for (int g = 0; g < 4; g++)
        for (int l = 0; l < 32; l++) {
            q[64 * g + l] = qs[32 * g + l] & 15;
            q[64 * g + 32 + l] = qs[32 * g + l] >> 4;
        }
}

void orc_q4k_dequant_block(const uint8_t* blk, float* out) {
    uint16_t dh, mh;
    uint8_t sc[8], m[8], q[256];
    orc_q4k_fields(blk, &dh, &mh, sc, m, q);
    float d = orc_f16_decode(dh), dmin = orc_f16_decode(mh);
    for (int j = 0; j < 8; j++) {
        float ds = d * (float)sc[j];
        float dm = dmin * (float)m[j];
        for (int i = 0; i < 32; i++) out[32 * j + i] = ds * (float)q[32 * j + i] - dm;
    }
}

void orc_q4k_dequant_rows(const uint8_t* W, int64_t N, int64_t K, float* out) {
    int64_t nb = K / 256;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++)
            orc_q4k_dequant_block(W + (n * nb + b) * 144, out + n * K + 256 * b);
}

/* ----------------------------------------------------------------- Q8_0 */

void orc_q8_0_quantize_block(const float* x, uint8_t* out) {
    float amax = 0.0f;
    for (int i = 0; i < 32; i++) {
        float a = fabsf(x[i]);
        if (a > amax) amax = a;
    }
    uint16_t dh = orc_f16_rne(amax / 127.0f);
    float d = orc_f16_decode(dh);
    out[0] = (uint8_t)(dh & 0xFF);
    out[1] = (uint8_t)(dh >> 8);
    for (int i = 0; i < 32; i++) {
        int q = 0;
        if (d > 0.0f) q = imax(-127, imin(127, (int)rintf(x[i] / d)));
        out[2 + i] = (uint8_t)(int8_t)q;
    }
}

int orc_q8_0_pack(const float* w, int64_t N, int64_t K, uint8_t* out) {
    if (N < 0 || K < 0 || K % 32 != 0) return -1;
    int64_t nb = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; n++)
        for (int64_t b = 0; b < nb; b++)
            orc_q8_0_quantize_block(w + n * K + 32 * b, out + (n * nb + b) * 34);
    return 0;
}

void orc_q8_0_dequant_block(const uint8_t* blk, float* out) {
    float d = orc_f16_decode((uint16_t)(blk[0] | (blk[1] << 8)));
    for (int i = 0; i < 32; i++) out[i] = d * (float)(int8_t)blk[2 + i];
}

/* -------------------------------------------------------------- matvec */

static void row_dot(const float* w, const float* x, int64_t K, double* y, double* a) {
    double s = 0.0, sa = 0.0;
    for (int64_t k = 0; k < K; k++) {
        double p = (double)w[k] * (double)x[k];
        s += p;
        sa += fabs(p);
    }
    *y = s;
    if (a) *a = sa;
}

void orc_gemv_q4k(const uint8_t* W, int64_t N, int64_t K, const float* x, double* y, double* a) {
    int64_t nb = K / 256;
#pragma omp parallel
    {
        float* row = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; n++) {
            for (int64_t b = 0; b < nb; b++) orc_q4k_dequant_block(W + (n * nb + b) * 144, row + 256 * b);
            row_dot(row, x, K, y + n, a ? a + n : NULL);
        }
        free(row);
    }
}

void orc_gemv_q8_0(const uint8_t* W, int64_t N, int64_t K, const float* x, double* y, double* a) {
    int64_t nb = K / 32;
#pragma omp parallel
    {
        float* row = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; n++) {
            for (int64_t b = 0; b < nb; b++) orc_q8_0_dequant_block(W + (n * nb + b) * 34, row + 32 * b);
            row_dot(row, x, K, y + n, a ? a + n : NULL);
        }
        free(row);
    }
}

void orc_gemv_batch_q4k(const uint8_t* W, int64_t N, int64_t K, const float* X, int64_t M,
                        double* Y, double* A) {
    for (int64_t mi = 0; mi < M; mi++)
        orc_gemv_q4k(W, N, K, X + mi * K, Y + mi * N, A ? A + mi * N : NULL);
}

void orc_gemm_q4k(const uint8_t* W, int64_t N, int64_t K, const uint16_t* X, int64_t P,
                  double* Y, double* A) {
    float* xf = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
    for (int64_t p = 0; p < P; p++) {
        for (int64_t k = 0; k < K; k++) xf[k] = orc_bf16_decode(X[p * K + k]);
        orc_gemv_q4k(W, N, K, xf, Y + p * N, A ? A + p * N : NULL);
    }
    free(xf);
}

void orc_gemm_q4k_sample(const uint8_t* W, int64_t N, int64_t K, const uint16_t* X, int64_t P,
                         const int64_t* rows, int64_t n_rows, const int64_t* toks, int64_t n_toks,
                         double* Y, double* A) {
    int64_t nb = K / 256;
    (void)N; (void)P;
#pragma omp parallel
    {
        float* row = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
        float* xf = (float*)malloc(sizeof(float) * (size_t)(K > 0 ? K : 1));
#pragma omp for schedule(static)
        for (int64_t j = 0; j < n_rows; j++) {
            for (int64_t b = 0; b < nb; b++)
                orc_q4k_dequant_block(W + (rows[j] * nb + b) * 144, row + 256 * b);
            for (int64_t i = 0; i < n_toks; i++) {
                for (int64_t k = 0; k < K; k++) xf[k] = orc_bf16_decode(X[toks[i] * K + k]);
                row_dot(row, xf, K, Y + i * n_rows + j, A ? A + i * n_rows + j : NULL);
            }
        }
        free(row);
        free(xf);
    }
}

void orc_rmsnorm(const double* x, int64_t n, double eps, double* out) {
    double ss = 0.0;
    for (int64_t i = 0; i < n; i++) ss += x[i] * x[i];
    double r = 1.0 / sqrt(ss / (double)n + eps);
    for (int64_t i = 0; i < n; i++) out[i] = x[i] * r;
}

void orc_swiglu(const double* g, const double* u, int64_t n, double* out) {
    for (int64_t i = 0; i < n; i++) out[i] = g[i] / (1.0 + exp(-g[i])) * u[i];
}

int64_t orc_argmax_f32(const float* v, int64_t n) {
    int64_t best = -1;
    for (int64_t i = 0; i < n; i++) {
        if (v[i] != v[i]) continue;
        if (best < 0 || v[i] > v[best]) best = i;
    }
    return best;
}

/* ------------------------------------------------------ int8 activations */

void orc_quantize_act_i8(const float* x, int64_t n, int8_t* X, float* d) {
    for (int64_t j = 0; j < n / 32; j++) {
        const float* xs = x + 32 * j;
        float am = 0.0f;
        for (int i = 0; i < 32; i++) {
            float v = fabsf(xs[i]);
            if (v > am) am = v;
        }
        if (!(am > 0.0f)) {
            d[j] = 0.0f;
            for (int i = 0; i < 32; i++) X[32 * j + i] = 0;
            continue;
        }
        float inv = 127.0f / am;
        d[j] = am / 127.0f;
        for (int i = 0; i < 32; i++) {
            float s = xs[i] * inv;
            X[32 * j + i] = (int8_t)imax(-127, imin(127, (int)rintf(s)));
        }
    }
}

void orc_gemv_q4k_act_i8(const uint8_t* W, int64_t N, int64_t K, const float* x, double* y, double* a) {
    int8_t* X = (int8_t*)malloc((size_t)K);
    float* d = (float*)malloc(sizeof(float) * (size_t)(K / 32));
    double* xq = (double*)malloc(sizeof(double) * (size_t)K);
    orc_quantize_act_i8(x, K, X, d);
    for (int64_t k = 0; k < K; k++) xq[k] = (double)d[k / 32] * (double)X[k];
    int64_t nb = K / 256;
#pragma omp parallel
    {
        float* row = (float*)malloc(sizeof(float) * K);
#pragma omp for schedule(static)
        for (int64_t n = 0; n < N; n++) {
            for (int64_t b = 0; b < nb; b++) orc_q4k_dequant_block(W + (n * nb + b) * 144, row + 256 * b);
            double s = 0.0, sa = 0.0;
            for (int64_t k = 0; k < K; k++) {
                double p = (double)row[k] * xq[k];
                s += p;
                sa += fabs(p);
            }
            y[n] = s;
            if (a) a[n] = sa;
        }
        free(row);
    }
    free(X);
    free(d);
    free(xq);
}

/* ------------------------------------------------------------- decode */

static void to_f32(const double* a, int64_t n, float* out) {
    for (int64_t i = 0; i < n; i++) out[i] = (float)a[i];
}

int64_t orc_decode_token(const orc_model* m, int64_t tok, double* h_out, float* logits,
                         double* logit_abs, float* kv_out) {
    const int64_t D = m->d_model, F = m->d_ff;
    int64_t tmax = m->gdn_in > m->fa_qg ? m->gdn_in : m->fa_qg;
    if (F > tmax) tmax = F;
    if (m->vocab > tmax) tmax = m->vocab;
    double* h = (double*)malloc(sizeof(double) * D);
    double* n = (double*)malloc(sizeof(double) * D);
    double* o = (double*)malloc(sizeof(double) * D);
    double* t = (double*)malloc(sizeof(double) * tmax);
    double* u = (double*)malloc(sizeof(double) * F);
    double* a = (double*)malloc(sizeof(double) * tmax);
    float* xf = (float*)malloc(sizeof(float) * tmax);
    int64_t fa_index = 0;

    for (int64_t i = 0; i < D; i++) h[i] = (double)m->embedding[tok * D + i];
    for (int64_t l = 0; l < m->n_layers; l++) {
        const orc_layer* L = &m->layers[l];
        /* mixer: projections around a body that is out of scope */
        orc_rmsnorm(h, D, m->eps, n);
        to_f32(n, D, xf);
        if (L->kind == ORC_LAYER_GDN) {
            orc_gemv_q4k(L->w_in, m->gdn_in, D, xf, t, NULL);
        } else {
            orc_gemv_q4k(L->w_in, m->fa_qg, D, xf, t, NULL);
            orc_gemv_q4k(L->w_k, m->fa_kv, D, xf, a, NULL);
            if (kv_out) to_f32(a, m->fa_kv, kv_out + (2 * fa_index) * m->fa_kv);
            orc_gemv_q4k(L->w_v, m->fa_kv, D, xf, a, NULL);
            if (kv_out) to_f32(a, m->fa_kv, kv_out + (2 * fa_index + 1) * m->fa_kv);
            fa_index++;
        }
        to_f32(t, m->n_mix, xf);                  /* out_proj / o input: t[0:n_mix] */
        orc_gemv_q4k(L->w_out, D, m->n_mix, xf, o, NULL);
        for (int64_t i = 0; i < D; i++) h[i] += o[i];
        /* MLP */
        orc_rmsnorm(h, D, m->eps, n);
        to_f32(n, D, xf);
        orc_gemv_q4k(L->w_gate, F, D, xf, t, NULL);
        orc_gemv_q4k(L->w_up, F, D, xf, u, NULL);
        orc_swiglu(t, u, F, a);
        to_f32(a, F, xf);
        orc_gemv_q4k(L->w_down, D, F, xf, o, NULL);
        for (int64_t i = 0; i < D; i++) h[i] += o[i];
    }
    if (h_out) memcpy(h_out, h, sizeof(double) * D);
    orc_rmsnorm(h, D, m->eps, n);
    to_f32(n, D, xf);
    orc_gemv_q8_0(m->lm_head, m->vocab, D, xf, t, logit_abs);
    float* lf = logits ? logits : (float*)malloc(sizeof(float) * m->vocab);
    to_f32(t, m->vocab, lf);
    int64_t best = orc_argmax_f32(lf, m->vocab);
    if (!logits) free(lf);
    free(h); free(n); free(o); free(t); free(u); free(a); free(xf);
    return best;
}

int64_t orc_decode_weight_bytes(const orc_model* m) {
    const int64_t D = m->d_model, F = m->d_ff;
    int64_t q4 = 0;   /* Q4_K weights, counted as 144 bytes per 256 */
    for (int64_t l = 0; l < m->n_layers; l++) {
        if (m->layers[l].kind == ORC_LAYER_GDN)
            q4 += m->gdn_in * D + D * m->n_mix;
        else
            q4 += m->fa_qg * D + 2 * m->fa_kv * D + D * m->n_mix;
        q4 += 2 * F * D + D * F;
    }
    return q4 / 256 * 144 + m->vocab * D / 32 * 34;
}
