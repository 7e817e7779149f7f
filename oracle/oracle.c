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

/* ------------------------------------------------------- mixer bodies */

static double silu(double x) { return x / (1.0 + exp(-x)); }
static double sigmoid(double x) { return 1.0 / (1.0 + exp(-x)); }
static double softplus(double x) { return x > 20.0 ? x : log1p(exp(x)); }

void orc_causal_conv_step(const float* w, double* state, const double* x, int64_t n, int64_t K, double* y) {
    for (int64_t c = 0; c < n; c++) {
        double* s = state + c * (K - 1);
        const float* wc = w + c * K;
        double acc = 0.0;
        for (int64_t j = 0; j < K - 1; j++) acc += (double)wc[j] * s[j];
        acc += (double)wc[K - 1] * x[c];
        y[c] = acc;
        for (int64_t j = 0; j + 1 < K - 1; j++) s[j] = s[j + 1];
        s[K - 2] = x[c];
    }
}

void orc_gdn_step(const orc_mixer_dims* d, const orc_mixer_params* p, const double* t, double* conv_state,
                  double* S, double* out, double* o_raw) {
    const int64_t nk = d->nk, nv = d->nv, dk = d->dk, dv = d->dv, K = d->conv;
    const int64_t conv_dim = 2 * nk * dk + nv * dv;
    double* y = (double*)malloc(sizeof(double) * conv_dim);
    /* short causal conv over q|k|v, then silu */
    orc_causal_conv_step(p->conv_w, conv_state, t, conv_dim, K, y);
    for (int64_t c = 0; c < conv_dim; c++) y[c] = silu(y[c]);
    double* q = y;
    double* k = y + nk * dk;
    const double* v = y + 2 * nk * dk;
    const double* z = t + conv_dim;
    const double* b = z + nv * dv;
    const double* a = b + nv;
    /* per key head: L2 normalization; queries also scaled by 1/sqrt(dk) */
    for (int64_t h = 0; h < nk; h++) {
        double sq = 0.0, sk = 0.0;
        for (int64_t i = 0; i < dk; i++) {
            sq += q[h * dk + i] * q[h * dk + i];
            sk += k[h * dk + i] * k[h * dk + i];
        }
        double rq = 1.0 / sqrt(sq + d->eps) / sqrt((double)dk), rk = 1.0 / sqrt(sk + d->eps);
        for (int64_t i = 0; i < dk; i++) {
            q[h * dk + i] *= rq;
            k[h * dk + i] *= rk;
        }
    }
    double* o = (double*)malloc(sizeof(double) * dv);
    double* delta = (double*)malloc(sizeof(double) * dv);
    for (int64_t h = 0; h < nv; h++) {
        const int64_t kh = h / (nv / nk);
        const double* qh = q + kh * dk;
        const double* khv = k + kh * dk;
        const double* vh = v + h * dv;
        double* Sh = S + h * dk * dv;                /* Sh[i][j], i over dk, j over dv */
        const double beta = sigmoid(b[h]);
        const double g = -exp((double)p->a_log[h]) * softplus(a[h] + (double)p->dt_bias[h]);
        const double alpha = exp(g);
        for (int64_t i = 0; i < dk * dv; i++) Sh[i] *= alpha;
        for (int64_t j = 0; j < dv; j++) {           /* delta = beta (v - S^T k) */
            double kv = 0.0;
            for (int64_t i = 0; i < dk; i++) kv += Sh[i * dv + j] * khv[i];
            delta[j] = beta * (vh[j] - kv);
        }
        for (int64_t i = 0; i < dk; i++)             /* S += k delta^T */
            for (int64_t j = 0; j < dv; j++) Sh[i * dv + j] += khv[i] * delta[j];
        for (int64_t j = 0; j < dv; j++) {           /* o = S^T q */
            double acc = 0.0;
            for (int64_t i = 0; i < dk; i++) acc += Sh[i * dv + j] * qh[i];
            o[j] = acc;
        }
        if (o_raw) memcpy(o_raw + h * dv, o, sizeof(double) * dv);
        double ss = 0.0;                             /* gated RMSNorm with the swish gate z */
        for (int64_t j = 0; j < dv; j++) ss += o[j] * o[j];
        const double r = 1.0 / sqrt(ss / (double)dv + d->eps);
        for (int64_t j = 0; j < dv; j++)
            out[h * dv + j] = o[j] * r * (double)p->norm_w[j] * silu(z[h * dv + j]);
    }
    free(o);
    free(delta);
    free(y);
}

static void head_rmsnorm(const double* x, int64_t n, double eps, const float* gain, double* out) {
    double ss = 0.0;
    for (int64_t i = 0; i < n; i++) ss += x[i] * x[i];
    const double r = 1.0 / sqrt(ss / (double)n + eps);
    for (int64_t i = 0; i < n; i++) out[i] = x[i] * r * (double)gain[i];
}

static void rope(double* x, int64_t rot, int64_t pos, double theta) {
    const int64_t half = rot / 2;
    for (int64_t i = 0; i < half; i++) {
        const double ang = (double)pos * pow(theta, -2.0 * (double)i / (double)rot);
        const double c = cos(ang), s = sin(ang);
        const double x1 = x[i], x2 = x[i + half];
        x[i] = x1 * c - x2 * s;
        x[i + half] = x2 * c + x1 * s;
    }
}

void orc_attn_step(const orc_mixer_dims* d, const orc_mixer_params* p, const double* qg, const double* k,
                   const double* v, int64_t pos, int64_t max_ctx, double* kc, double* vc, double* out) {
    const int64_t nq = d->nq, nkv = d->nkv, dh = d->dh;
    for (int64_t g = 0; g < nkv; g++) {              /* this position's keys and values into the cache */
        double* kp = kc + (g * max_ctx + pos) * dh;
        head_rmsnorm(k + g * dh, dh, d->eps, p->k_norm_w, kp);
        rope(kp, d->rot, pos, d->theta);
        memcpy(vc + (g * max_ctx + pos) * dh, v + g * dh, sizeof(double) * dh);
    }
    double* q = (double*)malloc(sizeof(double) * dh);
    double* w = (double*)malloc(sizeof(double) * (pos + 1));
    for (int64_t h = 0; h < nq; h++) {
        const int64_t g = h / (nq / nkv);
        head_rmsnorm(qg + h * 2 * dh, dh, d->eps, p->q_norm_w, q);
        rope(q, d->rot, pos, d->theta);
        double mx = -INFINITY;
        for (int64_t s = 0; s <= pos; s++) {
            const double* kp = kc + (g * max_ctx + s) * dh;
            double acc = 0.0;
            for (int64_t i = 0; i < dh; i++) acc += q[i] * kp[i];
            w[s] = acc / sqrt((double)dh);
            if (w[s] > mx) mx = w[s];
        }
        double sum = 0.0;
        for (int64_t s = 0; s <= pos; s++) {
            w[s] = exp(w[s] - mx);
            sum += w[s];
        }
        const double* gate = qg + h * 2 * dh + dh;
        for (int64_t i = 0; i < dh; i++) {
            double acc = 0.0;
            for (int64_t s = 0; s <= pos; s++) acc += w[s] * vc[(g * max_ctx + s) * dh + i];
            out[h * dh + i] = acc / sum * sigmoid(gate[i]);
        }
    }
    free(q);
    free(w);
}

struct orc_mixer_state {
    int64_t n_layers, max_ctx, pos;
    double** conv;   /* per layer (GDN) or NULL */
    double** S;
    double** kc;     /* per layer (FA) or NULL */
    double** vc;
};

orc_mixer_state* orc_mixer_state_create(const orc_model* m, const orc_mixer_dims* d, int64_t max_ctx) {
    orc_mixer_state* st = (orc_mixer_state*)calloc(1, sizeof(orc_mixer_state));
    const int64_t L = m->n_layers, conv_dim = 2 * d->nk * d->dk + d->nv * d->dv;
    st->n_layers = L;
    st->max_ctx = max_ctx;
    st->conv = (double**)calloc(L, sizeof(double*));
    st->S = (double**)calloc(L, sizeof(double*));
    st->kc = (double**)calloc(L, sizeof(double*));
    st->vc = (double**)calloc(L, sizeof(double*));
    for (int64_t l = 0; l < L; l++) {
        if (m->layers[l].kind == ORC_LAYER_GDN) {
            st->conv[l] = (double*)calloc(conv_dim * (d->conv - 1), sizeof(double));
            st->S[l] = (double*)calloc(d->nv * d->dk * d->dv, sizeof(double));
        } else {
            st->kc[l] = (double*)calloc(d->nkv * max_ctx * d->dh, sizeof(double));
            st->vc[l] = (double*)calloc(d->nkv * max_ctx * d->dh, sizeof(double));
        }
    }
    return st;
}

void orc_mixer_state_destroy(orc_mixer_state* st) {
    if (!st) return;
    for (int64_t l = 0; l < st->n_layers; l++) {
        free(st->conv[l]);
        free(st->S[l]);
        free(st->kc[l]);
        free(st->vc[l]);
    }
    free(st->conv);
    free(st->S);
    free(st->kc);
    free(st->vc);
    free(st);
}

int64_t orc_decode_token_mixer(const orc_model* m, const orc_mixer_dims* d, const orc_mixer_params* mp,
                               orc_mixer_state* st, int64_t tok, double* h_out, float* logits,
                               double* logit_abs) {
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
    double* kk = (double*)malloc(sizeof(double) * m->fa_kv);
    double* vv = (double*)malloc(sizeof(double) * m->fa_kv);
    double* mix = (double*)malloc(sizeof(double) * m->n_mix);
    float* xf = (float*)malloc(sizeof(float) * tmax);

    for (int64_t i = 0; i < D; i++) h[i] = (double)m->embedding[tok * D + i];
    for (int64_t l = 0; l < m->n_layers; l++) {
        const orc_layer* L = &m->layers[l];
        orc_rmsnorm(h, D, m->eps, n);
        to_f32(n, D, xf);
        if (L->kind == ORC_LAYER_GDN) {
            orc_gemv_q4k(L->w_in, m->gdn_in, D, xf, t, NULL);
            orc_gdn_step(d, &mp[l], t, st->conv[l], st->S[l], mix, NULL);
        } else {
            orc_gemv_q4k(L->w_in, m->fa_qg, D, xf, t, NULL);
            orc_gemv_q4k(L->w_k, m->fa_kv, D, xf, kk, NULL);
            orc_gemv_q4k(L->w_v, m->fa_kv, D, xf, vv, NULL);
            orc_attn_step(d, &mp[l], t, kk, vv, st->pos, st->max_ctx, st->kc[l], st->vc[l], mix);
        }
        to_f32(mix, m->n_mix, xf);                /* out_proj / o input: the mixer's output */
        orc_gemv_q4k(L->w_out, D, m->n_mix, xf, o, NULL);
        for (int64_t i = 0; i < D; i++) h[i] += o[i];
        orc_rmsnorm(h, D, m->eps, n);
        to_f32(n, D, xf);
        orc_gemv_q4k(L->w_gate, F, D, xf, t, NULL);
        orc_gemv_q4k(L->w_up, F, D, xf, u, NULL);
        orc_swiglu(t, u, F, a);
        to_f32(a, F, xf);
        orc_gemv_q4k(L->w_down, D, F, xf, o, NULL);
        for (int64_t i = 0; i < D; i++) h[i] += o[i];
    }
    st->pos++;
    if (h_out) memcpy(h_out, h, sizeof(double) * D);
    orc_rmsnorm(h, D, m->eps, n);
    to_f32(n, D, xf);
    orc_gemv_q8_0(m->lm_head, m->vocab, D, xf, t, logit_abs);
    float* lf = logits ? logits : (float*)malloc(sizeof(float) * m->vocab);
    to_f32(t, m->vocab, lf);
    int64_t best = orc_argmax_f32(lf, m->vocab);
    if (!logits) free(lf);
    free(h); free(n); free(o); free(t); free(u); free(a); free(kk); free(vv); free(mix); free(xf);
    return best;
}

/* ------------------------------------------------------- prefill forward */

uint16_t orc_bf16_rne(float v) {
    union { float f; uint32_t u; } c;
    c.f = v;
    if ((c.u & 0x7F800000u) == 0x7F800000u && (c.u & 0x7FFFFFu)) return (uint16_t)((c.u >> 16) | 0x40);
    const uint32_t lsb = (c.u >> 16) & 1u;
    return (uint16_t)((c.u + 0x7FFFu + lsb) >> 16);
}

static void rows_to_bf16(const double* a, int64_t rows, int64_t n, int64_t stride, uint16_t* out) {
    for (int64_t r = 0; r < rows; r++)
        for (int64_t i = 0; i < n; i++) out[r * n + i] = orc_bf16_rne((float)a[r * stride + i]);
}

int64_t orc_prefill_forward(const orc_model* m, const int64_t* toks, int64_t P, double* h_out, float* logits,
                            double* logit_abs) {
    const int64_t D = m->d_model, F = m->d_ff;
    const int64_t tn = m->gdn_in > m->fa_qg ? m->gdn_in : m->fa_qg;
    double* h = (double*)malloc(sizeof(double) * P * D);
    double* n = (double*)malloc(sizeof(double) * P * D);
    double* t = (double*)malloc(sizeof(double) * P * tn);
    double* o = (double*)malloc(sizeof(double) * P * D);
    double* g = (double*)malloc(sizeof(double) * P * F);
    double* u = (double*)malloc(sizeof(double) * P * F);
    uint16_t* xb = (uint16_t*)malloc(sizeof(uint16_t) * P * (F > tn ? F : tn));
    for (int64_t p = 0; p < P; p++)
        for (int64_t i = 0; i < D; i++) h[p * D + i] = (double)m->embedding[toks[p] * D + i];
    for (int64_t l = 0; l < m->n_layers; l++) {
        const orc_layer* L = &m->layers[l];
        const int64_t nin = L->kind == ORC_LAYER_GDN ? m->gdn_in : m->fa_qg;
        for (int64_t p = 0; p < P; p++) orc_rmsnorm(h + p * D, D, m->eps, n + p * D);
        rows_to_bf16(n, P, D, D, xb);
        orc_gemm_q4k(L->w_in, nin, D, xb, P, t, NULL);
        rows_to_bf16(t, P, m->n_mix, nin, xb);        /* out_proj / o input: t[:, 0:n_mix] */
        orc_gemm_q4k(L->w_out, D, m->n_mix, xb, P, o, NULL);
        for (int64_t i = 0; i < P * D; i++) h[i] += o[i];
        for (int64_t p = 0; p < P; p++) orc_rmsnorm(h + p * D, D, m->eps, n + p * D);
        rows_to_bf16(n, P, D, D, xb);
        orc_gemm_q4k(L->w_gate, F, D, xb, P, g, NULL);
        orc_gemm_q4k(L->w_up, F, D, xb, P, u, NULL);
        orc_swiglu(g, u, P * F, g);
        rows_to_bf16(g, P, F, F, xb);
        orc_gemm_q4k(L->w_down, D, F, xb, P, o, NULL);
        for (int64_t i = 0; i < P * D; i++) h[i] += o[i];
    }
    if (h_out) memcpy(h_out, h, sizeof(double) * P * D);
    float* xf = (float*)malloc(sizeof(float) * D);
    orc_rmsnorm(h + (P - 1) * D, D, m->eps, n);
    to_f32(n, D, xf);
    double* y = (double*)malloc(sizeof(double) * m->vocab);
    orc_gemv_q8_0(m->lm_head, m->vocab, D, xf, y, logit_abs);
    float* lf = logits ? logits : (float*)malloc(sizeof(float) * m->vocab);
    to_f32(y, m->vocab, lf);
    int64_t best = orc_argmax_f32(lf, m->vocab);
    if (!logits) free(lf);
    free(h); free(n); free(t); free(o); free(g); free(u); free(xb); free(xf); free(y);
    return best;
}
