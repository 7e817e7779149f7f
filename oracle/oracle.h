/*
 * Q4_K / Q8_0 weight-only dequantize-and-multiply: the CPU ORACLE.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg call this code.  The product path never links it and
 * shares no code with it.
 *
 * Everything here is the plain definition, written for a reader to check by
 * eye against the pages this project follows ("Mac Qwen3.6-27B Metal Q4_K perf
 * diagnosis", TL;DR and section 4b; "Qwen3.6-27B on Apple M3 Pro -- the llama.cpp
 * parity bar", model architecture and the reconciliation table):
 *   dequantize every weight to f32, then accumulate the dot product in f64,
 *   in index order.  No blocking, fusion or reordering.
 *
 * Q4_K byte layout (block_q4_K, 144 bytes per 256 weights, little-endian):
 *   [0,2)   d     binary16        [2,4)   dmin  binary16
 *   [4,16)  s[12] packed 6-bit scales sc_0..7 and mins m_0..7:
 *             j<4 : sc_j = s[j] & 63,                 m_j = s[j+4] & 63
 *             j>=4: sc_j = (s[j+4] & 15) | (s[j-4] >> 6) << 4
 *                   m_j  = (s[j+4] >> 4) | (s[j]   >> 6) << 4
 *   [16,144) qs[128]: qs[32g+l] low nibble = q of weight 64g+l,
 *                      high nibble = q of weight 64g+32+l       (g<4, l<32)
 *   weight i (sub-block j = i/32):  w = d*sc_j*q_i - dmin*m_j
 * Q8_0 (block_q8_0, 34 bytes per 32 weights): binary16 d, then 32 int8 q; w = d*q.
 *
 * The quantizers (covering min/max for Q4_K, absmax for Q8_0) are the pinned
 * readings listed in the design notes; the pages name the format only.
 */
#ifndef FAK_ORACLE_H
#define FAK_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* binary16 helpers, written from IEEE 754-2008 (no library conversion). */
float    orc_f16_decode(uint16_t h);
uint16_t orc_f16_round_up(float v);   /* smallest binary16 >= v, for v >= 0; saturates at 65504 */
uint16_t orc_f16_rne(float v);        /* round to nearest, ties to even; saturates at +-65504 */
float    orc_bf16_decode(uint16_t b);

/* Q4_K */
void orc_q4k_quantize_superblock(const float* x256, uint8_t* out144);
int  orc_q4k_pack(const float* w, int64_t N, int64_t K, uint8_t* out);   /* out: N*(K/256)*144 bytes */
void orc_q4k_fields(const uint8_t* blk, uint16_t* d, uint16_t* dmin, uint8_t sc[8], uint8_t m[8],
                    uint8_t q[256]);
void orc_q4k_dequant_block(const uint8_t* blk, float* out256);
void orc_q4k_dequant_rows(const uint8_t* W, int64_t N, int64_t K, float* out);

/* Q8_0 */
void orc_q8_0_quantize_block(const float* x32, uint8_t* out34);
int  orc_q8_0_pack(const float* w, int64_t N, int64_t K, uint8_t* out);  /* out: N*(K/32)*34 bytes */
void orc_q8_0_dequant_block(const uint8_t* blk, float* out32);

/* y[n] = sum_k What[n,k]*x[k] in f64 (k ascending); a[n] = sum_k |What[n,k]*x[k]| (may be NULL). */
void orc_gemv_q4k(const uint8_t* W, int64_t N, int64_t K, const float* x, double* y, double* a);
void orc_gemv_q8_0(const uint8_t* W, int64_t N, int64_t K, const float* x, double* y, double* a);
/* M independent GEMVs: Y[m,n], A[m,n] for X[m,:]. */
void orc_gemv_batch_q4k(const uint8_t* W, int64_t N, int64_t K, const float* X, int64_t M,
                        double* Y, double* A);
/* Y[p,n] = sum_k What[n,k]*bf16(X[p,k]) in f64; X holds bfloat16 bit patterns. */
void orc_gemm_q4k(const uint8_t* W, int64_t N, int64_t K, const uint16_t* X, int64_t P,
                  double* Y, double* A);

/* Y[i,j] = sum_k What[rows[j],k]*bf16(X[toks[i],k]) in f64 for sampled rows and tokens. */
void orc_gemm_q4k_sample(const uint8_t* W, int64_t N, int64_t K, const uint16_t* X, int64_t P,
                         const int64_t* rows, int64_t n_rows, const int64_t* toks, int64_t n_toks,
                         double* Y, double* A);

/* out = x / sqrt(mean(x^2) + eps), f64. */
void orc_rmsnorm(const double* x, int64_t n, double eps, double* out);
/* out = g / (1 + exp(-g)) * u, f64. */
void orc_swiglu(const double* g, const double* u, int64_t n, double* out);
/* index of the largest value; the lowest index wins ties; NaNs are skipped. */
int64_t orc_argmax_f32(const float* v, int64_t n);

/* int8 activations of the int8-SDOT decode GEMV ("Qwen3.6-27B on Apple M3 Pro",
 * reconciliation table; the pages give no granularity or rounding, so this is
 * the reading taken): per 32-element sub-block j of x (n % 32 == 0),
 *   am_j = max |x_i|,  d_j = am_j / 127,  X_i = clamp(rint(x_i * (127 / am_j)), -127, 127)
 * in f32 (each division and the product one IEEE-rounded operation, rint ties to
 * even); d_j = 0 and X = 0 for an all-zero sub-block.  X[n], d[n/32]. */
void orc_quantize_act_i8(const float* x, int64_t n, int8_t* X, float* d);
/* y[n] = sum_k What[n,k] * (d_j * X_k) in f64 with (X, d) = orc_quantize_act_i8(x):
 * the GEMV of the int8 activations; a[n] = sum_k |What[n,k] * d_j * X_k|. */
void orc_gemv_q4k_act_i8(const uint8_t* W, int64_t N, int64_t K, const float* x, double* y, double* a);

/* ---- one decode token of the hybrid stack ---- */
enum { ORC_LAYER_GDN = 0, ORC_LAYER_FA = 1 };
typedef struct {
    int32_t kind;
    const uint8_t* w_in;    /* GDN in_proj / FA q+gate, [n_in x d_model] Q4_K */
    const uint8_t* w_k;     /* FA only, [n_kv x d_model] */
    const uint8_t* w_v;     /* FA only */
    const uint8_t* w_out;   /* GDN out_proj / FA o, [d_model x n_mix] */
    const uint8_t* w_gate;  /* [d_ff x d_model] */
    const uint8_t* w_up;
    const uint8_t* w_down;  /* [d_model x d_ff] */
} orc_layer;
typedef struct {
    int64_t n_layers, d_model, d_ff, vocab;
    int64_t gdn_in, fa_qg, fa_kv, n_mix;   /* in_proj rows, q+gate rows, k/v rows, mixer-out input width */
    double eps;
    const orc_layer* layers;
    const uint8_t* lm_head;   /* [vocab x d_model] Q8_0 */
    const float* embedding;   /* [vocab x d_model] f32 */
} orc_model;
/*
 * h = E[tok]; per layer: n = rms(h); mixer projections; h += out(t[0:n_mix]);
 * n = rms(h); h += down(swiglu(gate(n), up(n))).  Then logits = lm_head(rms(h)).
 * h stays f64 between ops; each matmul input is rounded to f32 first.
 * Outputs (each may be NULL): h_out[d_model] (final hidden, before the final
 * norm), logits[vocab] (f32), logit_abs[vocab] (sum |w*x| per logit, for the
 * tolerance), kv_out[n_layers/4 * 2 * fa_kv] (f32 k then v of each FA layer).
 * Returns argmax(logits).
 */
int64_t orc_decode_token(const orc_model* m, int64_t tok, double* h_out, float* logits,
                         double* logit_abs, float* kv_out);
/* Raw bytes of weights one token streams (Q4_K matrices plus the Q8_0 lm_head). */
int64_t orc_decode_weight_bytes(const orc_model* m);

/* ---- the mixer bodies of the hybrid stack, for the decode that runs them ----
 * "Qwen3.6-27B on Apple M3 Pro", model architecture list: Gated DeltaNet layers with a
 * short causal conv (kernel 4), 16 key heads / 48 value heads of 128, an f32 recurrent
 * state and a swish output gate; full-attention layers with 24 query / 4 KV heads of 256,
 * an output gate, qk-norm and partial RoPE (a quarter of each head) with theta 1e7.  The
 * pages name these parts only; the steps below are the published Gated DeltaNet
 * recurrence (Yang, Kautz and Hatamizadeh, "Gated Delta Networks: Improving Mamba2 with
 * Delta Rule", ICLR 2025) and gated softmax attention, in the plainest reading (listed
 * with the other readings in the design notes).  Everything in f64. */
typedef struct {
    int64_t nk, nv, dk, dv;   /* GDN key heads, value heads, key dim, value dim */
    int64_t conv;             /* causal conv taps */
    int64_t nq, nkv, dh;      /* full-attention query heads, KV heads, head dim */
    int64_t rot;              /* rotary dims at the front of each attention head */
    double theta;             /* RoPE base */
    double eps;               /* epsilon of every norm inside the mixers */
} orc_mixer_dims;
typedef struct {              /* per layer; the other kind's fields are NULL */
    const float* conv_w;      /* GDN [conv_dim][conv], conv_dim = 2*nk*dk + nv*dv */
    const float* a_log;       /* GDN [nv] */
    const float* dt_bias;     /* GDN [nv] */
    const float* norm_w;      /* GDN [dv]: gain of the gated RMSNorm */
    const float* q_norm_w;    /* FA [dh]: gain of the query RMSNorm */
    const float* k_norm_w;    /* FA [dh]: gain of the key RMSNorm */
} orc_mixer_params;
/* One step of a depthwise causal conv with K taps over n channels: y_c = sum_{j<K-1}
 * w[c][j]*state[c][j] + w[c][K-1]*x_c (no activation), then state[c] (the last K-1
 * inputs, oldest first) shifts in x_c.  w [n][K], state [n][K-1]. */
void orc_causal_conv_step(const float* w, double* state, const double* x, int64_t n, int64_t K, double* y);
/*
 * One Gated DeltaNet step.  t = in_proj output, laid out q [nk*dk] | k [nk*dk] |
 * v [nv*dv] | z [nv*dv] | b [nv] | a [nv].
 *  conv: channel c of q|k|v: y_c = silu(sum_{j<conv-1} w[c][j]*s[c][j] + w[c][conv-1]*t_c),
 *        then the state s[c] (the last conv-1 inputs, oldest first) shifts in t_c;
 *  q, k per key head: x / sqrt(sum x^2 + eps), q further times 1/sqrt(dk);
 *  per value head h (key head h / (nv/nk)): beta = sigmoid(b_h),
 *        g = -exp(a_log_h) * softplus(a_h + dt_bias_h),
 *        S_h = exp(g) S_h;  delta = beta (v_h - S_h^T k);  S_h += k delta^T;  o_h = S_h^T q
 *        (S_h is dk x dv);
 *  out_h = o_h / sqrt(mean(o_h^2) + eps) * norm_w * silu(z_h).
 * conv_state [conv_dim][conv-1] and S [nv][dk][dv] are updated in place; out [nv*dv];
 * o_raw [nv*dv] (may be NULL) receives o before the gated norm.
 */
void orc_gdn_step(const orc_mixer_dims* d, const orc_mixer_params* p, const double* t, double* conv_state,
                  double* S, double* out, double* o_raw);
/*
 * One gated full-attention step at position pos.  qg = q+gate output, per query head h:
 * q_h = qg[h*2dh, h*2dh+dh), gate_h = qg[h*2dh+dh, (h+1)*2dh); k, v [nkv*dh].
 *  q_h, k per head: x / sqrt(mean(x^2) + eps) * gain;
 *  RoPE on dims [0, rot): for i < rot/2, angle = pos * theta^(-2i/rot),
 *        (x_i, x_{i+rot/2}) -> (x_i cos - x_{i+rot/2} sin, x_{i+rot/2} cos + x_i sin);
 *  the normed, rotated k and v are written at position pos of kc, vc [nkv][max_ctx][dh];
 *  query head h reads KV head h / (nq/nkv): scores q.k_p / sqrt(dh) for p <= pos,
 *        softmax, o_h = sum_p w_p v_p;  out_h = o_h * sigmoid(gate_h).
 * out [nq*dh].
 */
void orc_attn_step(const orc_mixer_dims* d, const orc_mixer_params* p, const double* qg, const double* k,
                   const double* v, int64_t pos, int64_t max_ctx, double* kc, double* vc, double* out);

/* The recurrent state of a decode that runs the mixer bodies: per GDN layer the conv
 * state and S, per FA layer the KV cache, and the position.  Zeroed at creation. */
typedef struct orc_mixer_state orc_mixer_state;
orc_mixer_state* orc_mixer_state_create(const orc_model* m, const orc_mixer_dims* d, int64_t max_ctx);
void orc_mixer_state_destroy(orc_mixer_state* st);
/* orc_decode_token with the mixer bodies: the out_proj / o input is the GDN step's or the
 * attention step's output instead of t[0:n_mix]; the state advances by one token.
 * mp: per layer.  Outputs as orc_decode_token. */
int64_t orc_decode_token_mixer(const orc_model* m, const orc_mixer_dims* d, const orc_mixer_params* mp,
                               orc_mixer_state* st, int64_t tok, double* h_out, float* logits,
                               double* logit_abs);

/* ---- the prefill forward, projections only ----
 * P tokens through the stack in one pass, the mixer bodies left out as in
 * orc_decode_token (the out_proj / o input is t[0:n_mix]): the matmul-only floor
 * of the prefill ladder ("Qwen3.6-27B GDN-hybrid Metal prefill -- isolation
 * split", rung 3: both skips set, GEMMs and norms).  Every matmul input is an
 * activation rounded to f32 and then to bfloat16 (the prefill GEMM's operand,
 * orc_gemm_q4k); h stays f64.  Per layer and token p:
 *   n = bf16(rms(h_p)); t = W_in n; h_p += W_out bf16(t[0:n_mix]);
 *   n = bf16(rms(h_p)); h_p += W_down bf16(swiglu(W_gate n, W_up n)).
 * FA layers' k and v projections do not reach any output and are not computed.
 * Then logits = lm_head(f32(rms(h_{P-1}))) (Q8_0).  h_out [P][d_model] (may be
 * NULL) receives the final hidden states.  Returns argmax(logits). */
uint16_t orc_bf16_rne(float v);   /* nearest bfloat16, ties to even (NaN stays NaN) */
int64_t orc_prefill_forward(const orc_model* m, const int64_t* toks, int64_t P, double* h_out, float* logits,
                            double* logit_abs);

#ifdef __cplusplus
}
#endif
#endif
