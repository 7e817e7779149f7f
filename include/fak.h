/*
 * fak.h -- C ABI of the GB300 (sm_103a) Q4_K weight-only dequantize-and-multiply
 * library (libfak.so).
 *
 * The method follows three pages about one engine ("fak"):
 *   [diag]   "Mac Qwen3.6-27B Metal Q4_K perf diagnosis (2026-06-26)"
 *   [parity] "Qwen3.6-27B on Apple M3 Pro -- the llama.cpp parity bar"
 *   [prefill]"Qwen3.6-27B GDN-hybrid Metal prefill -- isolation split"
 * The pages give the problem (a Q4_K GEMV per projection, a GEMV batch in one
 * submission, a Q4_K prefill GEMM, and one GPU-resident submission per decode
 * token); they name the Q4_K format but print no layout or kernel, so the
 * byte layout below is the public GGML block_q4_K / block_q8_0 format.
 *
 * Conventions for every entry point:
 *  - Returns a fak_status (0 = FAK_OK).  Nothing throws across the ABI.
 *  - Shapes and alignment are validated on the host before any launch; a
 *    failed validation launches nothing.
 *  - "device" pointers are CUDA device (or managed) memory owned by the
 *    caller; the library never frees them.  "host" pointers are ordinary host
 *    memory owned by the caller.
 *  - Device calls are asynchronous on `stream` (a cudaStream_t, NULL = legacy
 *    default stream) and never synchronize, unless stated.
 *  - A launch error returns FAK_ERR_CUDA and clears the CUDA error state.
 *  - Errors found on the device (a bounded wait that timed out, a token id
 *    out of range) are written to a device status word and reported by
 *    fak_device_status() / fak_decode_status().
 *
 * Matrix layout: a weight matrix W has N rows (outputs) and K columns
 * (inputs), row-major, each row K/256 consecutive 144-byte Q4_K blocks
 * (or K/32 consecutive 34-byte Q8_0 blocks).
 *
 * Q4_K block (144 B, 256 weights, little-endian): binary16 d at byte 0,
 * binary16 dmin at byte 2, twelve bytes of packed 6-bit scales sc_0..7 and
 * mins m_0..7 at bytes 4..15, then 128 bytes of 4-bit quants: byte 16+32g+l
 * holds weight 64g+l in its low nibble and weight 64g+32+l in its high nibble.
 * Weight i of sub-block j = i/32 is d*sc_j*q_i - dmin*m_j.
 * Q8_0 block (34 B, 32 weights): binary16 d, then 32 int8 q; weight d*q.
 */
#ifndef FAK_H
#define FAK_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* fak_stream_t; /* identical to cudaStream_t */

typedef enum {
    FAK_OK = 0,
    FAK_ERR_INVALID_ARG = 1, /* null pointer or bad enum value */
    FAK_ERR_SHAPE = 2,       /* a dimension out of the supported range */
    FAK_ERR_ALIGN = 3,       /* a pointer not 16-byte aligned */
    FAK_ERR_CUDA = 4,        /* a CUDA runtime call or launch failed */
    FAK_ERR_TIMEOUT = 5,     /* a bounded device-side wait gave up */
    FAK_ERR_NOMEM = 6,       /* a workspace allocation failed */
    FAK_ERR_DEVICE = 7,      /* the device rejected an input (e.g. token id out of range) */
    FAK_ERR_UNSUPPORTED = 8  /* the current device is not sm_103 */
} fak_status;

/* Largest K (input length) the matrix-vector engine accepts: its quantized
 * copy of x must fit in shared memory next to the weight ring. */
#define FAK_ENGINE_MAX_K 18432

/* Short English description of a status code (static storage). */
const char* fak_strerror(int status);

/* Library version string (static storage). */
const char* fak_version(void);

/* ------------------------------------------------------------------ packers
 * Host-side quantizers ([diag] TL;DR and [parity] reconciliation table name
 * raw q4_k blocks resident in memory; the quantizer itself is not on the
 * pages: this is the covering min/max quantizer).
 *
 * fak_q4k_pack: w (host, f32, N x K row-major) -> out (host, N*(K/256)*144
 * bytes).  Per 256-weight super-block and 32-weight sub-block j:
 *   lo_j = min(0, min x), hi_j = max x, mn_j = -lo_j;
 *   dmin = smallest binary16 >= max_j(mn_j)/63;  m_j = min(63, ceil(mn_j/dmin));
 *   r_j = hi_j + dmin*m_j;  d = smallest binary16 >= max_j(r_j)/945;
 *   sc_j = min(63, ceil(r_j/(15*d)));  q = clamp(rint((x + dmin*m_j)/(d*sc_j)), 0, 15)
 * in f32 arithmetic (no fused multiply-add), 0 where a divisor is 0.  Every
 * weight then round-trips within half a quant step d*sc_j/2.
 * K % 256 != 0 or N < 0 -> FAK_ERR_SHAPE; out_bytes must equal the size.
 * Multi-threaded; the bytes do not depend on the thread count.
 *
 * fak_q8_0_pack: w (host, f32, N x K) -> out (host, N*(K/32)*34 bytes).
 *   d = binary16 nearest (ties to even) to max|x|/127;
 *   q = clamp(rint(x/d), -127, 127), 0 if d == 0.   K % 32 != 0 -> FAK_ERR_SHAPE.
 */
int fak_q4k_pack(const float* w, int64_t N, int64_t K, void* out, size_t out_bytes);
int fak_q8_0_pack(const float* w, int64_t N, int64_t K, void* out, size_t out_bytes);

/* The same two quantizers on the GPU (one thread per block), for weights that
 * are already in device memory: w and out are device pointers (w 4-byte
 * aligned), asynchronous on `stream`.  The bytes equal the host packers' bit
 * for bit.  Same shape rules and sizes as the host versions. */
int fak_q4k_pack_device(const float* w, int64_t N, int64_t K, void* out, size_t out_bytes, fak_stream_t stream);
int fak_q8_0_pack_device(const float* w, int64_t N, int64_t K, void* out, size_t out_bytes, fak_stream_t stream);

/* ------------------------------------------------------------------ GEMV
 * y = W x for one activation vector ([diag] TL;DR: the Q4_K GEMV a decode
 * token runs per projection; section 4b: the single-GEMV benchmark).
 *   Wq: device, N rows of K/256 Q4_K blocks, 16-byte aligned.
 *   x:  device f32 [K], 16-byte aligned.     y: device f32 [N].
 *   1 <= N <= 2^31-1, 256 <= K <= FAK_ENGINE_MAX_K, K % 256 == 0.
 * Accumulates exactly in integers per sub-block after splitting x into a
 * 23-bit block-scaled fixed-point form (three byte limbs per element), then
 * in f32; |error| stays within 1e-5 * sum|w_i x_i| + 1e-6 of the exact dot.
 * Deterministic: the same inputs give bitwise identical y.
 */
int fak_q4k_gemv(const void* Wq, int64_t N, int64_t K, const float* x, float* y, fak_stream_t stream);

/* The int8-activation variant of fak_q4k_gemv ([parity] reconciliation table:
 * the int8-SDOT Metal decode GEMV path, checked by cosine).  Each 32-element
 * sub-block of x becomes d_j * X_k with d_j = max|x| / 127 and
 * X_k = rint(x_k * (127 / max|x|)) in [-127, 127] (f32 arithmetic, ties to
 * even); y is then the f32-accumulate dot of W with that quantized x, exact
 * per sub-block in integers, so it meets 1e-5 * sum|w_i x~_i| + 1e-6 against
 * the quantized activations x~ -- not against x: the quantization itself
 * moves each element by up to max|x| / 254 of its sub-block.  One third of
 * the integer work of fak_q4k_gemv.  Same arguments, limits and determinism. */
int fak_q4k_gemv_i8x(const void* Wq, int64_t N, int64_t K, const float* x, float* y, fak_stream_t stream);

/* Same for a Q8_0 matrix (the lm_head format of [diag] section 2, lm_head_q8).
 * K % 256 == 0 (so rows stay 16-byte aligned), K <= FAK_ENGINE_MAX_K. */
int fak_q8_0_gemv(const void* Wq, int64_t N, int64_t K, const float* x, float* y, fak_stream_t stream);

/* ------------------------------------------------------------------ batched GEMV
 * Y[m,:] = W X[m,:] for M activation rows against one resident weight
 * ([diag] section 4b: GEMVBatch, N GEMVs of one weight in one submission).
 *   X: device f32 [M, K] row-major, 16-byte aligned; Y: device f32 [M, N];
 *   1 <= M <= 64; 1 <= N < 2^31; 256 <= K <= 2^24, K % 256 == 0.
 *   W is read from HBM once per call, not once per row.  M == 1 is the
 *   matrix-vector engine (fak_q4k_gemv, limits as there).  M >= 2 runs on
 *   the tensor cores: x is split into two fp16 parts per 256-wide block with a
 *   power-of-two scale, sc*q is exact in fp16, and the per-block scales d,
 *   dmin are applied in f32, so the error bound is the f32 one of
 *   fak_q4k_gemv for finite X.  Two launches (x split, then the GEMV); the
 *   call takes a stream-ordered scratch of about 4*M'*K bytes (M' = M rounded
 *   up to 8, 16, 32 or 64), plus 4*splits*M*N bytes when few row tiles force a
 *   K split, and frees it on the same stream.  The scratch comes from a
 *   library-owned memory pool per device that keeps its memory for later
 *   calls until the process exits (while the stream is being captured into a
 *   graph: cudaMallocAsync, a graph memory node).  Returns FAK_ERR_NOMEM if
 *   that allocation fails.
 */
int fak_q4k_gemv_batch(const void* Wq, int64_t N, int64_t K, const float* X, int M, float* Y,
                       fak_stream_t stream);

/* ------------------------------------------------------------------ MLP decode
 * One batch-1 SwiGLU MLP on Q4_K weights ([diag] section 2, mlp_decode, 54% of
 * decode; [parity] architecture: RMSNorm eps 1e-6, SwiGLU):
 *   n = x / sqrt(mean(x^2) + eps);  a = silu(Wgate n) * (Wup n);  y = Wdown a
 * with unit RMSNorm gain.  Wgate, Wup: [d_ff x d_model]; Wdown: [d_model x d_ff].
 *   x: device f32 [d_model]; y: device f32 [d_model] (may not alias x).
 *   workspace: device, >= fak_mlp_workspace_bytes(d_ff) bytes, 256-byte
 *   aligned, owned by the caller, not shared with a concurrent call.
 * Runs as ONE kernel launch (both matmuls, the norm and SwiGLU inside, with a
 * bounded grid-wide wait between them).
 */
size_t fak_mlp_workspace_bytes(int64_t d_ff);
int fak_mlp_decode(const void* Wgate, const void* Wup, const void* Wdown, int64_t d_model, int64_t d_ff,
                   const float* x, float eps, float* y, void* workspace, size_t workspace_bytes,
                   fak_stream_t stream);

/* The same MLP for callers that cannot allocate device memory at call time
 * (a host-side memory planner owns the device, or the call sits where an
 * allocation's implicit synchronization is not allowed).  This entry point
 * has no counterpart on the pages; it is a packaging of fak_mlp_decode.
 * It allocates nothing: its scratch is a file-scope device array in the
 * library, sized for d_ff <= FAK_MLP_NOALLOC_MAX_FF (about 74 KB), held on
 * every GPU that loads the library until the process exits.  The first call
 * on a device looks up that array's device address and keeps it for the life
 * of the process, so make that first call before any stream capture; calls
 * after a cudaDeviceReset() of that device are not supported (the kept
 * address would be stale).  Larger d_ff returns FAK_ERR_SHAPE.  All calls
 * share the one array: calls that overlap on the GPU (different streams, no
 * ordering between them) race and give wrong results.  Other arguments,
 * limits and results as fak_mlp_decode. */
#define FAK_MLP_NOALLOC_MAX_FF 18432
int fak_mlp_decode_noalloc(const void* Wgate, const void* Wup, const void* Wdown, int64_t d_model, int64_t d_ff,
                           const float* x, float eps, float* y, fak_stream_t stream);

/* ------------------------------------------------------------------ prefill GEMM
 * Y = X W^T for P tokens ([diag] section 2: mlp_gate_up_proj and mlp_down_proj
 * dominate prefill; section 4b: the q4k_gemm prefill kernel).
 *   Wq: device Q4_K [N x K]; X: device bf16 [P, K] row-major (bit patterns);
 *   Y: device f32 [P, N].  K % 256 == 0, N >= 1, P >= 1 (a last partial
 *   128-row tile reads zero-filled rows past N and writes none of them).
 * Tensor cores (tcgen05, bf16 x bf16 -> f32): W is dequantized to bf16 in
 * shared memory, so |error| <= 5e-3 * sum|w_i x_i| + 1e-5.  Deterministic.
 * When whole 128 x 256 output tiles would fill the GPU poorly (few tiles, or a
 * last wave far from full), the work is split stream-K: the tiles' K ranges,
 * laid end to end, are cut into one equal range per SM; the pieces of a tile
 * met by several CTAs are summed in K order by a second, small kernel launched
 * right after (programmatic dependent launch; deterministic).  The call then
 * takes a stream-ordered workspace of 128 KB per tile and piece and frees it
 * on the same stream.  It comes from the same
 * library-owned pool as the batched GEMV's scratch (kept for later calls until
 * the process exits; a graph memory node under stream capture); FAK_ERR_NOMEM
 * if that fails.
 */
int fak_q4k_gemm(const void* Wq, int64_t N, int64_t K, const void* X, int64_t P, float* Y,
                 fak_stream_t stream);

/* Elementwise X2[p, i] = bf16(silu(Y1[p, i]) * Y1[p, half + i]) for i < half:
 * the SwiGLU between the fused gate||up prefill GEMM and the down GEMM.
 * Y1: device f32 [P, 2*half]; X2: device bf16 [P, half]. */
int fak_swiglu_bf16(const float* Y1, int64_t P, int64_t half, void* X2, fak_stream_t stream);

/* The gate||up prefill GEMM with the SwiGLU in its epilogue (the fused form of
 * fak_q4k_gemm then fak_swiglu_bf16; the pages' diagnosis, section 4b: the
 * q4k_gemm prefill kernel, and the SwiGLU of the MLP in section 2):
 *   X2[p, c] = bf16(silu(g) * u),  g = sum_k Wg[c, k] X[p, k],  u = sum_k Wu[c, k] X[p, k]
 * without writing the f32 [P, 2F] product.
 *   W13: device Q4_K [2F x K] in the interleaved row order written by
 *        fak_q4k_interleave_gate_up (rows 32b..32b+15 = gate channels
 *        16b..16b+15, rows 32b+16..32b+31 = up channels 16b..16b+15);
 *   X: device bf16 [P, K]; X2: device bf16 [P, F], 16-byte aligned.
 *   F % 64 == 0, K % 256 == 0, P >= 1.
 * Each (g, u) pair is accumulated exactly as fak_q4k_gemm accumulates that row
 * in a whole tile (same K order, never split), and silu(g)*u is the expression
 * fak_swiglu_bf16 uses, so X2 equals fak_swiglu_bf16(fak_q4k_gemm(W1)) bit for
 * bit whenever that GEMM takes whole tiles (W1 = gate rows then up rows).
 * Errors as fak_q4k_gemm.
 */
int fak_q4k_gemm_swiglu(const void* W13, int64_t F, int64_t K, const void* X, int64_t P, void* X2,
                        fak_stream_t stream);

/* Writes W13 (device, 2F * K/256 * 144 bytes) from the Q4_K gate and up
 * weights Wg, Wu (device, F * K/256 * 144 bytes each) in the row order
 * fak_q4k_gemm_swiglu reads: a row permutation, bytes copied unchanged.
 * F % 64 == 0, K % 256 == 0; all three pointers 16-byte aligned and W13
 * disjoint from Wg and Wu. */
int fak_q4k_interleave_gate_up(const void* Wg, const void* Wu, int64_t F, int64_t K, void* W13,
                               fak_stream_t stream);

/* ------------------------------------------------------------------ decode step
 * One decode token of the hybrid stack as ONE launch ([diag] section 4, the
 * "one-command-buffer-per-token GPU-resident decode forward": the activation
 * stays on the GPU across every projection and MLP matmul, one submission
 * per token).  Per token:
 *   h = E[tok]; for each layer: n = rms(h);
 *     GDN layer: t = Win n; h += Wout t[0:n_mix]
 *     FA  layer: t = Wqg n; k = Wk n; v = Wv n; h += Wo t[0:n_mix]
 *   (the mixer bodies between the projections are outside this library);
 *   n = rms(h); h += Wdown(silu(Wgate n) * (Wup n));
 *   finally logits = Wlm rms(h) (Q8_0) and tok' = argmax(logits), lowest
 *   index on ties.  RMSNorm gain is 1.
 */
enum { FAK_LAYER_GDN = 0, FAK_LAYER_FA = 1 };
/* ONE_LAUNCH: the whole token is one cooperative launch; PER_MATMUL: one launch
 * per step.  The _I8X modes are the same launch shapes with every Q4_K step on
 * int8 activations (fak_q4k_gemv_i8x); the Q8_0 lm_head keeps the exact form.
 * PER_MATMUL_HOST_WAIT is PER_MATMUL with the host waiting for each launch to
 * finish (cudaStreamSynchronize) before it issues the next: the shape of the
 * pages' Metal path, one command buffer per matmul, each committed and waited
 * on ("Mac Qwen3.6-27B Metal Q4_K perf diagnosis", TL;DR and section 4b).  It
 * returns after the token has finished on the device. */
enum { FAK_DECODE_ONE_LAUNCH = 0, FAK_DECODE_PER_MATMUL = 1, FAK_DECODE_ONE_LAUNCH_I8X = 2,
       FAK_DECODE_PER_MATMUL_I8X = 3, FAK_DECODE_PER_MATMUL_HOST_WAIT = 4 };

typedef struct {
    int32_t kind;          /* FAK_LAYER_GDN or FAK_LAYER_FA */
    const void* w_in;      /* GDN in_proj [gdn_in x d_model] / FA q+gate [fa_qg x d_model], Q4_K, device */
    const void* w_k;       /* FA only: [fa_kv x d_model] Q4_K, device (NULL for GDN) */
    const void* w_v;       /* FA only */
    const void* w_out;     /* GDN out_proj / FA o: [d_model x n_mix] Q4_K, device */
    const void* w_gate;    /* [d_ff x d_model] Q4_K, device */
    const void* w_up;      /* [d_ff x d_model] */
    const void* w_down;    /* [d_model x d_ff] */
} fak_layer_desc;

typedef struct {
    int32_t n_layers;
    int32_t d_model, d_ff, vocab;
    int32_t gdn_in, fa_qg, fa_kv, n_mix;
    float eps;
    int32_t mode;                 /* FAK_DECODE_ONE_LAUNCH, _PER_MATMUL, _ONE_LAUNCH_I8X, _PER_MATMUL_I8X
                                     or _PER_MATMUL_HOST_WAIT */
    const fak_layer_desc* layers; /* host array of n_layers; copied by fak_decode_create */
    const void* lm_head;          /* [vocab x d_model] Q8_0, device */
    const float* embedding;       /* [vocab x d_model] f32, device */
    const struct fak_mixer_desc* mixer; /* NULL: projections only (the out_proj / o input is
                                           t[0:n_mix]); else the mixer bodies run, below */
} fak_decode_desc;

/* ------------------------------------------------------------------ mixer bodies
 * With desc.mixer set, each layer runs its mixer between the input projections
 * and out_proj / o ("Qwen3.6-27B on Apple M3 Pro", model architecture list: Gated
 * DeltaNet layers with a causal conv of 4 taps, key / value heads of 128 and an
 * f32 recurrent state, a swish output gate; full-attention layers with GQA,
 * head dim 256, an output gate, qk-norm and partial RoPE; "Mac Qwen3.6-27B Metal
 * Q4_K perf diagnosis", section 4: the recurrence and attention run on the GPU
 * inside the one-submission decode).  The steps are the published Gated DeltaNet
 * recurrence and gated softmax attention; each layer adds one step to the launch.
 *
 * GDN layer, in_proj output t laid out q [nk*dk] | k [nk*dk] | v [nv*dv] |
 * z [nv*dv] | b [nv] | a [nv] (so gdn_in = 2*nk*dk + 2*nv*dv + 2*nv):
 *   causal conv over q|k|v (taps conv_w[c][0..3], the newest input on tap 3),
 *   silu; q, k per key head divided by sqrt(sum^2 + eps), q also by sqrt(dk);
 *   per value head h (key head h / (nv/nk)): beta = sigmoid(b_h),
 *   g = -exp(a_log_h) * softplus(a_h + dt_bias_h), S_h = exp(g) S_h,
 *   S_h += k (beta (v_h - S_h^T k))^T, o_h = S_h^T q;
 *   out_h = o_h / sqrt(mean(o_h^2) + eps) * norm_w * silu(z_h).
 * FA layer, q+gate output laid out per query head [q (dh) | gate (dh)]:
 *   q_h and k per head: x / sqrt(mean(x^2) + eps) * gain; RoPE on dims [0, rot)
 *   (pairs (i, i + rot/2), angle pos * theta^(-2i/rot)); k, v appended to the
 *   KV cache at the position; query head h attends KV head h / (nq/nkv) over
 *   positions 0..pos with scores q.k / sqrt(dh); out_h = softmax-weighted v *
 *   sigmoid(gate_h).
 * The state (conv states, S, KV cache, position) lives in the context, starts at
 * zero and advances one token per fak_decode_step; fak_decode_reset clears it.
 * Supported: dk = dv = 128, dh = 256, conv = 4, nv <= 152 and nq <= 152 (one
 * CTA per head), nv % nk == 0, nq % nkv == 0, rot even and <= dh,
 * n_mix == nv*dv == nq*dh.  A step past max_ctx positions records
 * FAK_ERR_DEVICE (attention uses the first max_ctx positions only): its
 * attention output is zero, the KV cache is not written, the step still ends
 * at once, and fak_decode_status, on reporting it, clears the state (the next
 * step is position 0 of a new sequence).
 */
typedef struct {
    const float* conv_w;     /* GDN: [2*nk*dk + nv*dv][4] f32, device */
    const float* a_log;      /* GDN: [nv] f32, device */
    const float* dt_bias;    /* GDN: [nv] f32, device */
    const float* norm_w;     /* GDN: [dv] f32, device (gated RMSNorm gain) */
    const float* q_norm_w;   /* FA: [dh] f32, device (query RMSNorm gain) */
    const float* k_norm_w;   /* FA: [dh] f32, device (key RMSNorm gain) */
} fak_mixer_layer;

typedef struct fak_mixer_desc {
    int32_t gdn_nk, gdn_nv, gdn_dk, gdn_dv;  /* GDN key heads, value heads, key dim, value dim */
    int32_t fa_nq, fa_nkv, fa_dh, fa_rot;    /* FA query heads, KV heads, head dim, rotary dims */
    float rope_theta, eps;
    int32_t max_ctx;                         /* KV cache positions */
    const fak_mixer_layer* layers;           /* host array of n_layers; copied by fak_decode_create */
} fak_mixer_desc;

typedef struct fak_decode fak_decode;

/* Validates the description and allocates the context's device scratch
 * (hidden state, projection outputs, k/v outputs, SwiGLU output, argmax
 * candidates, sync counters, status word, the op list).  The weights stay
 * owned by the caller and must outlive the context.  Limits: d_model,
 * n_mix, d_ff <= FAK_ENGINE_MAX_K and multiples of 256; n_mix <= max(gdn_in,
 * fa_qg).  ONE_LAUNCH needs a device that can co-schedule one block per SM. */
int fak_decode_create(const fak_decode_desc* desc, fak_decode** out);

/* One token: reads d_tok_in (device int32), writes d_tok_out (device int32;
 * may equal d_tok_in), and, if d_logits (device f32 [vocab]) is not NULL,
 * the logits.  Asynchronous; ONE_LAUNCH issues a single kernel launch,
 * PER_MATMUL one launch per matmul (same arithmetic, bitwise identical
 * results).  Returns a status left on the device by an earlier step without
 * synchronizing (it reads the status word only after a previous
 * fak_decode_status). */
int fak_decode_step(fak_decode* ctx, const int32_t* d_tok_in, int32_t* d_tok_out, float* d_logits,
                    fak_stream_t stream);

/* Synchronizes `stream`, reads and clears the context's device status word:
 * FAK_OK, FAK_ERR_TIMEOUT (a grid-wide wait gave up; the counters are reset
 * so the context stays usable) or FAK_ERR_DEVICE (token id out of range). */
int fak_decode_status(fak_decode* ctx, fak_stream_t stream);

/* Clears the state a decode with the mixer bodies carries from token to token
 * (conv states, S, KV cache, position) and the context's tagged buffers, on
 * `stream`: the next step starts a new sequence at position 0. */
int fak_decode_reset(fak_decode* ctx, fak_stream_t stream);

/* Copies part of the context's state after a step into dst (host or device
 * memory, caller-owned), stream-ordered on `stream`:
 *   which = 0: the hidden state h [d_model] (before the final norm);
 *   which = 1: the k and v projections of every FA layer, [n_fa][2][fa_kv];
 *   which = 2: the mixer output of the last layer, [n_mix] (the out_proj / o
 *              input; with desc.mixer == NULL, t[0:n_mix] of the last layer).
 * `count` must equal the number of floats of that buffer. */
int fak_decode_read_state(fak_decode* ctx, int which, float* dst, size_t count, fak_stream_t stream);

/* Number of kernel launches one fak_decode_step issues. */
int fak_decode_launches_per_step(const fak_decode* ctx);

/* Test hook: the grid-wide wait timeout in nanoseconds (default 1 s).  A
 * step whose wait cannot complete within it returns early with
 * FAK_ERR_TIMEOUT in the status word instead of hanging. */
int fak_decode_set_timeout_ns(fak_decode* ctx, int64_t ns);

/* Test hook: make op `op_index` of the next step wait for one more arrival
 * than the grid can provide (a wait that can never complete), to check the
 * bounded-wait error path.  -1 clears it. */
int fak_decode_debug_unreachable_wait(fak_decode* ctx, int op_index);

void fak_decode_destroy(fak_decode* ctx);

/* ------------------------------------------------------------------ prefill forward
 * P prompt tokens through the whole stack as ONE submission ("Mac Qwen3.6-27B
 * Metal Q4_K perf diagnosis", section 4: the resident prefill forward that runs
 * the whole prefill in one command buffer; "Qwen3.6-27B GDN-hybrid Metal
 * prefill -- isolation split": the P = 256 / 512 / 1024 ladder, rung 3 with both
 * stage skips set -- GEMMs and norms only).  Same model description as the
 * decode (desc.mixer must be NULL: the mixer bodies are left out, the out_proj /
 * o input is t[:, 0:n_mix]).  Per layer, for every token p:
 *   n = bf16(rms(h_p)); t = W_in n (FA: also W_k n, W_v n); h_p += W_out bf16(t[0:n_mix]);
 *   n = bf16(rms(h_p)); h_p += W_down bf16(silu(W_gate n) * (W_up n))
 * on the tcgen05 dequant-GEMM (bf16 operands, f32 accumulate: the fak_q4k_gemm
 * error bar per matmul), then logits = lm_head(rms(h_{P-1})) (Q8_0, f32) and the
 * argmax (lowest index on ties).
 *
 * fak_prefill_create allocates the activations for P tokens (1 <= P <= 16384),
 * an interleaved copy of every layer's gate / up weights (2 * d_ff * d_model /
 * 256 * 144 bytes per layer, for the SwiGLU fused into the GEMM epilogue), a
 * copy of every FA layer's q+gate, k and v weights as one matrix ((fa_qg + 2 *
 * fa_kv) * d_model / 256 * 144 bytes, so that the three share one GEMM), and
 * records the forward into a CUDA graph.  The weights stay caller-owned and
 * must outlive the context.  d_model <= 8192; gdn_in and fa_qg multiples of 4,
 * fa_kv of 2, n_mix of 256, d_ff of 64 (else FAK_ERR_SHAPE).
 * fak_prefill_run: d_tokens (device int32 [P]) in; d_tok_out (device int32) =
 * the argmax of the last token's logits; d_logits (device f32 [vocab], nullable).
 * One graph launch (plus the copies of the tokens in and the results out),
 * asynchronous on `stream`.
 * fak_prefill_read_hidden: the final hidden states h [P, d_model] (before the
 * final norm) into dst (host or device), count = P * d_model.
 * fak_prefill_kernels: kernel launches in the recorded graph.
 * fak_prefill_status: synchronizes `stream`, then reads and clears the device
 * status (FAK_ERR_DEVICE: a token id out of range; FAK_ERR_TIMEOUT: a GEMM wait). */
typedef struct fak_prefill fak_prefill;
int fak_prefill_create(const fak_decode_desc* desc, int64_t P, fak_prefill** out);
int fak_prefill_run(fak_prefill* ctx, const int32_t* d_tokens, int32_t* d_tok_out, float* d_logits,
                    fak_stream_t stream);
int fak_prefill_read_hidden(fak_prefill* ctx, float* dst, size_t count, fak_stream_t stream);
int fak_prefill_kernels(const fak_prefill* ctx);
int fak_prefill_status(fak_prefill* ctx, fak_stream_t stream);
void fak_prefill_destroy(fak_prefill* ctx);

/* ------------------------------------------------------------------ status
 * Synchronizes `stream`, then reads and clears the status word shared by the
 * stateless calls (GEMV, batched GEMV, MLP, GEMM). */
int fak_device_status(fak_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* FAK_H */
