// The prefill forward as one submission: P prompt tokens through the whole
// stack with every activation resident on the GPU, captured once into a CUDA
// graph and replayed by one graph launch per prefill ("Mac Qwen3.6-27B Metal
// Q4_K perf diagnosis", section 4: the resident prefill forward, mg_prefill,
// runs the whole prefill in one command buffer; "Qwen3.6-27B GDN-hybrid Metal
// prefill -- isolation split": the P = 256 / 512 / 1024 ladder, whose rung 3,
// both stage skips set, is the matmul-only floor built here).
//
// Per layer: n = bf16(rms(h)); t = W_in n; h += W_out bf16(t[:, 0:n_mix]);
// n = bf16(rms(h)); h += W_down bf16(silu(W_gate n) * (W_up n)); the mixer
// bodies are left out as in the projections-only decode.  The matmuls are the
// tcgen05 dequant-GEMMs of gemm.cu (the gate / up GEMM with the SwiGLU in its
// epilogue, on an interleaved copy of the two weights made at creation); the
// norms, residual adds and bf16 conversions are the small kernels below, one
// CTA per token row.  The last token's logits come from the matrix-vector
// engine (Q8_0 lm_head) and an argmax kernel.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <vector>

#include "fak.h"
#include "fak_device.cuh"

namespace {

constexpr int kRowThreads = 256;

__device__ int g_prefill_status;

// h[p, :] = E[toks[p], :]; an out-of-range token records FAK_ERR_DEVICE and reads row 0.
__global__ void __launch_bounds__(kRowThreads) embed_rows_kernel(const int32_t* toks, const float* E, int64_t vocab,
                                                                 int D, float* h) {
  const int p = blockIdx.x;
  int tok = toks[p];
  if (tok < 0 || tok >= vocab) {
    if (threadIdx.x == 0) atomicCAS(&g_prefill_status, 0, FAK_ERR_DEVICE);
    tok = 0;
  }
  const float4* src = reinterpret_cast<const float4*>(E + (int64_t)tok * D);
  float4* dst = reinterpret_cast<float4*>(h + (int64_t)p * D);
  for (int i = threadIdx.x; i < D / 4; i += kRowThreads) dst[i] = src[i];
}

// Sum over the block in a fixed order (every thread gets the same value).
__device__ __forceinline__ float row_sum(float v, float* scr) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) scr[threadIdx.x >> 5] = v;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int w = 0; w < kRowThreads / 32; ++w) t += scr[w];
  __syncthreads();
  return t;
}

// Row p: optionally h += y (the residual add of the previous matmul), then
// n = bf16(h / sqrt(mean(h^2) + eps)).  D % 128 == 0, D <= 8 * 4 * kRowThreads.
// When pc.ws is set, y came from a stream-K GEMM whose cut tiles were left as pieces: the columns of
// such a tile are the sum of its pieces in K order (as the GEMM's own fix-up would sum them), read
// here instead of y; the other tiles were written to y.
__global__ void __launch_bounds__(kRowThreads) add_rms_bf16_kernel(float* h, const float* y, const FakGemmPieces pc,
                                                                   int D, float eps, __nv_bfloat16* n) {
  __shared__ float scr[kRowThreads / 32];
  __shared__ int npc[64];  // pieces of each 128-row tile in this token's tile column
  const int64_t p = blockIdx.x, off = p * D;
  const int pt = (int)(p / 256), col = (int)(p % 256);
  if (y && pc.ws) {
    for (int j = threadIdx.x; j < D / 128; j += kRowThreads) {
      const int64_t t = (int64_t)j * pc.n_tiles_p + pt;
      const int64_t tb = t * pc.nsb, te = tb + pc.nsb;
      const int64_t cf = ((tb + 1) * pc.gs + pc.work - 1) / pc.work - 1, cl = (te * pc.gs + pc.work - 1) / pc.work - 1;
      npc[j] = (int)(cl - cf + 1);
    }
    __syncthreads();
  }
  float4 v[8];
  float ss = 0.0f;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = threadIdx.x + k * kRowThreads;
    if (i < D / 4) {
      v[k] = reinterpret_cast<const float4*>(h + off)[i];
      if (y) {
        const int j = i >> 5, q = 4 * (i & 31);  // 128-row tile of these four columns, and the row in it
        float4 r;
        if (pc.ws && npc[j] > 1) {
          const float4* src = reinterpret_cast<const float4*>(
              pc.ws + (((int64_t)j * pc.n_tiles_p + pt) * pc.maxp * 256 + col) * 128 + q);
          r = __ldcg(src);
          for (int kk = 1; kk < npc[j]; ++kk) {
            const float4 u = __ldcg(src + (int64_t)kk * (256 * 128 / 4));
            r.x += u.x;
            r.y += u.y;
            r.z += u.z;
            r.w += u.w;
          }
        } else {
          r = reinterpret_cast<const float4*>(y + off)[i];
        }
        v[k].x += r.x;
        v[k].y += r.y;
        v[k].z += r.z;
        v[k].w += r.w;
        reinterpret_cast<float4*>(h + off)[i] = v[k];
      }
      ss = fmaf(v[k].x, v[k].x, fmaf(v[k].y, v[k].y, fmaf(v[k].z, v[k].z, fmaf(v[k].w, v[k].w, ss))));
    }
  }
  const float r = 1.0f / sqrtf(row_sum(ss, scr) / (float)D + eps);
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int i = threadIdx.x + k * kRowThreads;
    if (i < D / 4) {
      __nv_bfloat162 a = __floats2bfloat162_rn(v[k].x * r, v[k].y * r);
      __nv_bfloat162 b = __floats2bfloat162_rn(v[k].z * r, v[k].w * r);
      reinterpret_cast<__nv_bfloat162*>(n + off)[2 * i] = a;
      reinterpret_cast<__nv_bfloat162*>(n + off)[2 * i + 1] = b;
    }
  }
}

// h += y for every row, then the last row's RMSNorm in f32 (the lm_head input).
__global__ void __launch_bounds__(kRowThreads) add_rows_kernel(float* h, const float* y, int64_t n4) {
  for (int64_t i = (int64_t)blockIdx.x * kRowThreads + threadIdx.x; i < n4; i += (int64_t)gridDim.x * kRowThreads) {
    float4 a = reinterpret_cast<float4*>(h)[i];
    const float4 b = reinterpret_cast<const float4*>(y)[i];
    a.x += b.x;
    a.y += b.y;
    a.z += b.z;
    a.w += b.w;
    reinterpret_cast<float4*>(h)[i] = a;
  }
}

__global__ void __launch_bounds__(kRowThreads) last_rms_kernel(const float* hrow, int D, float eps, float* out) {
  __shared__ float scr[kRowThreads / 32];
  float ss = 0.0f;
  for (int i = threadIdx.x; i < D; i += kRowThreads) ss = fmaf(hrow[i], hrow[i], ss);
  const float r = 1.0f / sqrtf(row_sum(ss, scr) / (float)D + eps);
  for (int i = threadIdx.x; i < D; i += kRowThreads) out[i] = hrow[i] * r;
}

// X2[p, i] = bf16(T[p, i]) for i < n (the out_proj / o input: the first n channels of t).
// ld % 4 == 0, n % 4 == 0: four channels per float4 load and one 8-byte store, eight loads of a
// thread in flight before its stores.
__global__ void __launch_bounds__(kRowThreads) slice_bf16_kernel(const float* T, int64_t ld, int n,
                                                                 __nv_bfloat16* X2) {
  const int64_t p = blockIdx.x;
  const float4* src = reinterpret_cast<const float4*>(T + p * ld);
  uint2* dst = reinterpret_cast<uint2*>(X2 + p * n);
  const int n4 = n / 4;
  for (int i0 = threadIdx.x; i0 < n4; i0 += 8 * kRowThreads) {
    float4 v[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = i0 + k * kRowThreads;
      if (i < n4) v[k] = src[i];
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int i = i0 + k * kRowThreads;
      if (i < n4) {
        const __nv_bfloat162 a = __floats2bfloat162_rn(v[k].x, v[k].y), b = __floats2bfloat162_rn(v[k].z, v[k].w);
        dst[i] = make_uint2(*reinterpret_cast<const uint32_t*>(&a), *reinterpret_cast<const uint32_t*>(&b));
      }
    }
  }
}

// argmax with the lowest index on ties (NaN skipped): every thread folds its values into one
// 64-bit key (order-preserving value bits, then the complemented index) with atomicMax.
__device__ __forceinline__ unsigned long long argmax_key(float v, int idx) {
  const uint32_t u = __float_as_uint(v);
  const uint32_t ord = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)ord << 32) | (uint32_t)(0xFFFFFFFFu - (uint32_t)idx);
}

__global__ void __launch_bounds__(kRowThreads) argmax_kernel(const float* v, int n, unsigned long long* slot) {
  unsigned long long best = 0;
  for (int i = blockIdx.x * kRowThreads + threadIdx.x; i < n; i += gridDim.x * kRowThreads) {
    const float x = v[i];
    if (x == x) best = max(best, argmax_key(x, i));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) best = max(best, __shfl_xor_sync(0xffffffffu, best, o));
  if ((threadIdx.x & 31) == 0 && best) atomicMax(slot, best);
}

__global__ void argmax_finish_kernel(const unsigned long long* slot, int32_t* tok) {
  const unsigned long long k = *slot;
  *tok = k ? (int32_t)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFull)) : 0;
}

}  // namespace

struct fak_prefill {
  fak_decode_desc desc;
  std::vector<fak_layer_desc> layers;
  int64_t P = 0;
  int sms = 0;
  int32_t* toks = nullptr;
  float* h = nullptr;              // [P, D]
  __nv_bfloat16* n = nullptr;      // [P, D]
  float* T = nullptr;              // [P, max(gdn_in, fa_qg + 2 fa_kv)]
  __nv_bfloat16* X2 = nullptr;     // [P, max(n_mix, d_ff)]
  float* Y = nullptr;              // [P, D]
  float* ws = nullptr;             // stream-K pieces of the out_proj / o and down GEMMs, summed by add+RMSNorm
  size_t ws_bytes = 0;
  float* nlast = nullptr;          // [D]
  float* logits = nullptr;         // [vocab]
  unsigned long long* slot = nullptr;
  int32_t* tok = nullptr;
  std::vector<uint8_t*> w13;       // per layer: gate / up rows interleaved for the fused SwiGLU GEMM
  std::vector<uint8_t*> wqkv;      // per FA layer: q+gate, k and v rows in one matrix (one GEMM); GDN: null
  cudaGraph_t graph = nullptr;
  cudaGraphExec_t exec = nullptr;
  size_t kernels = 0;
};

namespace {

void free_prefill(fak_prefill* c) {
  if (!c) return;
  if (c->exec) cudaGraphExecDestroy(c->exec);
  if (c->graph) cudaGraphDestroy(c->graph);
  for (uint8_t* w : c->w13) cudaFree(w);
  for (uint8_t* w : c->wqkv) cudaFree(w);
  cudaFree(c->toks);
  cudaFree(c->h);
  cudaFree(c->n);
  cudaFree(c->T);
  cudaFree(c->X2);
  cudaFree(c->Y);
  cudaFree(c->ws);
  cudaFree(c->nlast);
  cudaFree(c->logits);
  cudaFree(c->slot);
  cudaFree(c->tok);
  delete c;
}

int launch_status(cudaError_t e) { return fak_cuda_status(e == cudaSuccess ? cudaGetLastError() : e); }

// The whole forward on stream s (captured into the graph by fak_prefill_create).
int record_forward(fak_prefill* c, cudaStream_t s) {
  const fak_decode_desc& d = c->desc;
  const int D = d.d_model, F = d.d_ff;
  const int64_t P = c->P;
  int st;
  embed_rows_kernel<<<(unsigned)P, kRowThreads, 0, s>>>(c->toks, d.embedding, d.vocab, D, c->h);
  if ((st = launch_status(cudaSuccess)) != FAK_OK) return st;
  const float* pending = nullptr;  // a matmul output still to be added into h
  FakGemmPieces pend_pc{};         // ... and its stream-K pieces, if it left them
  for (int l = 0; l < d.n_layers; ++l) {
    const fak_layer_desc& L = c->layers[l];
    // FA: q+gate, k and v share their input, so they run as one GEMM on the concatenated copy
    // (t[:, fa_qg:] holds k and v: they belong to the forward's work; the mixer body that reads them
    // is left out)
    const bool fa = L.kind == FAK_LAYER_FA;
    const int64_t nin = fa ? d.fa_qg + 2 * d.fa_kv : d.gdn_in;
    add_rms_bf16_kernel<<<(unsigned)P, kRowThreads, 0, s>>>(c->h, pending, pend_pc, D, d.eps, c->n);
    if ((st = launch_status(cudaSuccess)) != FAK_OK) return st;
    if ((st = fak_q4k_gemm(fa ? c->wqkv[l] : L.w_in, nin, D, c->n, P, c->T, s)) != FAK_OK) return st;
    slice_bf16_kernel<<<(unsigned)P, kRowThreads, 0, s>>>(c->T, nin, d.n_mix, c->X2);
    if ((st = launch_status(cudaSuccess)) != FAK_OK) return st;
    // the residual add + RMSNorm that follows sums the GEMM's stream-K pieces itself: no fix-up
    // kernel, no round trip of the cut tiles through Y
    FakGemmPieces pc{};
    if ((st = fak_q4k_gemm_pieces(L.w_out, D, d.n_mix, c->X2, P, c->Y, c->ws, c->ws_bytes, &pc, s)) != FAK_OK)
      return st;
    add_rms_bf16_kernel<<<(unsigned)P, kRowThreads, 0, s>>>(c->h, c->Y, pc, D, d.eps, c->n);
    if ((st = launch_status(cudaSuccess)) != FAK_OK) return st;
    if ((st = fak_q4k_gemm_swiglu(c->w13[l], F, D, c->n, P, c->X2, s)) != FAK_OK) return st;
    // the last layer's output goes to the all-rows add, which reads Y only
    pend_pc = FakGemmPieces{};
    if (l + 1 < d.n_layers)
      st = fak_q4k_gemm_pieces(L.w_down, D, F, c->X2, P, c->Y, c->ws, c->ws_bytes, &pend_pc, s);
    else
      st = fak_q4k_gemm(L.w_down, D, F, c->X2, P, c->Y, s);
    if (st != FAK_OK) return st;
    pending = c->Y;
  }
  if (pending) {
    add_rows_kernel<<<(unsigned)std::min<int64_t>(1024, (P * D / 4 + kRowThreads - 1) / kRowThreads), kRowThreads, 0,
                      s>>>(c->h, pending, P * D / 4);
    if ((st = launch_status(cudaSuccess)) != FAK_OK) return st;
  }
  last_rms_kernel<<<1, kRowThreads, 0, s>>>(c->h + (P - 1) * D, D, d.eps, c->nlast);
  if ((st = launch_status(cudaSuccess)) != FAK_OK) return st;
  if ((st = fak_q8_0_gemv(d.lm_head, d.vocab, D, c->nlast, c->logits, s)) != FAK_OK) return st;
  if ((st = fak_cuda_status(cudaMemsetAsync(c->slot, 0, sizeof(unsigned long long), s))) != FAK_OK) return st;
  argmax_kernel<<<(unsigned)c->sms, kRowThreads, 0, s>>>(c->logits, d.vocab, c->slot);
  if ((st = launch_status(cudaSuccess)) != FAK_OK) return st;
  argmax_finish_kernel<<<1, 1, 0, s>>>(c->slot, c->tok);
  return launch_status(cudaSuccess);
}

}  // namespace

extern "C" int fak_prefill_create(const fak_decode_desc* d, int64_t P, fak_prefill** out) {
  if (!d || !out || !d->layers || !d->lm_head || !d->embedding) return FAK_ERR_INVALID_ARG;
  *out = nullptr;
  if (d->mixer) return FAK_ERR_UNSUPPORTED;  // the prefill forward is the projections-only floor
  auto okdim = [](int64_t v) { return v >= 256 && v % 256 == 0 && v <= FAK_ENGINE_MAX_K; };
  if (P < 1 || P > 16384 || d->n_layers < 0 || !okdim(d->d_model) || d->d_model > 8192 || !okdim(d->d_ff) ||
      !okdim(d->n_mix) || d->vocab < 1 || d->gdn_in < 1 || d->fa_qg < 1 ||
      d->fa_kv < 1 || d->d_ff % 64 || d->n_mix % 256 || d->gdn_in % 4 || d->fa_qg % 4 || d->fa_kv % 2)
    return FAK_ERR_SHAPE;
  for (int l = 0; l < d->n_layers; ++l) {
    const fak_layer_desc& L = d->layers[l];
    if (L.kind != FAK_LAYER_GDN && L.kind != FAK_LAYER_FA) return FAK_ERR_INVALID_ARG;
    if (!L.w_in || !L.w_out || !L.w_gate || !L.w_up || !L.w_down) return FAK_ERR_INVALID_ARG;
    if (L.kind == FAK_LAYER_FA && (!L.w_k || !L.w_v)) return FAK_ERR_INVALID_ARG;
    if (d->n_mix > (L.kind == FAK_LAYER_GDN ? d->gdn_in : d->fa_qg)) return FAK_ERR_SHAPE;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FAK_ERR_CUDA;
  fak_prefill* c = new fak_prefill();
  cudaDeviceGetAttribute(&c->sms, cudaDevAttrMultiProcessorCount, dev);
  c->desc = *d;
  c->layers.assign(d->layers, d->layers + d->n_layers);
  c->desc.layers = c->layers.data();
  c->P = P;
  const int64_t D = d->d_model, F = d->d_ff, tn = std::max(d->gdn_in, d->fa_qg + 2 * d->fa_kv);
  const int64_t x2 = std::max<int64_t>(d->n_mix, F);
  bool ok = cudaMalloc(&c->toks, P * 4) == cudaSuccess && cudaMalloc(&c->h, P * D * 4) == cudaSuccess &&
            cudaMalloc(&c->n, P * D * 2) == cudaSuccess && cudaMalloc(&c->T, P * tn * 4) == cudaSuccess &&
            cudaMalloc(&c->X2, P * x2 * 2) == cudaSuccess &&
            cudaMalloc(&c->Y, P * D * 4) == cudaSuccess && cudaMalloc(&c->nlast, D * 4) == cudaSuccess &&
            cudaMalloc(&c->logits, (size_t)d->vocab * 4) == cudaSuccess &&
            cudaMalloc(&c->slot, sizeof(unsigned long long)) == cudaSuccess && cudaMalloc(&c->tok, 4) == cudaSuccess;
  c->ws_bytes = std::max(fak_gemm_pieces_bytes(D, d->n_mix, P), fak_gemm_pieces_bytes(D, F, P));
  if (ok && c->ws_bytes) ok = cudaMalloc(&c->ws, c->ws_bytes) == cudaSuccess;
  const size_t w13_bytes = (size_t)(2 * F) * (D / 256) * 144;
  const size_t row_bytes = (size_t)(D / 256) * 144;
  for (int l = 0; ok && l < d->n_layers; ++l) {
    uint8_t* w = nullptr;
    ok = cudaMalloc(&w, w13_bytes) == cudaSuccess;
    if (ok) c->w13.push_back(w);
    uint8_t* q = nullptr;
    if (ok && d->layers[l].kind == FAK_LAYER_FA)
      ok = cudaMalloc(&q, (size_t)(d->fa_qg + 2 * d->fa_kv) * row_bytes) == cudaSuccess;
    if (ok) c->wqkv.push_back(q);
  }
  if (!ok) {
    (void)cudaGetLastError();
    free_prefill(c);
    return FAK_ERR_NOMEM;
  }
  cudaStream_t s = nullptr;
  if (cudaStreamCreateWithFlags(&s, cudaStreamNonBlocking) != cudaSuccess) {
    free_prefill(c);
    return FAK_ERR_CUDA;
  }
  int st = FAK_OK;
  for (int l = 0; st == FAK_OK && l < d->n_layers; ++l) {
    st = fak_q4k_interleave_gate_up(c->layers[l].w_gate, c->layers[l].w_up, F, D, c->w13[l], s);
    if (st == FAK_OK && c->wqkv[l]) {
      // rows are contiguous Q4_K blocks: the concatenation is three plain copies
      const fak_layer_desc& L = c->layers[l];
      uint8_t* q = c->wqkv[l];
      const size_t bq = (size_t)d->fa_qg * row_bytes, bk = (size_t)d->fa_kv * row_bytes;
      cudaError_t e = cudaMemcpyAsync(q, L.w_in, bq, cudaMemcpyDeviceToDevice, s);
      if (e == cudaSuccess) e = cudaMemcpyAsync(q + bq, L.w_k, bk, cudaMemcpyDeviceToDevice, s);
      if (e == cudaSuccess) e = cudaMemcpyAsync(q + bq + bk, L.w_v, bk, cudaMemcpyDeviceToDevice, s);
      st = fak_cuda_status(e);
    }
  }
  if (st == FAK_OK) st = fak_cuda_status(cudaStreamSynchronize(s));
  // the forward recorded once into a graph: each prefill is then one submission
  if (st == FAK_OK) st = fak_cuda_status(cudaStreamBeginCapture(s, cudaStreamCaptureModeThreadLocal));
  if (st == FAK_OK) {
    const int rs = record_forward(c, s);
    const cudaError_t e = cudaStreamEndCapture(s, &c->graph);
    st = rs != FAK_OK ? rs : fak_cuda_status(e);
  }
  if (st == FAK_OK) st = fak_cuda_status(cudaGraphInstantiate(&c->exec, c->graph, 0));
  if (st == FAK_OK) {
    size_t nn = 0;
    cudaGraphGetNodes(c->graph, nullptr, &nn);
    std::vector<cudaGraphNode_t> nodes(nn);
    cudaGraphGetNodes(c->graph, nodes.data(), &nn);
    for (cudaGraphNode_t g : nodes) {
      cudaGraphNodeType t;
      if (cudaGraphNodeGetType(g, &t) == cudaSuccess && t == cudaGraphNodeTypeKernel) ++c->kernels;
    }
  }
  cudaStreamDestroy(s);
  if (st != FAK_OK) {
    free_prefill(c);
    return st;
  }
  *out = c;
  return FAK_OK;
}

extern "C" int fak_prefill_run(fak_prefill* c, const int32_t* d_tokens, int32_t* d_tok_out, float* d_logits,
                               fak_stream_t stream) {
  if (!c || !d_tokens || !d_tok_out) return FAK_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  int st = fak_cuda_status(cudaMemcpyAsync(c->toks, d_tokens, c->P * 4, cudaMemcpyDeviceToDevice, s));
  if (st == FAK_OK) st = fak_cuda_status(cudaGraphLaunch(c->exec, s));
  if (st == FAK_OK) st = fak_cuda_status(cudaMemcpyAsync(d_tok_out, c->tok, 4, cudaMemcpyDeviceToDevice, s));
  if (st == FAK_OK && d_logits)
    st = fak_cuda_status(
        cudaMemcpyAsync(d_logits, c->logits, (size_t)c->desc.vocab * 4, cudaMemcpyDeviceToDevice, s));
  return st;
}

extern "C" int fak_prefill_read_hidden(fak_prefill* c, float* dst, size_t count, fak_stream_t stream) {
  if (!c || !dst) return FAK_ERR_INVALID_ARG;
  if (count != (size_t)c->P * c->desc.d_model) return FAK_ERR_SHAPE;
  return fak_cuda_status(cudaMemcpyAsync(dst, c->h, count * 4, cudaMemcpyDefault, (cudaStream_t)stream));
}

extern "C" int fak_prefill_kernels(const fak_prefill* c) { return c ? (int)c->kernels : 0; }

extern "C" int fak_prefill_status(fak_prefill* c, fak_stream_t stream) {
  if (!c) return FAK_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return fak_cuda_status(e);
  int v = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&v, g_prefill_status, sizeof(int));
  if (e != cudaSuccess) return fak_cuda_status(e);
  cudaMemcpyToSymbol(g_prefill_status, &zero, sizeof(int));
  const int g = fak_gemm_take_status();
  return v != 0 ? v : g;
}

extern "C" void fak_prefill_destroy(fak_prefill* c) { free_prefill(c); }
