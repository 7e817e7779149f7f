// Prefill path: SwiGLU between the two prefill GEMMs (the tensor-core GEMM is
// added in this file next).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fak.h"
#include "fak_device.cuh"

namespace {
__global__ void swiglu_bf16_kernel(const float* __restrict__ Y1, int64_t P, int64_t half,
                                   __nv_bfloat16* __restrict__ X2) {
  const int64_t total = P * half;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t p = i / half, c = i - p * half;
    const float g = Y1[p * 2 * half + c], u = Y1[p * 2 * half + half + c];
    X2[i] = __float2bfloat16_rn(g / (1.0f + expf(-g)) * u);
  }
}
}  // namespace

extern "C" int fak_swiglu_bf16(const float* Y1, int64_t P, int64_t half, void* X2, fak_stream_t stream) {
  if (!Y1 || !X2) return FAK_ERR_INVALID_ARG;
  if (P < 1 || half < 1) return FAK_ERR_SHAPE;
  const int64_t total = P * half;
  const int grid = (int)((total + 255) / 256 < 152 * 16 ? (total + 255) / 256 : 152 * 16);
  swiglu_bf16_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(Y1, P, half, static_cast<__nv_bfloat16*>(X2));
  return fak_cuda_status(cudaGetLastError());
}

extern "C" int fak_q4k_gemm(const void* Wq, int64_t N, int64_t K, const void* X, int64_t P, float* Y,
                            fak_stream_t stream) {
  if (!Wq || !X || !Y) return FAK_ERR_INVALID_ARG;
  if (K < 256 || K % 256 || N < 128 || N % 128 || P < 1) return FAK_ERR_SHAPE;
  (void)stream;
  return FAK_ERR_UNSUPPORTED;
}
