// Device-side Q4_K / Q8_0 quantizers: the same covering min/max (Q4_K) and
// absmax (Q8_0) rules as the host packer, one thread per block, for loading
// a model whose f32 weights are already on the GPU.  Every f32 operation is
// written as an explicitly rounded intrinsic (no fused multiply-add
// contraction), so the bytes equal the host packer's bit for bit.
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "fak.h"
#include "fak_device.cuh"

namespace {

__device__ __forceinline__ uint16_t f16_ceil_dev(float v) {
  if (!(v > 0.0f)) return 0;
  if (v >= 65504.0f) return 0x7BFF;
  return __half_as_ushort(__float2half_ru(v));
}

__device__ __forceinline__ uint16_t f16_nearest_dev(float v) {
  uint16_t b = __half_as_ushort(__float2half_rn(v));
  if ((b & 0x7FFF) == 0x7C00) b = (uint16_t)((b & 0x8000) | 0x7BFF);
  return b;
}

__device__ __forceinline__ float f16_value_dev(uint16_t b) { return __half2float(__ushort_as_half(b)); }

__global__ void q4k_pack_kernel(const float* __restrict__ w, int64_t nblocks, int64_t blocks_per_row, int64_t K,
                                uint8_t* __restrict__ out) {
  for (int64_t blk = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; blk < nblocks;
       blk += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = blk / blocks_per_row, c = blk - n * blocks_per_row;
    const float* x = w + n * K + 256 * c;
    float neg[8], top[8];
    float worst_neg = 0.0f;
    for (int j = 0; j < 8; ++j) {
      float mn = 0.0f, mx = x[32 * j];
      for (int l = 0; l < 32; ++l) {
        const float v = x[32 * j + l];
        mn = fminf(mn, v);
        mx = fmaxf(mx, v);
      }
      neg[j] = -mn;
      top[j] = mx;
      worst_neg = fmaxf(worst_neg, neg[j]);
    }
    const uint16_t dmin_bits = f16_ceil_dev(__fdiv_rn(worst_neg, 63.0f));
    const float dmin = f16_value_dev(dmin_bits);
    int mins[8], scales[8];
    float reach[8], worst_reach = 0.0f;
    for (int j = 0; j < 8; ++j) {
      mins[j] = 0;
      if (dmin > 0.0f) mins[j] = min(63, (int)ceilf(__fdiv_rn(neg[j], dmin)));
      reach[j] = __fadd_rn(top[j], __fmul_rn(dmin, (float)mins[j]));
      worst_reach = fmaxf(worst_reach, reach[j]);
    }
    const uint16_t d_bits = f16_ceil_dev(__fdiv_rn(worst_reach, 945.0f));
    const float d = f16_value_dev(d_bits);
    const float d15 = __fmul_rn(15.0f, d);
    for (int j = 0; j < 8; ++j) scales[j] = d > 0.0f ? min(63, max(0, (int)ceilf(__fdiv_rn(reach[j], d15)))) : 0;

    uint8_t* o = out + blk * 144;
    uint8_t hdr[16];
    hdr[0] = (uint8_t)d_bits;
    hdr[1] = (uint8_t)(d_bits >> 8);
    hdr[2] = (uint8_t)dmin_bits;
    hdr[3] = (uint8_t)(dmin_bits >> 8);
    for (int i = 0; i < 4; ++i) {
      hdr[4 + i] = (uint8_t)((scales[i] & 63) | ((scales[i + 4] >> 4) << 6));
      hdr[8 + i] = (uint8_t)((mins[i] & 63) | ((mins[i + 4] >> 4) << 6));
      hdr[12 + i] = (uint8_t)((scales[i + 4] & 15) | ((mins[i + 4] & 15) << 4));
    }
    for (int i = 0; i < 16; ++i) o[i] = hdr[i];
    for (int g = 0; g < 4; ++g) {
      const int jl = 2 * g, jh = 2 * g + 1;
      const float lift_l = __fmul_rn(dmin, (float)mins[jl]), step_l = __fmul_rn(d, (float)scales[jl]);
      const float lift_h = __fmul_rn(dmin, (float)mins[jh]), step_h = __fmul_rn(d, (float)scales[jh]);
      for (int l = 0; l < 32; ++l) {
        int ql = 0, qh = 0;
        if (scales[jl] > 0)
          ql = min(15, max(0, (int)rintf(__fdiv_rn(__fadd_rn(x[32 * jl + l], lift_l), step_l))));
        if (scales[jh] > 0)
          qh = min(15, max(0, (int)rintf(__fdiv_rn(__fadd_rn(x[32 * jh + l], lift_h), step_h))));
        o[16 + 32 * g + l] = (uint8_t)(ql | (qh << 4));
      }
    }
  }
}

__global__ void q8_0_pack_kernel(const float* __restrict__ w, int64_t nblocks, int64_t blocks_per_row, int64_t K,
                                 uint8_t* __restrict__ out) {
  for (int64_t blk = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; blk < nblocks;
       blk += (int64_t)gridDim.x * blockDim.x) {
    const int64_t n = blk / blocks_per_row, c = blk - n * blocks_per_row;
    const float* x = w + n * K + 32 * c;
    float amax = 0.0f;
    for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(x[i]));
    const uint16_t d_bits = f16_nearest_dev(__fdiv_rn(amax, 127.0f));
    const float d = f16_value_dev(d_bits);
    uint8_t* o = out + blk * 34;
    o[0] = (uint8_t)d_bits;
    o[1] = (uint8_t)(d_bits >> 8);
    for (int i = 0; i < 32; ++i) {
      int q = 0;
      if (d > 0.0f) q = min(127, max(-127, (int)rintf(__fdiv_rn(x[i], d))));
      o[2 + i] = (uint8_t)(int8_t)q;
    }
  }
}

int launch_pack(bool q4, const float* w, int64_t N, int64_t K, void* out, size_t out_bytes, cudaStream_t s) {
  if (!w || !out) return FAK_ERR_INVALID_ARG;
  const int64_t bk = q4 ? 256 : 32, bb = q4 ? 144 : 34;
  if (N < 0 || K <= 0 || K % bk != 0) return FAK_ERR_SHAPE;
  const int64_t per_row = K / bk;
  if ((size_t)(N * per_row * bb) != out_bytes) return FAK_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(w) & 3)) return FAK_ERR_ALIGN;
  const int64_t nblocks = N * per_row;
  if (nblocks == 0) return FAK_OK;
  const int threads = 128;
  const int64_t want = (nblocks + threads - 1) / threads;
  const int grid = (int)(want < 65536 ? want : 65536);
  if (q4)
    q4k_pack_kernel<<<grid, threads, 0, s>>>(w, nblocks, per_row, K, static_cast<uint8_t*>(out));
  else
    q8_0_pack_kernel<<<grid, threads, 0, s>>>(w, nblocks, per_row, K, static_cast<uint8_t*>(out));
  return fak_cuda_status(cudaGetLastError());
}

}  // namespace

extern "C" int fak_q4k_pack_device(const float* w, int64_t N, int64_t K, void* out, size_t out_bytes,
                                   fak_stream_t stream) {
  return launch_pack(true, w, N, K, out, out_bytes, (cudaStream_t)stream);
}

extern "C" int fak_q8_0_pack_device(const float* w, int64_t N, int64_t K, void* out, size_t out_bytes,
                                    fak_stream_t stream) {
  return launch_pack(false, w, N, K, out, out_bytes, (cudaStream_t)stream);
}
