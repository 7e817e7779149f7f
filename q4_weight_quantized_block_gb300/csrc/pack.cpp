// Host-side Q4_K and Q8_0 quantizers (the library's own packer).
//
// The pages keep raw q4_k blocks resident and name the format only ("Mac
// Qwen3.6-27B Metal Q4_K perf diagnosis", TL;DR; "Qwen3.6-27B on Apple M3 Pro",
// reconciliation table, resident-q4k row); the quantizer is the covering
// min/max rule stated in include/fak.h.  Compiled with -ffp-contract=off: every
// f32 expression below is a sequence of individually rounded IEEE operations,
// so the bytes are the same on every host.  binary16 rounding uses the CUDA
// host-side conversions (round-up for d/dmin, round-to-nearest-even for Q8_0).
#include <cuda_fp16.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "fak.h"

namespace {

inline uint16_t half_bits(__half h) { return __half_as_ushort(h); }

// smallest binary16 >= v (v >= 0), saturating at the largest finite value
inline uint16_t f16_ceil(float v) {
  if (!(v > 0.0f)) return 0;
  if (v >= 65504.0f) return 0x7BFF;
  return half_bits(__float2half_ru(v));
}

inline uint16_t f16_nearest(float v) {
  __half h = __float2half_rn(v);
  uint16_t b = half_bits(h);
  if ((b & 0x7FFF) == 0x7C00) b = (uint16_t)((b & 0x8000) | 0x7BFF);
  return b;
}

inline float f16_value(uint16_t b) { return __half2float(__ushort_as_half(b)); }

struct SubRange {
  float neg_min;  // -min(0, min x) >= 0
  float top;      // max x
};

void quantize_q4k_block(const float* __restrict x, uint8_t* __restrict blk) {
  SubRange sr[8];
  float worst_neg = 0.0f;
  for (int j = 0; j < 8; ++j) {
    const float* s = x + 32 * j;
    float mn = std::min(0.0f, *std::min_element(s, s + 32));
    float mx = *std::max_element(s, s + 32);
    sr[j].neg_min = -mn;
    sr[j].top = mx;
    worst_neg = std::max(worst_neg, sr[j].neg_min);
  }
  const uint16_t dmin_bits = f16_ceil(worst_neg / 63.0f);
  const float dmin = f16_value(dmin_bits);

  int mins[8], scales[8];
  float reach[8], worst_reach = 0.0f;
  for (int j = 0; j < 8; ++j) {
    mins[j] = 0;
    if (dmin > 0.0f) mins[j] = std::min(63, (int)std::ceil(sr[j].neg_min / dmin));
    const float lift = dmin * (float)mins[j];
    reach[j] = sr[j].top + lift;
    worst_reach = std::max(worst_reach, reach[j]);
  }
  const uint16_t d_bits = f16_ceil(worst_reach / 945.0f);
  const float d = f16_value(d_bits);
  const float d15 = 15.0f * d;
  for (int j = 0; j < 8; ++j) {
    int sc = 0;
    if (d > 0.0f) sc = std::min(63, std::max(0, (int)std::ceil(reach[j] / d15)));
    scales[j] = sc;
  }

  std::memset(blk, 0, 144);
  blk[0] = (uint8_t)d_bits;
  blk[1] = (uint8_t)(d_bits >> 8);
  blk[2] = (uint8_t)dmin_bits;
  blk[3] = (uint8_t)(dmin_bits >> 8);
  uint8_t* s = blk + 4;
  for (int j = 0; j < 8; ++j) {
    if (j < 4) {
      s[j] |= (uint8_t)(scales[j] & 63);
      s[j + 4] |= (uint8_t)(mins[j] & 63);
    } else {
      const int i = j - 4;
      s[i] |= (uint8_t)((scales[j] >> 4) << 6);
      s[i + 4] |= (uint8_t)((mins[j] >> 4) << 6);
      s[i + 8] |= (uint8_t)((scales[j] & 15) | ((mins[j] & 15) << 4));
    }
  }

  uint8_t* qs = blk + 16;
  for (int j = 0; j < 8; ++j) {
    const float lift = dmin * (float)mins[j];
    const float step = d * (float)scales[j];
    const int g = j >> 1;
    const int shift = (j & 1) ? 4 : 0;
    for (int l = 0; l < 32; ++l) {
      int q = 0;
      if (scales[j] > 0) {
        q = (int)std::nearbyint((x[32 * j + l] + lift) / step);
        q = std::min(15, std::max(0, q));
      }
      qs[32 * g + l] |= (uint8_t)(q << shift);
    }
  }
}

void quantize_q8_0_block(const float* __restrict x, uint8_t* __restrict blk) {
  float amax = 0.0f;
  for (int i = 0; i < 32; ++i) amax = std::max(amax, std::fabs(x[i]));
  const uint16_t d_bits = f16_nearest(amax / 127.0f);
  const float d = f16_value(d_bits);
  blk[0] = (uint8_t)d_bits;
  blk[1] = (uint8_t)(d_bits >> 8);
  for (int i = 0; i < 32; ++i) {
    int q = 0;
    if (d > 0.0f) q = std::min(127, std::max(-127, (int)std::nearbyint(x[i] / d)));
    blk[2 + i] = (uint8_t)(int8_t)q;
  }
}

template <typename F>
void parallel_rows(int64_t rows, F&& body) {
  unsigned hw = std::thread::hardware_concurrency();
  int64_t nt = std::max<int64_t>(1, std::min<int64_t>(hw ? hw : 1, rows / 4 + 1));
  if (nt <= 1) {
    body(0, rows);
    return;
  }
  std::vector<std::thread> pool;
  pool.reserve((size_t)nt);
  for (int64_t t = 0; t < nt; ++t) {
    int64_t a = rows * t / nt, b = rows * (t + 1) / nt;
    pool.emplace_back([&body, a, b] { body(a, b); });
  }
  for (auto& th : pool) th.join();
}

}  // namespace

extern "C" int fak_q4k_pack(const float* w, int64_t N, int64_t K, void* out, size_t out_bytes) {
  if (!w || !out) return FAK_ERR_INVALID_ARG;
  if (N < 0 || K <= 0 || K % 256 != 0) return FAK_ERR_SHAPE;
  const int64_t per_row = K / 256 * 144;
  if ((size_t)(N * per_row) != out_bytes) return FAK_ERR_SHAPE;
  uint8_t* dst = static_cast<uint8_t*>(out);
  parallel_rows(N, [&](int64_t a, int64_t b) {
    for (int64_t n = a; n < b; ++n)
      for (int64_t c = 0; c < K / 256; ++c)
        quantize_q4k_block(w + n * K + 256 * c, dst + n * per_row + 144 * c);
  });
  return FAK_OK;
}

extern "C" int fak_q8_0_pack(const float* w, int64_t N, int64_t K, void* out, size_t out_bytes) {
  if (!w || !out) return FAK_ERR_INVALID_ARG;
  if (N < 0 || K <= 0 || K % 32 != 0) return FAK_ERR_SHAPE;
  const int64_t per_row = K / 32 * 34;
  if ((size_t)(N * per_row) != out_bytes) return FAK_ERR_SHAPE;
  uint8_t* dst = static_cast<uint8_t*>(out);
  parallel_rows(N, [&](int64_t a, int64_t b) {
    for (int64_t n = a; n < b; ++n)
      for (int64_t c = 0; c < K / 32; ++c) quantize_q8_0_block(w + n * K + 32 * c, dst + n * per_row + 34 * c);
  });
  return FAK_OK;
}
