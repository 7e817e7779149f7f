// Batched Q4_K GEMV, Y[m, n] = sum_k W[n, k] * X[m, k] for up to 64 input
// rows, with W streamed from HBM once per call ("Mac Qwen3.6-27B Metal Q4_K
// perf diagnosis", section 3: GEMVBatch, many GEMVs on one resident weight).
//
// Arithmetic.  In super-block b of row n (256 weights; fp16 d, dmin; 6-bit
// sc_j, m_j per 32-weight sub-block j) each weight is
//     w = d * (sc_j * q) - dmin * m_j,
// and sc_j * q <= 63 * 15 = 945 is an integer that fp16 holds exactly.  Hence
//     sum_k w_k x_k = d * sum_k (sc_j q_k) x_k  -  dmin * sum_j m_j S_j
// with S_j the sum of x over sub-block j.  The first sum is a dense
// contraction whose weight operand is exact in fp16: the tensor core computes
// it per super-block into its own TMEM accumulator.  x enters as two fp16
// parts, x * 2^e = hi + lo, where e (per input row and super-block) puts
// max|x| in [2^14, 2^15); hi and lo are the MMA's N columns [0, MP) and
// [MP, 2 MP).  The epilogue adds d * 2^-e * (acc_hi + acc_lo) and subtracts
// dmin * sum_j m_j S_j (S_j summed in f64 by the split kernel, rounded once to
// f32) on the CUDA cores.  Relative error per product is about 2^-21.
//
// One CTA per (128-row tile, K split), 11 warps:
//   warp 0      TMA: W tile of one super-block, 128 rows x 144 bytes
//   warp 1      TMA: x parts of one super-block per ring slot, four 64-wide K
//               chunks of [hi; lo] (128-byte swizzle), plus S and 2^-e of the
//               super-block (bulk copies)
//   warps 2-9   dequant sc*q to fp16 straight into TMEM (the MMA's A operand;
//               thread = row, the two warps of a TMEM lane quadrant take one K
//               half each), then the epilogue of an earlier super-block (the
//               same two warps split the input rows)
//   warp 10     TMEM owner and MMA issuer: 16 x tcgen05.mma M128 N(2 MP) K16
//               per super-block, A from TMEM, B from shared memory
// TMEM: kNBuf A buffers (128 columns each) and as many accumulators, so
// dequant, MMA and epilogue of consecutive super-blocks overlap (three of each
// for up to 16 input rows, two above).  Every wait
// is bounded; on a timeout the kernel records FAK_ERR_TIMEOUT, lets what it
// issued land, frees TMEM and returns.
//
// A single input row (M = 1) goes to the matrix-vector engine instead
// (fak_q4k_gemv): the tensor core spends the same time per MMA whatever N is,
// so one row gains nothing from it.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "fak.h"
#include "fak_device.cuh"
#include "fak_tc.cuh"

namespace {

constexpr int kBM = 128;                 // weight rows per tile (MMA M)
constexpr int kWStages = 4;              // W super-block tiles in flight
constexpr int kWTileBytes = kBM * 144;   // 18432
constexpr int kSIStages = 8;             // S / 2^-e records in flight
constexpr int kBRingBytes = 131072;      // x-part ring
constexpr int kKParts = 2;                    // dequant warps per TMEM lane quadrant, each 256 / kKParts of K
constexpr int kDqWarps = 4 * kKParts;         // dequant + epilogue warps
constexpr int kMmaWarp = 2 + kDqWarps;        // TMEM owner and MMA issuer
constexpr int kThreadsB = 32 * (kMmaWarp + 1);
constexpr uint32_t kTmemColsB = 512;

template <int MP>
struct BCfg {
  static constexpr int kChunkBytes = 2 * MP * 128;  // one 64-wide K chunk of the [hi; lo] rows
  static constexpr int kSlotBytes = 4 * kChunkBytes;  // one super-block: one barrier, one commit
  static constexpr int kBStages = (kBRingBytes / kSlotBytes) > 32 ? 32 : (kBRingBytes / kSlotBytes);
  static constexpr int kSIBytes = 36 * MP;  // S [MP][8] f32, then 2^-e [MP] f32
  static constexpr int kOffB = 0;
  static constexpr int kOffW = kOffB + kBStages * kSlotBytes;
  static constexpr int kOffSI = kOffW + kWStages * kWTileBytes;
  static constexpr int kOffBar = kOffSI + kSIStages * kSIBytes;
  static constexpr int kSmem = kOffBar + 1024;
  static constexpr int kSmemAlloc = kSmem + 1024;
  static constexpr int kMq = MP / kKParts;  // input rows per epilogue warp
  // Super-blocks in flight between dequant, MMA and epilogue: kNBuf A buffers in TMEM (128
  // columns each) and as many accumulators (kAccW columns each, >= 2 MP); the epilogue runs
  // kNBuf - 1 super-blocks behind the dequant, so a super-block's MMAs have that long to finish.
  static constexpr int kNBuf = MP <= 16 ? 3 : 2;
  static constexpr int kLag = kNBuf - 1;
  static constexpr uint32_t kAccCol = 128u * kNBuf;
  static constexpr uint32_t kAccW = MP <= 16 ? 32u : 128u;
  static_assert(kAccCol + kNBuf * kAccW <= kTmemColsB && 2 * MP <= (int)kAccW, "TMEM columns");
  // kind::f16 instruction descriptor: D f32, A fp16, B fp16, both K-major, N = 2 MP, M = 128
  static constexpr uint32_t kIdesc = (1u << 4) | ((uint32_t)((2 * MP) >> 3) << 17) | ((uint32_t)(kBM >> 4) << 24);
  static_assert(kSmemAlloc <= 232448, "shared memory");
  static_assert(kChunkBytes % 1024 == 0, "swizzle atom alignment");
};

struct BgParams {
  float* Y;              // [M, N]
  float* partial;        // [splits, M, N] when splits > 1
  unsigned* counters;    // [tiles], zeroed by the split kernel
  const float* S;        // [nsb, MP, 8]
  const float* inv;      // [nsb, MP]
  int64_t N;
  int M, nsb, tiles, splits, sb_per_split;
  unsigned long long timeout_ns;
};

__device__ int g_bgemv_status;

// x[m, :] -> fp16 parts hi / lo of x * 2^e per 256-wide super-block, the
// sub-block sums S (f64, rounded once) and 2^-e.  One warp per (m, super-block);
// rows m in [M, MP) are written as zeros.
template <int MP>
__global__ void __launch_bounds__(256) bgemv_split_kernel(const float* __restrict__ X, int M, int64_t K, int nsb,
                                                          __half* __restrict__ Xs, float* __restrict__ S,
                                                          float* __restrict__ inv, unsigned* __restrict__ counters,
                                                          int ncounters) {
  pdl_launch_dependents();
  if (blockIdx.x == 0)
    for (int i = threadIdx.x; i < ncounters; i += blockDim.x) counters[i] = 0u;
  const int gw = (int)((blockIdx.x * (unsigned)blockDim.x + threadIdx.x) >> 5), lane = threadIdx.x & 31;
  if (gw >= MP * nsb) return;
  const int m = gw % MP, sb = gw / MP;
  const int64_t k0 = (int64_t)sb * 256 + 8 * lane;
  uint4 hi4 = make_uint4(0, 0, 0, 0), lo4 = make_uint4(0, 0, 0, 0);
  float s_out = 0.0f, inv_out = 0.0f;
  if (m < M) {
    const float4 a = *reinterpret_cast<const float4*>(X + (int64_t)m * K + k0);
    const float4 b = *reinterpret_cast<const float4*>(X + (int64_t)m * K + k0 + 4);
    const float v[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float amax = 0.0f;
#pragma unroll
    for (int t = 0; t < 8; ++t) amax = fmaxf(amax, fabsf(v[t]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    int e = 0;
    if (amax > 0.0f && amax <= 3.4028235e38f) {
      int E = 0;
      frexpf(amax, &E);  // amax = f * 2^E, f in [0.5, 1)
      e = 15 - E;
      if (e > 149) e = 149;
    }
    uint32_t hw[4], lw[4];
    double part = 0.0;
#pragma unroll
    for (int t = 0; t < 8; t += 2) {
      const float x0 = ldexpf(v[t], e), x1 = ldexpf(v[t + 1], e);
      const __half h0 = __float2half_rn(x0), h1 = __float2half_rn(x1);
      const __half l0 = __float2half_rn(x0 - __half2float(h0)), l1 = __float2half_rn(x1 - __half2float(h1));
      hw[t / 2] = (uint32_t)__half_as_ushort(h0) | ((uint32_t)__half_as_ushort(h1) << 16);
      lw[t / 2] = (uint32_t)__half_as_ushort(l0) | ((uint32_t)__half_as_ushort(l1) << 16);
      part += (double)v[t];
      part += (double)v[t + 1];
    }
    part += __shfl_xor_sync(0xffffffffu, part, 1);
    part += __shfl_xor_sync(0xffffffffu, part, 2);
    hi4 = make_uint4(hw[0], hw[1], hw[2], hw[3]);
    lo4 = make_uint4(lw[0], lw[1], lw[2], lw[3]);
    s_out = (float)part;
    inv_out = ldexpf(1.0f, -e);
  }
  *reinterpret_cast<uint4*>(Xs + (int64_t)m * K + k0) = hi4;
  *reinterpret_cast<uint4*>(Xs + (int64_t)(MP + m) * K + k0) = lo4;
  if ((lane & 3) == 0) S[((int64_t)sb * MP + m) * 8 + (lane >> 2)] = s_out;
  if (lane == 0) inv[(int64_t)sb * MP + m] = inv_out;
}

// sc * q for the 8 weights of one 32-bit word of nibbles, as four fp16 pairs:
// (1024 + q) is built from the nibble bits, and one fused fp16 multiply-add
// (1024 + q) * sc - 1024 * sc gives sc * q exactly.  lo[0..1] are the low
// nibbles of bytes (0,1), (2,3); hi[0..1] the high nibbles, taken in place as
// (1024 + 16 q) (no shift: 16 q sits in mantissa bits 4-7, and 1024 + 16 q <= 1264
// is exact) with mul_h = sc / 16 and add_h = -64 sc, both exact in fp16 for
// sc <= 63, so the single rounding again gives sc * q exactly.
FAK_DEV void scq_word(uint32_t v, uint32_t mul_l, uint32_t add_l, uint32_t mul_h, uint32_t add_h, uint32_t& lo0,
                      uint32_t& lo1, uint32_t& hi0, uint32_t& hi1) {
  const uint32_t t0 = prmt(v, 0u, 0x4140u), t1 = prmt(v, 0u, 0x4342u);
  lo0 = hfma2_bits(lop3_and_or(t0, 0x000F000Fu, 0x64006400u), mul_l, add_l);
  lo1 = hfma2_bits(lop3_and_or(t1, 0x000F000Fu, 0x64006400u), mul_l, add_l);
  hi0 = hfma2_bits(lop3_and_or(t0, 0x00F000F0u, 0x64006400u), mul_h, add_h);
  hi1 = hfma2_bits(lop3_and_or(t1, 0x00F000F0u, 0x64006400u), mul_h, add_h);
}

FAK_DEV uint32_t half2_splat(float f) {
  const uint32_t h = (uint32_t)__half_as_ushort(__float2half_rn(f));
  return h | (h << 16);
}

template <int MP>
__global__ void __launch_bounds__(kThreadsB, 1)
    bgemv_kernel(const __grid_constant__ CUtensorMap wmap, const __grid_constant__ CUtensorMap xmap,
                 const __grid_constant__ BgParams p) {
  using C = BCfg<MP>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* wfull = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* wempty = wfull + kWStages;
  uint64_t* bfull = wempty + kWStages;
  uint64_t* bempty = bfull + C::kBStages;
  uint64_t* sfull = bempty + C::kBStages;
  uint64_t* sempty = sfull + kSIStages;
  uint64_t* afull = sempty + kSIStages;
  // cfull[a]: the MMAs of the super-block in buffer pair a are done, so its
  // accumulator is ready for the epilogue and its A buffer free for the dequant
  uint64_t* cfull = afull + C::kNBuf;
  uint64_t* cempty = cfull + C::kNBuf;
  uint64_t* drain = cempty + C::kNBuf;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = reinterpret_cast<volatile int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tile = blockIdx.x % p.tiles, split = blockIdx.x / p.tiles;
  const int sb0 = split * p.sb_per_split;
  const int nloc = min(p.nsb, sb0 + p.sb_per_split) - sb0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kWStages; ++s) {
      mbar_init(&wfull[s], 1);
      mbar_init(&wempty[s], kDqWarps);
    }
    for (int s = 0; s < C::kBStages; ++s) {
      mbar_init(&bfull[s], 1);
      mbar_init(&bempty[s], 1);
    }
    for (int s = 0; s < kSIStages; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], kDqWarps);
    }
    for (int a = 0; a < C::kNBuf; ++a) {
      mbar_init(&afull[a], kDqWarps);
      mbar_init(&cfull[a], 1);
      mbar_init(&cempty[a], kDqWarps);
    }
    mbar_init(drain, 1);
    *abort = 0;
    *last_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&wmap);
    prefetch_tensormap(&xmap);
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemColsB)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const uint64_t tmo = p.timeout_ns;
  auto fail = [&]() {
    atomicCAS(&g_bgemv_status, 0, FAK_ERR_TIMEOUT);
    *abort = 1;
  };

  if (warp == 0) {
    // ---------------- W tiles (read once: evict first from L2)
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      int issued = 0;
      for (int i = 0; i < nloc && !*abort; ++i) {
        const int ws = i % kWStages;
        if (i >= kWStages && !mbar_wait_bounded(&wempty[ws], ((i / kWStages) - 1) & 1, abort, tmo)) {
          if (!*abort) fail();
          break;
        }
        mbar_arrive_expect_tx(&wfull[ws], kWTileBytes);
        tma_load_2d_tx_hint(smem + C::kOffW + ws * kWTileBytes, &wmap, (sb0 + i) * 144, tile * kBM, &wfull[ws], pol);
        issued = i + 1;
      }
      for (int i = issued - kWStages < 0 ? 0 : issued - kWStages; i < issued; ++i) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&wfull[i % kWStages], (i / kWStages) & 1))
          if (globaltimer_ns() - t0 > 200000000ull) break;
      }
    }
  } else if (warp == 1) {
    // ---------------- x parts, S and 2^-e (written by the split kernel just before)
    if (lane == 0) {
      pdl_wait();
      int issued_b = 0, issued_s = 0;
      for (int i = 0; i < nloc && !*abort; ++i) {
        const int sb = sb0 + i;
        bool ok = true;
        const int slot = i % C::kBStages;
        if (i >= C::kBStages && !mbar_wait_bounded(&bempty[slot], ((i / C::kBStages) - 1) & 1, abort, tmo)) ok = false;
        if (ok) {
          mbar_arrive_expect_tx(&bfull[slot], C::kSlotBytes);
          for (int c = 0; c < 4; ++c)
            tma_load_2d_tx(smem + C::kOffB + slot * C::kSlotBytes + c * C::kChunkBytes, &xmap, sb * 256 + 64 * c, 0,
                           &bfull[slot]);
          issued_b = i + 1;
        }
        const int s = i % kSIStages;
        if (ok && i >= kSIStages && !mbar_wait_bounded(&sempty[s], ((i / kSIStages) - 1) & 1, abort, tmo)) ok = false;
        if (!ok) {
          if (!*abort) fail();
          break;
        }
        mbar_arrive_expect_tx(&sfull[s], C::kSIBytes);
        uint8_t* dst = smem + C::kOffSI + s * C::kSIBytes;
        bulk_g2s_nohint(dst, p.S + (int64_t)sb * MP * 8, 32 * MP, &sfull[s]);
        bulk_g2s_nohint(dst + 32 * MP, p.inv + (int64_t)sb * MP, 4 * MP, &sfull[s]);
        issued_s = i + 1;
      }
      for (int q = issued_b - C::kBStages < 0 ? 0 : issued_b - C::kBStages; q < issued_b; ++q) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&bfull[q % C::kBStages], (q / C::kBStages) & 1))
          if (globaltimer_ns() - t0 > 200000000ull) break;
      }
      for (int q = issued_s - kSIStages < 0 ? 0 : issued_s - kSIStages; q < issued_s; ++q) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&sfull[q % kSIStages], (q / kSIStages) & 1))
          if (globaltimer_ns() - t0 > 200000000ull) break;
      }
    }
  } else if (warp == kMmaWarp) {
    // ---------------- MMA issuer
    if (lane == 0) {
      for (int i = 0; i < nloc && !*abort; ++i) {
        const int a = i % C::kNBuf, use = i / C::kNBuf;
        if (!mbar_wait_bounded(&afull[a], use & 1, abort, tmo) ||
            (use >= 1 && !mbar_wait_bounded(&cempty[a], (use - 1) & 1, abort, tmo))) {
          if (!*abort) fail();
          break;
        }
        tc_fence_after_sync();
        const uint32_t d_tmem = tmem + C::kAccCol + C::kAccW * (uint32_t)a;
        const uint32_t a_tmem = tmem + 128u * (uint32_t)a;
        const int slot = i % C::kBStages;
        const bool ok = mbar_wait_bounded(&bfull[slot], (i / C::kBStages) & 1, abort, tmo);
        if (ok) {
          tc_fence_after_sync();
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint64_t bdesc =
                umma_desc_sw128(smem_u32(smem + C::kOffB + slot * C::kSlotBytes + c * C::kChunkBytes));
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              umma_f16_ts(d_tmem, a_tmem + (uint32_t)(32 * c + 8 * kk), bdesc + (uint64_t)(2 * kk), C::kIdesc,
                          (c | kk) != 0);
          }
          umma_commit(&bempty[slot]);
        }
        if (!ok) {
          if (!*abort) fail();
          break;
        }
        umma_commit(&cfull[a]);
      }
      umma_commit(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0))
        if (globaltimer_ns() - t0 > 200000000ull) break;
    }
  } else {
    // ---------------- dequant into TMEM + epilogue
    const int mw = warp - 2;        // 0 .. kDqWarps - 1
    const int q = warp & 3;         // TMEM lanes 32q .. 32q+31 (fixed by the warp's rank)
    const int kp = mw >> 2;         // K part (dequant) and input-row part (epilogue) of this warp
    const int r = 32 * q + lane;    // row within the tile
    const int64_t n = (int64_t)tile * kBM + r;
    const uint32_t lane_base = (uint32_t)(32 * q) << 16;
    float y[C::kMq];
#pragma unroll
    for (int mm = 0; mm < C::kMq; ++mm) y[mm] = 0.0f;

    auto epilogue = [&](int j, uint4 hd) -> bool {
      const int a = j % C::kNBuf;
      if (!mbar_wait_bounded(&cfull[a], (j / C::kNBuf) & 1, abort, tmo)) return false;
      tc_fence_after_sync();
      uint32_t rh[C::kMq], rl[C::kMq];
      const uint32_t acc = tmem + lane_base + C::kAccCol + C::kAccW * (uint32_t)a;
      tmem_ld_cols<C::kMq>(acc + (uint32_t)(kp * C::kMq), rh);
      tmem_ld_cols<C::kMq>(acc + (uint32_t)(MP + kp * C::kMq), rl);
      tmem_wait_ld();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(&cempty[a]);
      const int s = j % kSIStages;
      if (!mbar_wait_bounded(&sfull[s], (j / kSIStages) & 1, abort, tmo)) return false;
      const float4* S4 = reinterpret_cast<const float4*>(smem + C::kOffSI + s * C::kSIBytes);
      const float* iv = reinterpret_cast<const float*>(smem + C::kOffSI + s * C::kSIBytes + 32 * MP);
      const float d = half_bits_to_float(hd.x & 0xFFFF), dmin = half_bits_to_float(hd.x >> 16);
      const uint32_t m_lo = hd.z & 0x3F3F3F3Fu;
      const uint32_t m_hi = ((hd.w >> 4) & 0x0F0F0F0Fu) | ((hd.z >> 2) & 0x30303030u);
      float mj[8];
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        mj[t] = (float)((m_lo >> (8 * t)) & 0xFF);
        mj[4 + t] = (float)((m_hi >> (8 * t)) & 0xFF);
      }
#pragma unroll
      for (int mm = 0; mm < C::kMq; ++mm) {
        const int m = kp * C::kMq + mm;
        const float4 s0 = S4[2 * m], s1 = S4[2 * m + 1];
        float ms = mj[0] * s0.x;
        ms = fmaf(mj[1], s0.y, ms);
        ms = fmaf(mj[2], s0.z, ms);
        ms = fmaf(mj[3], s0.w, ms);
        ms = fmaf(mj[4], s1.x, ms);
        ms = fmaf(mj[5], s1.y, ms);
        ms = fmaf(mj[6], s1.z, ms);
        ms = fmaf(mj[7], s1.w, ms);
        const float dot = __uint_as_float(rh[mm]) + __uint_as_float(rl[mm]);
        y[mm] = fmaf(d * iv[m], dot, y[mm]);
        y[mm] = fmaf(-dmin, ms, y[mm]);
      }
      // the record's loads are complete (consumed above, and the fence waits for them) before the
      // slot can be refilled by the next bulk copy
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      __syncwarp();
      if (lane == 0) mbar_arrive(&sempty[s]);
      return true;
    };

    // headers of the last kLag super-blocks (hq[k]: super-block i - 1 - k), for their epilogues
    uint4 hq[C::kLag];
#pragma unroll
    for (int k = 0; k < C::kLag; ++k) hq[k] = make_uint4(0, 0, 0, 0);
    bool ok = true;
    for (int i = 0; i < nloc && ok; ++i) {
      const int ws = i % kWStages;
      if (!mbar_wait_bounded(&wfull[ws], (i / kWStages) & 1, abort, tmo)) {
        ok = false;
        break;
      }
      const uint8_t* rowp = smem + C::kOffW + ws * kWTileBytes + r * 144;
      const uint4 hdr = *reinterpret_cast<const uint4*>(rowp);
      constexpr int kG = 4 / kKParts;  // 64-weight groups per warp: group g = sub-blocks 2g, 2g + 1
      uint4 qv[2 * kG];
#pragma unroll
      for (int c = 0; c < 2 * kG; ++c) qv[c] = *reinterpret_cast<const uint4*>(rowp + 16 + 32 * kG * kp + 16 * c);

      const int a = i % C::kNBuf, use = i / C::kNBuf;
      if (use >= 1 && !mbar_wait_bounded(&cfull[a], (use - 1) & 1, abort, tmo)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
#pragma unroll
      for (int gg = 0; gg < kG; ++gg) {
        const int g = kG * kp + gg;
        // 6-bit scales of sub-blocks 2g (low nibbles) and 2g + 1 (high nibbles): sub-blocks 0-3 in
        // the low 6 bits of header bytes 4-7, sub-blocks 4-7 from the low nibbles of bytes 12-15 and
        // the top 2 bits of bytes 4-7
        const uint32_t scw = g >= 2 ? ((hdr.w & 0x0F0F0F0Fu) | ((hdr.y >> 2) & 0x30303030u)) : (hdr.y & 0x3F3F3F3Fu);
        const int gi = g & 1;
        const float scl = (float)((scw >> (16 * gi)) & 0xFF), sch = (float)((scw >> (16 * gi + 8)) & 0xFF);
        const uint32_t mul_l = half2_splat(scl), add_l = half2_splat(-1024.0f * scl);
        const uint32_t mul_h = half2_splat(sch * 0.0625f), add_h = half2_splat(-64.0f * sch);
        const uint32_t wv[8] = {qv[2 * gg].x,     qv[2 * gg].y,     qv[2 * gg].z,     qv[2 * gg].w,
                                qv[2 * gg + 1].x, qv[2 * gg + 1].y, qv[2 * gg + 1].z, qv[2 * gg + 1].w};
        uint32_t out[32];
#pragma unroll
        for (int w = 0; w < 8; ++w)
          scq_word(wv[w], mul_l, add_l, mul_h, add_h, out[2 * w], out[2 * w + 1], out[16 + 2 * w],
                   out[16 + 2 * w + 1]);
        tmem_st32(tmem + lane_base + 128u * (uint32_t)a + (uint32_t)(32 * g), out);
      }
      tmem_wait_st();
      tc_fence_before_sync();
      __syncwarp();
      // the W slot is released only once its loads have fed the TMEM stores: an arrive right after
      // the loads let the slot's TMA refill land before loads still in flight (seen in the prefill
      // GEMM's per-step W ring)
      if (lane == 0) {
        mbar_arrive(&afull[a]);
        mbar_arrive(&wempty[ws]);
      }
      if (i >= C::kLag && !epilogue(i - C::kLag, hq[C::kLag - 1])) {
        ok = false;
        break;
      }
#pragma unroll
      for (int k = C::kLag - 1; k > 0; --k) hq[k] = hq[k - 1];
      hq[0] = hdr;
    }
    // the last kLag epilogues (hq[k] holds super-block nloc - 1 - k)
#pragma unroll
    for (int k = C::kLag - 1; k >= 0; --k) {
      const int j = nloc - 1 - k;
      if (ok && j >= 0 && !epilogue(j, hq[k])) ok = false;
    }
    if (!ok && !*abort) fail();

    // ---------------- output
    if (p.splits == 1) {
      if (n < p.N) {
#pragma unroll
        for (int mm = 0; mm < C::kMq; ++mm) {
          const int m = kp * C::kMq + mm;
          if (m < p.M) p.Y[(int64_t)m * p.N + n] = y[mm];
        }
      }
    } else {
      pdl_wait();
      float* part = p.partial + (int64_t)split * p.M * p.N;
      if (n < p.N) {
#pragma unroll
        for (int mm = 0; mm < C::kMq; ++mm) {
          const int m = kp * C::kMq + mm;
          if (m < p.M) part[(int64_t)m * p.N + n] = y[mm];
        }
      }
      __threadfence();
      named_bar_sync(1, 32 * kDqWarps);
      if (mw == 0 && lane == 0) {
        const unsigned prev = atomicAdd(&p.counters[tile], 1u);
        *last_flag = prev == (unsigned)(p.splits - 1) ? 1 : 0;
      }
      named_bar_sync(1, 32 * kDqWarps);
      if (*last_flag) {
        __threadfence();
        if (n < p.N) {
#pragma unroll 1
          for (int mm = 0; mm < C::kMq; ++mm) {
            const int m = kp * C::kMq + mm;
            if (m >= p.M) continue;
            float acc = 0.0f;
            for (int sp = 0; sp < p.splits; ++sp) acc += __ldcg(p.partial + ((int64_t)sp * p.M + m) * p.N + n);
            p.Y[(int64_t)m * p.N + n] = acc;
          }
        }
      }
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kMmaWarp) {
    __syncwarp();
    tc_fence_after_sync();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemColsB) : "memory");
  }
}

// ------------------------------------------------------------------ host side
std::mutex g_bg_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_bg_encode = nullptr;
bool g_bg_attr[64] = {};
int g_bg_sms[64] = {};

template <int MP>
cudaError_t set_attr() {
  return cudaFuncSetAttribute(bgemv_kernel<MP>, cudaFuncAttributeMaxDynamicSharedMemorySize, BCfg<MP>::kSmemAlloc);
}

int bg_setup(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fak_cuda_status(e);
  if (dev < 0 || dev >= 64) return FAK_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_bg_mu);
  if (!g_bg_attr[dev]) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (major != 10 || minor != 3) return FAK_ERR_UNSUPPORTED;
    cudaDeviceGetAttribute(&g_bg_sms[dev], cudaDevAttrMultiProcessorCount, dev);
    if (!g_bg_encode) {
      cudaDriverEntryPointQueryResult q;
      void* fn = nullptr;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return FAK_ERR_CUDA;
      g_bg_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cudaError_t es[4] = {set_attr<8>(), set_attr<16>(), set_attr<32>(), set_attr<64>()};
    for (cudaError_t x : es)
      if (x != cudaSuccess) return fak_cuda_status(x);
    g_bg_attr[dev] = true;
  }
  *sms = g_bg_sms[dev];
  return FAK_OK;
}

template <int MP>
int launch_bgemv(const uint8_t* W, int64_t N, int64_t K, const float* X, int M, float* Y, int sms, cudaStream_t s) {
  const int nsb = (int)(K / 256);
  const int tiles = (int)((N + kBM - 1) / kBM);
  int splits = 1, per = nsb;
  const int want = sms / tiles;
  if (want >= 2) {
    per = (nsb + want - 1) / want;
    splits = (nsb + per - 1) / per;
  }
  auto up = [](size_t b) { return (b + 255) & ~size_t(255); };
  const size_t b_xs = up((size_t)2 * MP * K * 2), b_s = up((size_t)nsb * MP * 32), b_inv = up((size_t)nsb * MP * 4);
  const size_t b_part = splits > 1 ? up((size_t)splits * M * N * 4) : 0, b_cnt = up((size_t)tiles * 4);
  void* buf = nullptr;
  cudaError_t e = fak_scratch_alloc(&buf, b_xs + b_s + b_inv + b_part + b_cnt, s);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return FAK_ERR_NOMEM;
  }
  uint8_t* base = static_cast<uint8_t*>(buf);
  __half* Xs = reinterpret_cast<__half*>(base);
  float* S = reinterpret_cast<float*>(base + b_xs);
  float* inv = reinterpret_cast<float*>(base + b_xs + b_s);
  float* part = splits > 1 ? reinterpret_cast<float*>(base + b_xs + b_s + b_inv) : nullptr;
  unsigned* cnt = reinterpret_cast<unsigned*>(base + b_xs + b_s + b_inv + b_part);

  CUtensorMap wmap, xmap;
  memset(&wmap, 0, sizeof(wmap));
  memset(&xmap, 0, sizeof(xmap));
  const cuuint64_t row_bytes = (cuuint64_t)nsb * 144;
  const cuuint64_t wdim[2] = {row_bytes, (cuuint64_t)N};
  const cuuint64_t wstride[1] = {row_bytes};
  const cuuint32_t wbox[2] = {144, kBM};
  const cuuint64_t xdim[2] = {(cuuint64_t)K, (cuuint64_t)(2 * MP)};
  const cuuint64_t xstride[1] = {(cuuint64_t)K * 2};
  const cuuint32_t xbox[2] = {64, 2 * MP};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r1 = g_bg_encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t*>(W), wdim, wstride, wbox,
                            estride, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  CUresult r2 = g_bg_encode(&xmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, Xs, xdim, xstride, xbox, estride,
                            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS) {
    cudaFreeAsync(buf, s);
    return FAK_ERR_CUDA;
  }

  const int warps = MP * nsb;
  bgemv_split_kernel<MP><<<(warps * 32 + 255) / 256, 256, 0, s>>>(X, M, K, nsb, Xs, S, inv, cnt, tiles);
  e = cudaGetLastError();
  if (e == cudaSuccess) {
    BgParams p;
    p.Y = Y;
    p.partial = part;
    p.counters = cnt;
    p.S = S;
    p.inv = inv;
    p.N = N;
    p.M = M;
    p.nsb = nsb;
    p.tiles = tiles;
    p.splits = splits;
    p.sb_per_split = per;
    p.timeout_ns = 2000000000ull;
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(tiles * splits);
    cfg.blockDim = dim3(kThreadsB);
    cfg.dynamicSmemBytes = BCfg<MP>::kSmemAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, bgemv_kernel<MP>, wmap, xmap, p);
  }
  cudaFreeAsync(buf, s);
  return fak_cuda_status(e);
}

}  // namespace

extern "C" int fak_q4k_gemv_batch(const void* Wq, int64_t N, int64_t K, const float* X, int M, float* Y,
                                  fak_stream_t stream) {
  if (!Wq || !X || !Y) return FAK_ERR_INVALID_ARG;
  if (M < 1 || M > 64 || N < 1 || N > 0x7fffffffLL || K < 256 || K % 256 != 0 || K > (1LL << 24))
    return FAK_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(Wq) & 15) || (reinterpret_cast<uintptr_t>(X) & 15) ||
      (reinterpret_cast<uintptr_t>(Y) & 3))
    return FAK_ERR_ALIGN;
  if (M == 1) return fak_q4k_gemv(Wq, N, K, X, Y, stream);
  int sms = 0;
  const int st = bg_setup(&sms);
  if (st != FAK_OK) return st;
  const uint8_t* W = static_cast<const uint8_t*>(Wq);
  cudaStream_t s = (cudaStream_t)stream;
  if (M <= 8) return launch_bgemv<8>(W, N, K, X, M, Y, sms, s);
  if (M <= 16) return launch_bgemv<16>(W, N, K, X, M, Y, sms, s);
  if (M <= 32) return launch_bgemv<32>(W, N, K, X, M, Y, sms, s);
  return launch_bgemv<64>(W, N, K, X, M, Y, sms, s);
}

int fak_bgemv_take_status() {
  int v = 0, zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&v, g_bgemv_status, sizeof(int));
  if (e != cudaSuccess) return fak_cuda_status(e);
  cudaMemcpyToSymbol(g_bgemv_status, &zero, sizeof(int));
  return v;
}
