// Prefill dequant-GEMM on the 5th-generation tensor cores (tcgen05 / TMEM),
// plus the SwiGLU between the two prefill GEMMs.
//
// Y[P, N] = X[P, K] * W[N, K]^T with W in Q4_K and X in bf16, f32 accumulate
// ("Mac Qwen3.6-27B Metal Q4_K perf diagnosis", section 2: mlp_gate_up_proj and
// mlp_down_proj take 73% of prefill; section 4b: the q4k_gemm prefill kernel).
//
// One CTA per SM, persistent over output tiles of 128 weight rows x 256 tokens,
// K in steps of 64 through a 4-stage shared-memory pipeline:
//   warp 0      TMA producer: X tile [256 tokens x 64] bf16, 128-byte swizzle
//   warp 1      TMEM owner + MMA issuer: 4 x tcgen05.mma (M128 N256 K16) per stage
//   warps 2-5   dequant producers of the even K steps, warps 11-14 of the odd ones:
//   and 11-14   128 W rows x 64 weights -> bf16, written in the same 128-byte-swizzled
//               K-major layout (one thread per row, reading its row's Q4_K header and
//               quants from the W ring in shared memory); two producer warps per
//               scheduler, so one's waits and hand-offs hide under the other's arithmetic
//   warps 6-9   epilogue: tcgen05.ld of the f32 accumulator -> Y (coalesced)
//   warp 10     TMA producer (W): per super-block the 128 rows' 16-byte block headers
//               into a two-slot ring, per K step the rows' 32 quant bytes of the step
//               into a six-slot ring (an even count: a slot always serves the same
//               producer warps, which wait on each of its phases in order)
// Two TMEM accumulators (2 x 256 columns) let the epilogue of one tile overlap
// the MMAs of the next.  Every wait is bounded; on a timeout the kernel records
// FAK_ERR_TIMEOUT, drains what it issued, frees TMEM and returns.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fak.h"
#include "fak_device.cuh"

namespace {

constexpr int BM = 128;  // weight rows per tile (MMA M)
constexpr int BN = 256;  // tokens per tile (MMA N)
constexpr int BK = 64;   // K per stage (one 128-byte swizzle atom of bf16)
constexpr int kStagesG = 4;
constexpr int kThreadsG = 480;
constexpr double kStreamKFixCost = 3.0;  // stream-K's extra cost, in super-block steps of one tile
constexpr int kWSlots = 6;                // quant slots in flight (one per K step; even)
constexpr int kWTile = 128 * 32;          // 128 rows x the step's 32 quant bytes
constexpr int kHSlots = 2;                // header slots (one per super-block)
constexpr int kHTile = 128 * 16;          // 128 rows x 16-byte block header
constexpr int kABytes = BM * BK * 2;  // 16 KB
constexpr int kBBytes = BN * BK * 2;  // 32 KB
constexpr int kOffA = 0;
constexpr int kOffB = kOffA + kStagesG * kABytes;
constexpr int kOffW = kOffB + kStagesG * kBBytes;
constexpr int kOffH = kOffW + kWSlots * kWTile;
constexpr int kOffBarG = kOffH + kHSlots * kHTile;
constexpr int kSmemG = kOffBarG + 512;
constexpr int kSmemAllocG = kSmemG + 1024;
constexpr uint32_t kTmemCols = 512;
static_assert(kSmemAllocG <= 232448, "GEMM shared memory exceeds the 227 KB per-block limit");
static_assert((2 * kStagesG + 5 + 2 * kWSlots + 2 * kHSlots) * 8 + 8 <= 512, "GEMM barriers exceed their area");
static_assert(kWSlots % 2 == 0 && kStagesG % 2 == 0, "each ring slot must serve one parity of K steps");

__device__ int g_gemm_status;

FAK_DEV void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
FAK_DEV void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

FAK_DEV uint64_t sw128_desc(uint32_t smem_addr) {
  // K-major, 128-byte swizzle: 8-row core groups 1024 bytes apart (SBO), LBO unused (1).
  uint64_t d = 0;
  d |= (uint64_t)((smem_addr >> 4) & 0x3FFF);
  d |= (uint64_t)1 << 16;
  d |= (uint64_t)(1024 >> 4) << 32;
  d |= (uint64_t)1 << 46;  // descriptor version for the 5th-generation tensor core
  d |= (uint64_t)2 << 61;  // SWIZZLE_128B
  return d;
}

// kind::f16 instruction descriptor: D f32, A bf16, B bf16, both K-major, N=BN, M=BM.
constexpr uint32_t kIdesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(BN >> 3) << 17) | ((uint32_t)(BM >> 4) << 24);

FAK_DEV void mma_bf16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(tmem_d),
      "l"(adesc), "l"(bdesc), "r"(kIdesc), "r"(accumulate)
      : "memory");
}

FAK_DEV void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

FAK_DEV void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
          smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
      : "memory");
}

FAK_DEV void tma_load_2d_hint(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1, {%2, "
      "%3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(pol)
      : "memory");
}

FAK_DEV void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%"
      "20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]),
        "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
        "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
        "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

struct GemmParams {
  const uint8_t* W;
  float* Y;
  int64_t N, K, P;
  int n_tiles_n, n_tiles_p;
  // whole tiles: unit u is tile u / splits over super-blocks [sb_per * (u % splits), +sb_per)
  // (the host sets splits = 1, sb_per = K / 256)
  int splits, sb_per;
  // stream-K (stream != 0, splits == 1): the super-blocks of all tiles' K ranges laid end to end
  // (tile-major, nsb per tile) are cut into gridDim.x equal contiguous ranges, one per CTA; each
  // piece of a tile met by several CTAs goes to ws ([tile][maxp][BN tokens][128 rows] f32, a
  // column of the tile contiguous) and streamk_fixup_kernel, launched next, sums them in K order
  int stream, nsb, maxp;
  // SwiGLU epilogue (fak_q4k_gemm_swiglu; splits == 1): W's rows are gate and up
  // channels interleaved by 16 (see there); the epilogue writes
  // x2[p, c] = bf16(silu(gate) * up) instead of Y
  __nv_bfloat16* x2;
  int64_t F;
  float* ws;
  unsigned long long timeout_ns;
};

// One CTA's work as a sequence of segments: a K range [k0, k1) (in 64-wide steps) of one tile,
// piece `piece` of the `npieces` pieces the tile's K range is cut into.
struct Seg {
  int tile, k0, k1, piece, npieces;
};
struct SegIter {
  int64_t pos, end;  // stream-K: this CTA's super-block range
  int u;             // units: the next unit (tile * splits + split)
};

FAK_DEV void seg_begin(const GemmParams& p, SegIter& it) {
  const int64_t W = (int64_t)p.n_tiles_n * p.n_tiles_p * p.nsb, G = gridDim.x, c = blockIdx.x;
  it.pos = W * c / G;
  it.end = W * (c + 1) / G;
  it.u = blockIdx.x;
}

FAK_DEV bool seg_next(const GemmParams& p, SegIter& it, Seg& sg) {
  if (p.stream) {
    if (it.pos >= it.end) return false;
    const int64_t W = (int64_t)p.n_tiles_n * p.n_tiles_p * p.nsb, G = gridDim.x;
    const int tile = (int)(it.pos / p.nsb);
    const int64_t tb = (int64_t)tile * p.nsb, te = tb + p.nsb;
    const int64_t se = it.end < te ? it.end : te;
    sg.tile = tile;
    sg.k0 = 4 * (int)(it.pos - tb);
    sg.k1 = 4 * (int)(se - tb);
    // CTA c's range starts at floor(c W / G): the CTAs that meet the tile are those holding its
    // first and its last super-block and all between (every range is non-empty: the host
    // launches G <= W CTAs)
    const int64_t cf = ((tb + 1) * G + W - 1) / W - 1, cl = (te * G + W - 1) / W - 1;
    sg.piece = (int)(blockIdx.x - cf);
    sg.npieces = (int)(cl - cf + 1);
    it.pos = se;
    return true;
  }
  const int total = p.n_tiles_n * p.n_tiles_p * p.splits;
  if (it.u >= total) return false;
  const int sp = it.u % p.splits;
  sg.tile = it.u / p.splits;
  sg.k0 = 4 * sp * p.sb_per;
  sg.k1 = min((int)(p.K / BK), sg.k0 + 4 * p.sb_per);
  sg.piece = sp;
  sg.npieces = p.splits;
  it.u += gridDim.x;
  return true;
}

// Dequantize the 64 weights of one row for K step g (0..3 within a super-block):
// low nibbles of qs[32g..32g+31] are k 0..31 (sub-block 2g), high nibbles k 32..63
// (sub-block 2g+1).  w = d*sc*q - dmin*m, rounded once to bf16.
// `h` is the row's 16-byte block header, q0 / q1 the 32 quant bytes of step g.
FAK_DEV void dequant_row_step(const uint4 h, const uint4 q0, const uint4 q1, int g, uint8_t* row_smem, int r8) {
  const uint32_t sc_lo = h.y & 0x3F3F3F3Fu, m_lo = h.z & 0x3F3F3F3Fu;
  const uint32_t sc_hi = (h.w & 0x0F0F0F0Fu) | ((h.y >> 2) & 0x30303030u);
  const uint32_t m_hi = ((h.w >> 4) & 0x0F0F0F0Fu) | ((h.z >> 2) & 0x30303030u);
  const uint32_t sel = (uint32_t)(2 * g) | ((uint32_t)(2 * g + 1) << 4);
  const uint32_t scp = prmt(sc_lo, sc_hi, sel), mp = prmt(m_lo, m_hi, sel);
  const float d = half_bits_to_float(h.x & 0xFFFF), dmin = half_bits_to_float(h.x >> 16);
  // w = a*q - b = (32a)*(0.5 + q/32) - (16a + b), with 0.5 + q/32 built exactly from the nibble bits
  float mul[2], add[2];
#pragma unroll
  for (int hsel = 0; hsel < 2; ++hsel) {
    const float a = d * (float)((scp >> (8 * hsel)) & 0xFF);
    const float b = dmin * (float)((mp >> (8 * hsel)) & 0xFF);
    mul[hsel] = 32.0f * a;
    add[hsel] = -(16.0f * a + b);
  }
  const uint32_t qw[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
#pragma unroll
  for (int hsel = 0; hsel < 2; ++hsel) {
#pragma unroll
    for (int c4 = 0; c4 < 4; ++c4) {  // 16-byte chunk (8 weights) c = 4*hsel + c4
      uint32_t packed[4];
#pragma unroll
      for (int wi = 0; wi < 2; ++wi) {
        const uint32_t wsrc = qw[2 * c4 + wi];
        const uint32_t t = hsel == 0 ? ((wsrc << 3) & 0x78787878u) : ((wsrc >> 1) & 0x78787878u);
        float f[4];
#pragma unroll
        for (int bi = 0; bi < 4; ++bi) {
          const uint32_t bits = prmt(t, 0x3F000000u, 0x7044u | ((uint32_t)bi << 8));
          f[bi] = fmaf(mul[hsel], __uint_as_float(bits), add[hsel]);
        }
        __nv_bfloat162 p0 = __floats2bfloat162_rn(f[0], f[1]);
        __nv_bfloat162 p1 = __floats2bfloat162_rn(f[2], f[3]);
        packed[2 * wi] = *reinterpret_cast<uint32_t*>(&p0);
        packed[2 * wi + 1] = *reinterpret_cast<uint32_t*>(&p1);
      }
      const int c = 4 * hsel + c4;
      *reinterpret_cast<uint4*>(row_smem + ((c ^ r8) << 4)) = make_uint4(packed[0], packed[1], packed[2], packed[3]);
    }
  }
}

// silu(g) * u; the one expression both SwiGLU paths use, so they agree bit for bit
FAK_DEV float silu_mul(float g, float u) { return g / (1.0f + expf(-g)) * u; }

__global__ void __launch_bounds__(kThreadsG, 1)
    q4k_gemm_kernel(const __grid_constant__ CUtensorMap xmap, const __grid_constant__ CUtensorMap wmap,
                    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ GemmParams p) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  // full[s]: stage s holds its X tile (TMA bytes) and its dequantized A tile (four warp arrivals)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kOffBarG);
  uint64_t* empty = full + kStagesG;
  uint64_t* tfull = empty + kStagesG;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* wfull = drain + 1;
  uint64_t* wempty = wfull + kWSlots;
  uint64_t* hfull = wempty + kWSlots;
  uint64_t* hempty = hfull + kHSlots;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(hempty + kHSlots);
  volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesG; ++s) {
      mbar_init(&full[s], 5);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], 4);
    }
    mbar_init(drain, 1);
    for (int w = 0; w < kWSlots; ++w) {
      mbar_init(&wfull[w], 1);
      mbar_init(&wempty[w], 4);  // the four producer warps of the slot's K-step parity
    }
    for (int h = 0; h < kHSlots; ++h) {
      mbar_init(&hfull[h], 1);
      mbar_init(&hempty[h], 8);  // all eight producer warps
    }
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // the stream-K fix-up (launched with programmatic serialization) may be scheduled from now on;
  // it waits for this grid's completion itself
  if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  const uint64_t tmo = p.timeout_ns;
  auto fail = [&]() {
    atomicCAS(&g_gemm_status, 0, FAK_ERR_TIMEOUT);
    *abort = 1;
  };

  if (warp == 0) {
    // ---------------- TMA producer (X)
    if (lane == 0) {
      int it = 0;
      SegIter si;
      Seg sg;
      seg_begin(p, si);
      while (!*abort && seg_next(p, si, sg)) {
        const int p0 = (sg.tile % p.n_tiles_p) * BN;
        for (int kt = sg.k0; kt < sg.k1; ++kt, ++it) {
          const int s = it % kStagesG;
          if (it >= kStagesG && !mbar_wait_bounded(&empty[s], ((it / kStagesG) - 1) & 1, abort, tmo)) {
            if (!*abort) fail();
            break;
          }
          mbar_arrive_expect_tx(&full[s], kBBytes);
          tma_load_2d(smem + kOffB + s * kBBytes, &xmap, kt * BK, p0, &full[s]);
        }
      }
      // let in-flight copies land before the CTA can exit (a stage's phase also takes the dequant
      // warps' arrivals, which come in every run that did not abort; an abort waits out the bound)
      const int last = it;
      for (int q = last - kStagesG < 0 ? 0 : last - kStagesG; q < last; ++q) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&full[q % kStagesG], (q / kStagesG) & 1))
          if (globaltimer_ns() - t0 > 200000000ull) break;
      }
    }
  } else if (warp == 1) {
    // ---------------- MMA issuer
    if (lane == 0) {
      // stage s's descriptors are stage 0's plus its offset (in 16-byte units; no carry out of the
      // 14-bit address field, which holds the whole 227 KB)
      const uint64_t ad0 = sw128_desc(smem_u32(smem + kOffA)), bd0 = sw128_desc(smem_u32(smem + kOffB));
      int it = 0, local = 0;
      SegIter si;
      Seg sg;
      seg_begin(p, si);
      for (; !*abort && seg_next(p, si, sg); ++local) {
        const int acc = local & 1;
        const int k0 = sg.k0, k1 = sg.k1;
        if (local >= 2 && !mbar_wait_bounded(&tempty[acc], ((local >> 1) - 1) & 1, abort, tmo)) {
          if (!*abort) fail();
          break;
        }
        tc_fence_after();
        const uint32_t dcol = tmem + (uint32_t)(acc * BN);
        bool ok = true;
        for (int kt = k0; kt < k1; ++kt, ++it) {
          const int s = it % kStagesG;
          const uint32_t ph = (it / kStagesG) & 1;
          if (!mbar_wait_bounded(&full[s], ph, abort, tmo)) {
            if (!*abort) fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = ad0 + (uint64_t)((s * kABytes) >> 4);
          const uint64_t bd = bd0 + (uint64_t)((s * kBBytes) >> 4);
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            mma_bf16(dcol, ad + (uint64_t)(2 * kk), bd + (uint64_t)(2 * kk), (kt != k0) || (kk != 0));
          mma_commit(&empty[s]);
        }
        if (!ok) break;
        mma_commit(&tfull[acc]);
      }
      // all issued MMAs complete before TMEM can be freed
      mma_commit(drain);
      const uint64_t t0 = globaltimer_ns();
      while (!mbar_try_wait(drain, 0))
        if (globaltimer_ns() - t0 > 200000000ull) break;
    }
  } else if (warp < 6 || warp >= 11) {
    // ---------------- dequant producers: thread t owns row t of each W tile; warps 2-5 take
    // the even K steps (it counts the CTA's K steps), warps 11-14 the odd ones
    const int par = warp >= 11 ? 1 : 0;
    const int t = (warp - (par ? 11 : 2)) * 32 + lane;
    const int r8 = t & 7;
    int it = 0;
    bool ok = true;
    SegIter si;
    Seg sg;
    seg_begin(p, si);
    while (ok && !*abort && seg_next(p, si, sg)) {
      uint4 hdr = make_uint4(0, 0, 0, 0);
      for (int kt = sg.k0; kt < sg.k1 && ok; ++kt, ++it) {
        if ((it & 1) != par) continue;
        const int g = kt & 3;  // segments hold whole super-blocks, so it and kt agree mod 4
        if (g == par) {
          // the warp's first step of the super-block (the CTA's (it / 4)-th): its rows' headers
          const int hu = it >> 2, h = hu % kHSlots;
          if (!mbar_wait_bounded(&hfull[h], (hu / kHSlots) & 1, abort, tmo)) {
            if (!*abort) fail();
            ok = false;
            break;
          }
          hdr = *reinterpret_cast<const uint4*>(smem + kOffH + h * kHTile + t * 16);
        }
        const int w = it % kWSlots;  // the quant ring advances one slot per K step, like the stages
        if (!mbar_wait_bounded(&wfull[w], (it / kWSlots) & 1, abort, tmo)) {
          if (!*abort) fail();
          ok = false;
          break;
        }
        const uint8_t* slot = smem + kOffW + w * kWTile;
        const uint4 q0 = *reinterpret_cast<const uint4*>(slot + t * 32);
        const uint4 q1 = *reinterpret_cast<const uint4*>(slot + t * 32 + 16);
        const int s = it % kStagesG;
        if (it >= kStagesG && !mbar_wait_bounded(&empty[s], ((it / kStagesG) - 1) & 1, abort, tmo)) {
          if (!*abort) fail();
          ok = false;
          break;
        }
        uint8_t* row_smem = smem + kOffA + s * kABytes + (t >> 3) * 1024 + r8 * 128;
        dequant_row_step(hdr, q0, q1, g, row_smem, r8);
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&full[s]);
          // the W slots are released only now: their loads fed the dequant's stores, which precede
          // the fence, so no TMA refill can land before the reads
          mbar_arrive(&wempty[w]);
          if (g == par) mbar_arrive(&hempty[(it >> 2) % kHSlots]);
        }
      }
    }
  } else if (warp < 10) {
    // ---------------- epilogue: TMEM lanes 32*(warp%4) .. +31
    const int q = warp & 3;
    int local = 0;
    SegIter si;
    Seg sg;
    seg_begin(p, si);
    for (; !*abort && seg_next(p, si, sg); ++local) {
      const int acc = local & 1;
      const int tile = sg.tile, sp = sg.piece;
      const bool pieces = sg.npieces > 1;
      if (!mbar_wait_bounded(&tfull[acc], (local >> 1) & 1, abort, tmo)) {
        if (!*abort) fail();
        break;
      }
      tc_fence_after();
      const int64_t n = (int64_t)(tile / p.n_tiles_p) * BM + 32 * q + lane;
      const int64_t p0 = (int64_t)(tile % p.n_tiles_p) * BN;
      // the partial tile of a tile cut into pieces, column-major: a warp's store of one column is
      // one 128-byte line
      float* pcol = pieces ? p.ws + ((int64_t)tile * p.maxp + sp) * (BM * BN) + 32 * q + lane : nullptr;
#pragma unroll 1
      for (int ch = 0; ch < BN / 32; ++ch) {
        uint32_t r[32];
        tmem_ld32(tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(acc * BN + 32 * ch), r);
        if (p.x2) {
          // rows 32 b + l (l < 16) are gate channel 16 b + l, rows 32 b + 16 + l its up channel:
          // lane l < 16 finishes tokens 0..15 of this chunk and lane l + 16 tokens 16..31
          const bool up = lane >= 16;
          const int64_t c = (n >> 5) * 16 + (lane & 15);
          const int64_t pb = p0 + 32 * ch + (up ? 16 : 0);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float mine = __uint_as_float(up ? r[j] : r[16 + j]);
            const float other = __shfl_xor_sync(0xffffffffu, mine, 16);
            const float g = up ? other : __uint_as_float(r[j]);
            const float u = up ? __uint_as_float(r[16 + j]) : other;
            if (pb + j < p.P) p.x2[(pb + j) * p.F + c] = __float2bfloat16_rn(silu_mul(g, u));
          }
        } else if (pieces) {
#pragma unroll
          for (int j = 0; j < 32; ++j) pcol[(32 * ch + j) * BM] = __uint_as_float(r[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t pp = p0 + 32 * ch + j;
            if (pp < p.P && n < p.N) p.Y[pp * p.N + n] = __uint_as_float(r[j]);
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
    }
  } else {
    // ---------------- TMA producer (W): read once per output tile row, evict first
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      const int nsb = (int)(p.K / 256);
      int wq = 0, nh = 0;  // quant and header loads issued
      SegIter si;
      Seg sg;
      seg_begin(p, si);
      while (!*abort && seg_next(p, si, sg)) {
        const int row0 = (sg.tile / p.n_tiles_p) * BM;
        for (int kt = sg.k0; kt < sg.k1 && kt < 4 * nsb; ++kt, ++wq) {
          if ((kt & 3) == 0) {
            // super-block kt / 4 (the CTA's (wq / 4)-th): the rows' headers, bytes [144 sb, +16)
            const int hu = wq >> 2, h = hu % kHSlots;
            if (hu >= kHSlots && !mbar_wait_bounded(&hempty[h], ((hu / kHSlots) - 1) & 1, abort, tmo)) {
              if (!*abort) fail();
              break;
            }
            mbar_arrive_expect_tx(&hfull[h], kHTile);
            tma_load_2d_hint(smem + kOffH + h * kHTile, &wmap, (kt >> 2) * 144, row0, &hfull[h], pol);
            ++nh;
          }
          const int w = wq % kWSlots;
          if (wq >= kWSlots && !mbar_wait_bounded(&wempty[w], ((wq / kWSlots) - 1) & 1, abort, tmo)) {
            if (!*abort) fail();
            break;
          }
          // K step g of the super-block: the rows' quants, bytes [144 sb + 16 + 32 g, +32)
          mbar_arrive_expect_tx(&wfull[w], kWTile);
          tma_load_2d_hint(smem + kOffW + w * kWTile, &qmap, (kt >> 2) * 144 + 16 + 32 * (kt & 3), row0, &wfull[w],
                           pol);
        }
        if (*abort) break;
      }
      // let in-flight copies land before the CTA can exit
      for (int q = wq - kWSlots < 0 ? 0 : wq - kWSlots; q < wq; ++q) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&wfull[q % kWSlots], (q / kWSlots) & 1))
          if (globaltimer_ns() - t0 > 200000000ull) break;
      }
      for (int q = nh - kHSlots < 0 ? 0 : nh - kHSlots; q < nh; ++q) {
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&hfull[q % kHSlots], (q / kHSlots) & 1))
          if (globaltimer_ns() - t0 > 200000000ull) break;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols) : "memory");
  }
}

__global__ void swiglu_bf16_kernel(const float* __restrict__ Y1, int64_t P, int64_t half,
                                   __nv_bfloat16* __restrict__ X2) {
  const int64_t total = P * half;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / half, c = i - r * half;
    const float g = Y1[r * 2 * half + c], u = Y1[r * 2 * half + half + c];
    X2[i] = __float2bfloat16_rn(silu_mul(g, u));
  }
}

// W13 row R = 32 b + l: gate row 16 b + l for l < 16, up row 16 b + l - 16 otherwise.
// Stream-K fix-up: every output of a tile cut into pieces is the sum of the tile's pieces in K
// order (piece 0 first), so the result does not depend on which CTA finished first.  Block b
// handles 8 columns (tokens) of tile b / (BN / 8); lane l of warp w the 4 rows 4l .. 4l + 3 of
// column 8 (b % (BN / 8)) + w.  Launched right after q4k_gemm_kernel with programmatic
// serialization: griddepcontrol.wait returns once that grid has completed and its writes are
// visible.  G is the GEMM's grid, work = tiles * nsb.
__global__ void __launch_bounds__(256) streamk_fixup_kernel(const __grid_constant__ GemmParams p, int64_t work,
                                                            int G) {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int tile = (int)(blockIdx.x / (BN / 8));
  const int col = (int)(blockIdx.x % (BN / 8)) * 8 + (int)(threadIdx.x >> 5);
  const int64_t tb = (int64_t)tile * p.nsb, te = tb + p.nsb;
  const int64_t cf = ((tb + 1) * G + work - 1) / work - 1, cl = (te * G + work - 1) / work - 1;
  const int np = (int)(cl - cf + 1);
  const int64_t pp = (int64_t)(tile % p.n_tiles_p) * BN + col;
  if (np < 2 || pp >= p.P) return;  // a whole tile was written by its CTA; a token past P has no row
  const int row = 4 * (threadIdx.x & 31);
  const float4* src = reinterpret_cast<const float4*>(p.ws + (int64_t)tile * p.maxp * (BM * BN) + (int64_t)col * BM + row);
  float4 a = __ldcg(src);
  for (int k = 1; k < np; ++k) {
    const float4 v = __ldcg(src + (int64_t)k * (BM * BN / 4));
    a.x += v.x;
    a.y += v.y;
    a.z += v.z;
    a.w += v.w;
  }
  const int64_t n = (int64_t)(tile / p.n_tiles_p) * BM + row;
  float* y = p.Y + pp * p.N + n;
  const float o[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int e = 0; e < 4; ++e)
    if (n + e < p.N) y[e] = o[e];
}

__global__ void interleave_gate_up_kernel(const uint4* __restrict__ Wg, const uint4* __restrict__ Wu, int64_t F,
                                          int64_t row16, uint4* __restrict__ W13) {
  const int64_t total = 2 * F * row16;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t R = i / row16, k = i - R * row16;
    const int64_t b = R >> 5, l = R & 31;
    const int64_t src = 16 * b + (l & 15);
    W13[i] = (l < 16 ? Wg : Wu)[src * row16 + k];
  }
}

std::mutex g_gemm_mu;
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
bool g_gemm_attr[64] = {};

int gemm_setup(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fak_cuda_status(e);
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (major != 10 || minor != 3) return FAK_ERR_UNSUPPORTED;
  cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, dev);
  std::lock_guard<std::mutex> lk(g_gemm_mu);
  if (!g_encode) {
    cudaDriverEntryPointQueryResult q;
    void* fn = nullptr;
    e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn) return fak_cuda_status(e);
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  if (dev >= 0 && dev < 64 && !g_gemm_attr[dev]) {
    e = cudaFuncSetAttribute(q4k_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAllocG);
    if (e != cudaSuccess) return fak_cuda_status(e);
    g_gemm_attr[dev] = true;
  }
  return FAK_OK;
}

}  // namespace

extern "C" int fak_swiglu_bf16(const float* Y1, int64_t P, int64_t half, void* X2, fak_stream_t stream) {
  if (!Y1 || !X2) return FAK_ERR_INVALID_ARG;
  if (P < 1 || half < 1) return FAK_ERR_SHAPE;
  const int64_t total = P * half;
  const int64_t want = (total + 255) / 256;
  const int grid = (int)(want < 152 * 16 ? want : 152 * 16);
  swiglu_bf16_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(Y1, P, half, static_cast<__nv_bfloat16*>(X2));
  return fak_cuda_status(cudaGetLastError());
}

namespace {
// The work split of an N x K x P GEMM on `sms` SMs: whole tiles, or stream-K (see launch_gemm).
struct SkPlan {
  int tiles, nsb, n_tiles_p, gs, maxp;
  int64_t work;
  bool stream;
};

SkPlan plan_gemm(int64_t N, int64_t K, int64_t P, int sms, bool x2) {
  SkPlan pl;
  pl.n_tiles_p = (int)((P + BN - 1) / BN);
  pl.tiles = (int)((N + BM - 1) / BM) * pl.n_tiles_p;
  pl.nsb = (int)(K / 256);
  // Stream-K when whole tiles fill the SMs poorly: the tiles' K work is cut into `sms` equal
  // ranges, one per CTA, at super-block granularity.  Cost model in super-blocks of work on the
  // critical path: whole tiles waves(tiles) * nsb; stream-K ceil(tiles * nsb / sms) +
  // kStreamKFixCost, the constant standing for writing the pieces and the fix-up kernel that sums
  // them; stream-K is taken below 0.85 x the whole-tile cost.  Both set by timing the two forms on
  // the prefill shapes (P = 128 .. 1024): stream-K won by 2-3x where it costs under 0.65 x the whole
  // tiles (down, out projections) and lost 0-8 % at 0.85-0.9 (gate||up, in_proj: several full
  // waves of whole tiles).  Not with the SwiGLU epilogue, which needs whole
  // tiles (so the fused gate||up GEMM equals the unfused one bit for bit when the unfused takes
  // whole tiles).
  pl.work = (int64_t)pl.tiles * pl.nsb;
  pl.gs = (int)std::min<int64_t>(sms, pl.work);  // stream-K CTAs: every range at least one super-block
  const double whole = (double)((pl.tiles + sms - 1) / sms) * pl.nsb;
  const double streamk = (double)((pl.work + pl.gs - 1) / pl.gs) + kStreamKFixCost;
  pl.stream = !x2 && streamk < 0.85 * whole;
  pl.maxp = 1;
  if (pl.stream) {
    // the most pieces any tile is cut into (CTA c's range starts at floor(c work / sms))
    for (int t = 0; t < pl.tiles; ++t) {
      const int64_t tb = (int64_t)t * pl.nsb, te = tb + pl.nsb;
      const int64_t cf = ((tb + 1) * pl.gs + pl.work - 1) / pl.work - 1, cl = (te * pl.gs + pl.work - 1) / pl.work - 1;
      pl.maxp = std::max<int>(pl.maxp, (int)(cl - cf + 1));
    }
  }
  return pl;
}

size_t pieces_bytes(const SkPlan& pl) {
  return pl.stream && pl.maxp > 1 ? (size_t)pl.tiles * pl.maxp * BM * BN * 4 : 0;
}

// ext_ws / out: the pieces of a stream-K split go to the caller's workspace (ext_ws_bytes must hold
// them) and *out describes them; no fix-up kernel runs, and the tiles cut into pieces are not
// written to Y.
int launch_gemm(const void* Wq, int64_t N, int64_t K, const void* X, int64_t P, float* Y, __nv_bfloat16* x2,
                fak_stream_t stream_arg, float* ext_ws = nullptr, size_t ext_ws_bytes = 0,
                FakGemmPieces* out = nullptr) {
  if (out) {
    out->ws = nullptr;
    out->work = 0;
    out->gs = out->nsb = out->maxp = out->n_tiles_p = 0;
  }
  if (K < 256 || K % 256 || N < 1 || N > (1LL << 31) - 1 || P < 1 || P > (1LL << 31) - 1 || K > (1LL << 31) - 1)
    return FAK_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(Wq) & 15) || (reinterpret_cast<uintptr_t>(X) & 15)) return FAK_ERR_ALIGN;
  int sms = 0;
  int st = gemm_setup(&sms);
  if (st != FAK_OK) return st;
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  const cuuint64_t gdim[2] = {(cuuint64_t)K, (cuuint64_t)P};
  const cuuint64_t gstride[1] = {(cuuint64_t)K * 2};
  const cuuint32_t box[2] = {BK, BN};
  const cuuint32_t estride[2] = {1, 1};
  CUresult r = g_encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(X), gdim, gstride, box, estride,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return FAK_ERR_CUDA;
  // W as bytes [N rows, K/256*144]: per K step a 128-row x 16-byte box of block headers and a
  // 128-row x 32-byte box of the step's quants
  CUtensorMap wmap, qmap;
  memset(&wmap, 0, sizeof(wmap));
  memset(&qmap, 0, sizeof(qmap));
  const cuuint64_t row_bytes = (cuuint64_t)(K / 256) * 144;
  const cuuint64_t wdim[2] = {row_bytes, (cuuint64_t)N};
  const cuuint64_t wstride[1] = {row_bytes};
  const cuuint32_t hbox[2] = {16, BM}, qbox[2] = {32, BM};
  r = g_encode(&wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(Wq), wdim, wstride, hbox, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return FAK_ERR_CUDA;
  r = g_encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(Wq), wdim, wstride, qbox, estride,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return FAK_ERR_CUDA;
  GemmParams gp;
  gp.W = static_cast<const uint8_t*>(Wq);
  gp.Y = Y;
  gp.N = N;
  gp.K = K;
  gp.P = P;
  gp.n_tiles_n = (int)((N + BM - 1) / BM);  // a last partial tile reads zero-filled rows past N, writes none
  gp.n_tiles_p = (int)((P + BN - 1) / BN);
  gp.timeout_ns = 2000000000ull;
  const SkPlan pl = plan_gemm(N, K, P, sms, x2 != nullptr);
  const int tiles = pl.tiles, nsb = pl.nsb, gs = pl.gs;
  const int64_t work = pl.work;
  const bool stream = pl.stream;
  gp.splits = 1;
  gp.sb_per = nsb;
  gp.stream = stream ? 1 : 0;
  gp.nsb = nsb;
  gp.maxp = pl.maxp;
  gp.x2 = x2;
  gp.F = N / 2;
  gp.ws = nullptr;
  cudaStream_t s = (cudaStream_t)stream_arg;
  void* buf = nullptr;
  bool fixup = stream && gp.maxp > 1;
  if (fixup && out && ext_ws && ext_ws_bytes >= pieces_bytes(pl)) {
    gp.ws = ext_ws;
    out->ws = ext_ws;
    out->work = work;
    out->gs = gs;
    out->nsb = nsb;
    out->maxp = gp.maxp;
    out->n_tiles_p = gp.n_tiles_p;
    fixup = false;
  } else if (fixup) {
    const size_t ws_bytes = (size_t)tiles * gp.maxp * BM * BN * 4;
    const cudaError_t e = fak_scratch_alloc(&buf, ws_bytes, s);
    if (e != cudaSuccess) {
      (void)cudaGetLastError();
      return FAK_ERR_NOMEM;
    }
    gp.ws = static_cast<float*>(buf);
  }
  const int grid = stream ? gs : (tiles < sms ? tiles : sms);
  q4k_gemm_kernel<<<grid, kThreadsG, kSmemAllocG, s>>>(map, wmap, qmap, gp);
  cudaError_t le = cudaGetLastError();
  if (fixup && le == cudaSuccess) {
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3((unsigned)tiles * (BN / 8));
    cfg.blockDim = dim3(256);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    le = cudaLaunchKernelEx(&cfg, streamk_fixup_kernel, gp, work, gs);
  }
  if (buf) cudaFreeAsync(buf, s);
  return fak_cuda_status(le);
}
}  // namespace

extern "C" int fak_q4k_gemm(const void* Wq, int64_t N, int64_t K, const void* X, int64_t P, float* Y,
                            fak_stream_t stream) {
  if (!Wq || !X || !Y) return FAK_ERR_INVALID_ARG;
  return launch_gemm(Wq, N, K, X, P, Y, nullptr, stream);
}

size_t fak_gemm_pieces_bytes(int64_t N, int64_t K, int64_t P) {
  int sms = 0;
  if (K < 256 || K % 256 || N < 1 || P < 1 || gemm_setup(&sms) != FAK_OK) return 0;
  return pieces_bytes(plan_gemm(N, K, P, sms, false));
}

int fak_q4k_gemm_pieces(const void* Wq, int64_t N, int64_t K, const void* X, int64_t P, float* Y, float* ws,
                        size_t ws_bytes, FakGemmPieces* out, fak_stream_t stream) {
  if (!Wq || !X || !Y || !out) return FAK_ERR_INVALID_ARG;
  return launch_gemm(Wq, N, K, X, P, Y, nullptr, stream, ws, ws_bytes, out);
}

extern "C" int fak_q4k_gemm_swiglu(const void* W13, int64_t F, int64_t K, const void* X, int64_t P, void* X2,
                                   fak_stream_t stream) {
  if (!W13 || !X || !X2) return FAK_ERR_INVALID_ARG;
  if (F < 64 || F % 64 || F > (1LL << 30)) return FAK_ERR_SHAPE;
  if (reinterpret_cast<uintptr_t>(X2) & 15) return FAK_ERR_ALIGN;
  return launch_gemm(W13, 2 * F, K, X, P, nullptr, static_cast<__nv_bfloat16*>(X2), stream);
}

extern "C" int fak_q4k_interleave_gate_up(const void* Wg, const void* Wu, int64_t F, int64_t K, void* W13,
                                          fak_stream_t stream) {
  if (!Wg || !Wu || !W13) return FAK_ERR_INVALID_ARG;
  if (F < 64 || F % 64 || K < 256 || K % 256 || F > (1LL << 30) || K > (1LL << 31) - 1) return FAK_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(Wg) | reinterpret_cast<uintptr_t>(Wu) | reinterpret_cast<uintptr_t>(W13)) & 15)
    return FAK_ERR_ALIGN;
  const int64_t row16 = K / 256 * 144 / 16;
  const int64_t want = (2 * F * row16 + 255) / 256;
  const int grid = (int)(want < 152 * 32 ? want : 152 * 32);
  interleave_gate_up_kernel<<<grid, 256, 0, (cudaStream_t)stream>>>(
      static_cast<const uint4*>(Wg), static_cast<const uint4*>(Wu), F, row16, static_cast<uint4*>(W13));
  return fak_cuda_status(cudaGetLastError());
}

int fak_gemm_take_status() {
  int v = 0, zero = 0;
  cudaError_t e;
  e = cudaMemcpyFromSymbol(&v, g_gemm_status, sizeof(int));
  if (e != cudaSuccess) return fak_cuda_status(e);
  cudaMemcpyToSymbol(g_gemm_status, &zero, sizeof(int));
  return v;
}
