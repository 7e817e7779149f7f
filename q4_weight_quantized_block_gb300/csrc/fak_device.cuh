// Small sm_100-family device helpers shared by the library's kernels: shared
// memory addresses, mbarriers, bulk (TMA) copies, acquire/release accesses,
// the global nanosecond timer and bounded waits.
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "fak.h"

#define FAK_DEV __device__ __forceinline__

FAK_DEV uint32_t smem_u32(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

FAK_DEV uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

FAK_DEV void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

FAK_DEV void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }

FAK_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

FAK_DEV void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

FAK_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// try_wait with a suspend-time hint: the thread sleeps until the phase
// completes or about `hint_ns` pass, instead of spinning and taking issue
// slots from the warps that share its scheduler.
FAK_DEV bool mbar_try_wait_suspend(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// Bounded wait on an mbarrier phase.  Gives up when `abort` becomes non-zero
// or after `timeout_ns`; returns false then.  Between checks the thread is
// suspended (at most ~20 us per check).
FAK_DEV bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort, uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait_suspend(bar, parity, 20000u)) return true;
    if (*abort) return false;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// L2 policy: data read once (weights) is evicted first.
FAK_DEV uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Bulk global->shared copy completing on an mbarrier.  dst, src 16-byte
// aligned, bytes a multiple of 16.
FAK_DEV void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

FAK_DEV uint32_t ld_acquire_gpu(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// Release-ordered add: this CTA's prior writes (made visible to thread 0 by
// the barrier before it) happen-before any acquire that observes the sum.
FAK_DEV void red_release_gpu_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

FAK_DEV float4 ld_cg_f4(const float* p) {
  float4 v;
  asm volatile("ld.global.cg.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p));
  return v;
}

FAK_DEV float ld_cg_f(const float* p) {
  float v;
  asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p));
  return v;
}

FAK_DEV int ld_cg_i(const int* p) {
  int v;
  asm volatile("ld.global.cg.s32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// Strong (relaxed, gpu scope) accesses for values that carry a version tag in
// their lowest significand bit: they are read from and written to L2, the
// point of coherence, so a poll that sees the tag it waits for sees the value
// stored with it (same 32-bit word).
FAK_DEV float4 ld_relaxed_f4(const float* p) {
  float4 v;
  asm volatile("ld.relaxed.gpu.global.v4.f32 {%0,%1,%2,%3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

FAK_DEV float ld_relaxed_f(const float* p) {
  float v;
  asm volatile("ld.relaxed.gpu.global.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
  return v;
}

// Stores v rounded to 22 significand bits (to nearest, ties to even: no drift
// over the many residual updates of a decode token) with the tag in the freed
// lowest bit; consumers read it back through untag.
FAK_DEV void st_tagged(float* p, float v, uint32_t tag) {
  uint32_t b = __float_as_uint(v);
  b = (b & 1u) ? ((b & 2u) ? b + 1u : b - 1u) : b;
  b |= tag;
  asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(b) : "memory");
}

// The value a tagged word stands for: its tag bit cleared.  Every consumer uses
// this, so a value does not depend on which tag it was stored with.
FAK_DEV float untag(float v) { return __uint_as_float(__float_as_uint(v) & ~1u); }
FAK_DEV float4 untag4(float4 v) { return make_float4(untag(v.x), untag(v.y), untag(v.z), untag(v.w)); }

// Non-zero when any of the eight values lacks the version tag `want`.
FAK_DEV uint32_t stale8(const float4& a, const float4& b, uint32_t want) {
  const uint32_t o = (__float_as_uint(a.x) ^ want) | (__float_as_uint(a.y) ^ want) | (__float_as_uint(a.z) ^ want) |
                     (__float_as_uint(a.w) ^ want) | (__float_as_uint(b.x) ^ want) | (__float_as_uint(b.y) ^ want) |
                     (__float_as_uint(b.z) ^ want) | (__float_as_uint(b.w) ^ want);
  return o & 1u;
}

// named barrier among `count` threads (count a multiple of 32)
FAK_DEV void named_bar_sync(int id, int count) { asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory"); }

FAK_DEV uint32_t dp4a_uu(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("dp4a.u32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
FAK_DEV int dp4a_us(uint32_t a, uint32_t b, int c) {  // a unsigned bytes, b signed bytes
  int d;
  asm("dp4a.u32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
FAK_DEV int dp4a_su(uint32_t a, uint32_t b, int c) {  // a signed bytes, b unsigned bytes
  int d;
  asm("dp4a.s32.u32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}
FAK_DEV int dp4a_ss(uint32_t a, uint32_t b, int c) {
  int d;
  asm("dp4a.s32.s32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

FAK_DEV uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
  return d;
}

FAK_DEV float half_bits_to_float(uint32_t h16) {
  float f;
  asm("{ .reg .b16 t; cvt.u16.u32 t, %1; cvt.f32.f16 %0, t; }" : "=f"(f) : "r"(h16));
  return f;
}

// Host-side launch-error mapping shared by the .cu files.
static inline int fak_cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return FAK_OK;
  (void)cudaGetLastError();
  return FAK_ERR_CUDA;
}

// Reads and clears the prefill GEMM's device status word (host side, after a sync).
int fak_gemm_take_status();
// The same for the batched GEMV.
int fak_bgemv_take_status();
// Stream-ordered scratch for one call: from a library-owned pool per device
// that keeps its memory for the next call (no allocation cost once warm), or,
// while the stream is being captured into a graph, cudaMallocAsync (a graph
// memory node).  Free with cudaFreeAsync on the same stream.
cudaError_t fak_scratch_alloc(void** p, size_t bytes, cudaStream_t s);

// Stream-K pieces of a prefill GEMM left to the caller's consumer instead of the fix-up kernel
// (the prefill forward's residual add + RMSNorm sums them itself).  ws holds
// [tiles][maxp][256 tokens][128 rows] f32 (tile t = row tile * n_tiles_p + token tile); the pieces
// of tile t are those of the CTAs cf .. cl with cf = ((t nsb + 1) gs + work - 1) / work - 1 and
// cl = ((t + 1) nsb gs + work - 1) / work - 1, summed in that order.  A tile met by one CTA was
// written to Y.  ws == null: Y is complete.
struct FakGemmPieces {
  const float* ws;
  int64_t work;  // tiles * nsb
  int gs, nsb, maxp, n_tiles_p;
};
// Bytes of the pieces an N x K x P fak_q4k_gemm would cut (0 when it takes whole tiles).
size_t fak_gemm_pieces_bytes(int64_t N, int64_t K, int64_t P);
// fak_q4k_gemm, but a stream-K split leaves its pieces in ws (when ws_bytes holds them) and
// describes them in *out; otherwise as fak_q4k_gemm, with out->ws = null.
int fak_q4k_gemm_pieces(const void* Wq, int64_t N, int64_t K, const void* X, int64_t P, float* Y, float* ws,
                        size_t ws_bytes, FakGemmPieces* out, fak_stream_t stream);
