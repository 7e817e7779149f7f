// The matrix-vector engine: Q4_K / Q8_0 weight-streaming GEMV on sm_103a, and
// a list of such matvecs (with RMSNorm on the input, SwiGLU / residual-add /
// argmax epilogues) run as ONE persistent launch with bounded grid-wide waits
// between dependent steps.
//
// What it computes follows "Mac Qwen3.6-27B Metal Q4_K perf diagnosis": the
// per-projection Q4_K GEMV (TL;DR), the lm_head_q8 matvec (section 2 profile)
// and the one-submission-per-token decode forward (section 4, "the lever"),
// where the activation stays on the GPU across every matmul of a token.
//
// Design (GB300-first):
//  * One CTA per SM, 12 warps, ~227 KB shared memory.  Each warp owns three
//    4.6 KB stage buffers (4 row slots x 8 Q4_K blocks, or 4 x 32 Q8_0 blocks)
//    and streams its weight rows HBM -> shared memory with 16-byte cp.async
//    (LDGSTS, L2-only), two stages in flight while it computes a third.
//    Weights do not depend on activations, so a warp that has finished its
//    part of a step issues the next step's third stage before the grid-wide
//    wait.  (Measured on GB300: per-warp LDGSTS streams at ~7.2 TB/s with no
//    compute, while 1 KB bulk copies from one issuing thread reach ~0.5 TB/s.)
//  * Every CTA quantizes x once per step into shared memory: per 256-element
//    super-block a power-of-two scale s with |x/s| <= 2^22, X = rint(x/s) split
//    into three byte limbs (X = X2*65536 + X1*256 + X0, X0/X1 unsigned, X2
//    signed).  The dot over each 32-weight sub-block is then exact integer
//    arithmetic (DP4A on 4-bit quants x byte limbs); the sub-block scales sc_j
//    are applied in integers, and one f32 conversion per 64 weights follows.
//    Relative to f32 activations this adds at most 2^-23 * max|x| per element
//    of its super-block.
//  * Lanes cover (block, 64-weight group) pairs, so the x limbs a lane holds in
//    registers serve all four row slots of a stage.  A step's rows are cut
//    into (4-row group, 8-block slab) units: small steps deal one CTA's units
//    to its warps ("split"), large steps give every warp of the grid its own
//    rows ("rows").  Row results are reduced with a fixed shuffle tree and
//    split groups are summed in slab order: bitwise deterministic.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <vector>

#include "fak.h"
#include "fak_device.cuh"

namespace {

constexpr int kNumConsumerWarps = 12;
constexpr int kSlots = 4;                         // weight row slots per stage
constexpr int kLanesPerSlot = 32 / kSlots;
constexpr int kThreads = 32 * kNumConsumerWarps;
constexpr int kConsumerThreads = 32 * kNumConsumerWarps;
constexpr int kBuffers = 3;                      // stage buffers per warp (two copies in flight)
constexpr int kStages = kBuffers * kNumConsumerWarps;
constexpr int kStageBytes = kSlots * 1152;       // row slots x 8 Q4_K blocks x 144 B
constexpr int kRowsPerGroup = kSlots;
constexpr int kQ4SlabBlocks = 8;         // Q4_K blocks per row per stage
constexpr int kQ8SlabBlocks = 32;        // Q8_0 blocks per row per stage
constexpr int kQ4StageRow = kQ4SlabBlocks * 144;  // 1152
constexpr int kQ8StageRow = kQ8SlabBlocks * 34;   // 1088
constexpr int kMaxSuper = FAK_ENGINE_MAX_K / 256; // 72
// x limbs of one 256-element super-block: four 208-byte group records (group g
// holds sub-blocks 2g and 2g+1: 3 x 32 limb bytes each, then 16 bytes of
// padding); 832-byte super-blocks keep the Q4_K lanes' 16-byte reads free of
// bank conflicts.
constexpr int kGroupRec = 208;
constexpr int kSuperBytes = 4 * kGroupRec;        // 832

constexpr int kOffRing = 0;
constexpr int kOffX = kOffRing + kStages * kStageBytes;
constexpr int kOffS = kOffX + kMaxSuper * kSuperBytes;
constexpr int kOffScale = kOffS + kMaxSuper * 8 * 4;
constexpr int kWarmStages = 4;                    // stages per warp warmed in L2 before a dependent launch's wait
constexpr int kMaxUnits = 200;                    // (row group, slab) units per CTA in split mode
constexpr int kOffPart = kOffScale + kMaxSuper * 4;
constexpr int kOffMisc = kOffPart + kMaxUnits * kSlots * 4;
constexpr int kOffDesc = kOffMisc + 256;          // the current and the next step's descriptor
constexpr int kSmemBytes = kOffDesc + 2 * 128;
constexpr int kSmemAlloc = kSmemBytes + 128;
static_assert(kSmemAlloc <= 232448, "engine shared memory exceeds the 227 KB per-block limit");

enum OpKind { OP_Q4K = 0, OP_Q4K_SWIGLU = 1, OP_Q8 = 2, OP_EMBED = 3, OP_ARGMAX_REDUCE = 4, OP_GDN = 5, OP_ATTN = 6 };
// F_WAIT: wait for the grid-wide arrival counter before the step; F_NOARRIVE: the CTA does not add
// to that counter after the step; F_TAGIN / F_TAGOUT: the step's input / outputs carry version tags
// (below) instead.
enum OpFlag { F_NORM = 1, F_RESID = 2, F_WAIT = 4, F_ARGMAX = 8, F_TAGIN = 16, F_TAGOUT = 32, F_NOARRIVE = 64 };

// Version tags.  In a multi-step launch a step's outputs are the next step's inputs.  Instead of a
// grid-wide barrier between the two, every output value carries the parity of its buffer's version
// in the lowest bit of its f32 significand (a change of at most one unit in the last place), and the
// consumer polls the values it needs until all of them carry the expected parity.  One bit is
// enough when every version of a buffer overwrites every element its readers read and each reader
// reads the same elements at every version: a CTA polling for version v has then already seen
// version v-1 at each of those elements, and L2 coherence never hands it an older value after a
// newer one.  (The decode's buffers are laid out so: with the mixer bodies, the full-attention
// layers' q+gate output has a buffer of its own, because it does not cover the GDN in_proj rows.)
// Tag of version v of buffer b in token k: (k * writes_per_token(b) + v) & 1, the host passing bit
// b of (k * writes_per_token(b)) & 1 in EngParams::flip; freshly zeroed buffers hold version 0.
// tags bits: [2:0] input buffer, [3] input version parity; per output segment s: [4s+6:4s+4] buffer,
// [4s+7] version parity.
FAK_DEV uint32_t tag_in_buf(int32_t t) { return (uint32_t)t & 7u; }
FAK_DEV uint32_t tag_in_par(int32_t t) { return ((uint32_t)t >> 3) & 1u; }
FAK_DEV uint32_t tag_out_buf(int32_t t, int s) { return ((uint32_t)t >> (4 + 4 * s)) & 7u; }
FAK_DEV uint32_t tag_out_par(int32_t t, int s) { return ((uint32_t)t >> (7 + 4 * s)) & 1u; }

struct EngOp {
  int32_t kind, flags, K, nseg;
  int32_t wait_extra, vocab;
  int64_t nrows;            // output rows (SWIGLU: rows of gate = rows of up)
  int64_t seg_end[3];       // cumulative row ends per segment
  const uint8_t* w[3];      // weights per segment (SWIGLU: w[0] gate, w[1] up)
  float* y[3];              // outputs per segment
  const float* x;           // input vector [K] (EMBED: the embedding table)
  float eps;
  int32_t tags;             // version tags of the input and the output segments (F_TAGIN / F_TAGOUT)
  int32_t wait_target;      // F_WAIT: arrivals per CTA the step waits for (plus wait_extra)
  int32_t pad;
};
static_assert(sizeof(EngOp) == 128, "step descriptors are copied to shared memory as 128 bytes");

struct EngParams {
  const EngOp* ops;         // device array, or NULL to use inl[]
  int n_ops;
  int first_wait;
  unsigned* sync;           // [0] steps done (sum over CTAs), [1] CTAs exited; NULL: no grid waits
  int* err;
  float* cand_val;
  int* cand_idx;
  const int* tok_in;
  int* tok_out;
  float* logits;
  unsigned long long timeout_ns;
  unsigned flip;            // bit b: version-tag flip of buffer b for this token; bit 8: token parity
  int* pos;                 // decode with the mixer bodies: the token's position (advanced by the argmax step)
  EngOp inl[2];             // used when ops == NULL (at most 2 steps)
};

// A mixer step's operands (device memory, one per layer; EngOp::x points at it).
struct MixDesc {
  const float* t;        // in_proj (GDN) / q+gate (FA) output, tagged
  const float* kin;      // FA: k projection, tagged
  const float* vin;      // FA: v projection, tagged
  float* out;            // the mixer output [n_mix], tagged
  const float* conv_w;   // GDN: [conv_dim][4]
  const float* a_log;    // GDN: [nv]
  const float* dt_bias;  // GDN: [nv]
  const float* norm_w;   // GDN: [128]
  float* conv_state;     // GDN: [2][conv_dim][3], double-buffered by token parity
  float* S;              // GDN: [nv][128][128]
  const float* q_norm_w; // FA: [256]
  const float* k_norm_w; // FA: [256]
  float* kc;             // FA: [nkv][max_ctx][256]
  float* vc;             // FA: [nkv][max_ctx][256]
  int32_t nk, nv, nq, nkv, rot, max_ctx;
  float theta, eps;
  double inv_freq[128];  // FA: theta^(-2i/rot) for i < rot / 2, in double (host pow)
};

__device__ int g_fak_status;  // status word of the stateless entry points


struct Geo {
  int U;          // output rows per group
  int bpr;        // blocks per row
  int slab;       // blocks per row per stage
  int nslab;
  int blk;        // bytes per block
  int srow;       // bytes between row slots in a stage
  bool pair, q8;
};

__device__ __forceinline__ Geo geo_of(const EngOp& op) {
  Geo g;
  g.q8 = op.kind == OP_Q8;
  g.pair = op.kind == OP_Q4K_SWIGLU;
  g.U = g.pair ? kSlots / 2 : kRowsPerGroup;
  g.bpr = g.q8 ? op.K / 32 : op.K / 256;
  g.slab = g.q8 ? kQ8SlabBlocks : kQ4SlabBlocks;
  g.nslab = g.q8 ? (g.bpr + kQ8SlabBlocks - 1) / kQ8SlabBlocks : (g.bpr + kQ4SlabBlocks - 1) / kQ4SlabBlocks;
  g.blk = g.q8 ? 34 : 144;
  g.srow = g.q8 ? kQ8StageRow : kQ4StageRow;
  return g;
}

__device__ __forceinline__ bool has_weights(int kind) {
  return kind == OP_Q4K || kind == OP_Q4K_SWIGLU || kind == OP_Q8;
}

// Work split of a step.  Each CTA owns a contiguous range of output rows,
// cut into groups of U rows; a (group, slab) pair is a unit.  When the CTA has
// at most kMaxUnits units ("split" mode) its warps take equal contiguous runs
// of units, so a group's slabs may be shared by two or three warps; each warp
// leaves one partial sum per segment (a maximal run of one group's slabs) in
// shared memory and the groups are summed afterwards in slab order.  Larger
// steps ("rows" mode) give every warp of the grid a contiguous range of rows,
// balanced to one row, and its groups are finished by the warp itself.
struct Plan {
  int r_lo, r_hi;      // row window: the CTA's rows (split) or the warp's rows
  int u0, u1;          // this warp's units; unit u is group u / nslab, slab u % nslab
  int ngroups;         // groups in the window
  int total;           // units of the CTA (split mode)
  bool split;
};

__device__ __forceinline__ Plan plan_of(const EngOp& op, const Geo& g, int cw) {
  Plan p;
  const int64_t c = blockIdx.x, G = gridDim.x;
  int64_t R0, R1;
  if (op.nrows <= 0x7fffffff / (G + 1)) {
    // every decode step: the products fit 32 bits, and a 32-bit division is a fraction of a 64-bit one
    const unsigned n = (unsigned)op.nrows, cu = (unsigned)c, Gu = (unsigned)G;
    R0 = n * cu / Gu;
    R1 = n * (cu + 1) / Gu;
  } else {
    R0 = op.nrows * c / G;
    R1 = op.nrows * (c + 1) / G;
  }
  const int64_t ng = (R1 - R0 + g.U - 1) / g.U;
  const int64_t total = ng * g.nslab;
  if (total <= kMaxUnits) {
    const int t = (int)total;
    p.split = true;
    p.r_lo = (int)R0;
    p.r_hi = (int)R1;
    p.ngroups = (int)ng;
    p.total = t;
    p.u0 = t * cw / kNumConsumerWarps;
    p.u1 = t * (cw + 1) / kNumConsumerWarps;
  } else {
    const int64_t GW = G * kNumConsumerWarps, gw = c * kNumConsumerWarps + cw;
    p.split = false;
    p.r_lo = (int)(op.nrows * gw / GW);
    p.r_hi = (int)(op.nrows * (gw + 1) / GW);
    p.ngroups = (p.r_hi - p.r_lo + g.U - 1) / g.U;
    p.total = 0;
    p.u0 = 0;
    p.u1 = p.ngroups * g.nslab;
  }
  return p;
}

__device__ __forceinline__ void set_error(const EngParams& P, int code, volatile int* abort) {
  int* e = P.err ? P.err : &g_fak_status;
  atomicCAS(e, 0, code);
  *abort = 1;
}

// ------------------------------------------------------------------ stage streaming
// A warp's stages, in order across the steps of the launch: for each step with
// weights, for each of the warp's row groups, all slabs.
struct Cursor {
  int op;          // step index, n_ops when exhausted
  int u, u1;       // current and end unit of the warp in this step
  int grp, s;      // group and slab of unit u
  int nslab;
  int r_lo, r_hi;
  // the step's descriptor fields the copies need, cached in registers when the
  // cursor enters the step (reading the descriptor per stage is a slow chain)
  const uint8_t* w0;
  const uint8_t* w1;
  const uint8_t* w2;
  int se0, se1;     // segment row ends (rows >= se1 come from w2)
  int row_bytes;    // bytes per weight row
  int bpr;          // blocks per row
  bool q8, pair;
  // this lane's row slot in the current stage: source (NULL if the slot is empty)
  // and 16-byte chunks to copy
  const uint8_t* src;
  int nch;
};

// Set src / nch of this lane's slot (row slot lane / kLanesPerSlot) for the cursor's unit.
__device__ __forceinline__ void cursor_slot(Cursor& c, int lane) {
  const int rl = lane / kLanesPerSlot;
  const int slab = c.q8 ? kQ8SlabBlocks : kQ4SlabBlocks;
  const int blk = c.q8 ? 34 : 144;
  const int nb = min(slab, c.bpr - c.s * slab);
  c.nch = nb * blk / 16;
  const int64_t off = (int64_t)c.s * slab * blk;
  const int row0 = c.r_lo + c.grp * (c.pair ? kSlots / 2 : kSlots);
  c.src = nullptr;
  if (c.pair) {
    const int row = row0 + (rl % (kSlots / 2));
    if (row < c.r_hi) c.src = (rl < kSlots / 2 ? c.w0 : c.w1) + (int64_t)row * c.row_bytes + off;
    return;
  }
  const int row = row0 + rl;
  if (row >= c.r_hi) return;
  const uint8_t* w = row < c.se0 ? c.w0 : (row < c.se1 ? c.w1 : c.w2);
  const int base = row < c.se0 ? 0 : (row < c.se1 ? c.se0 : c.se1);
  c.src = w + (int64_t)(row - base) * c.row_bytes + off;
}

__device__ __forceinline__ void cursor_load(const EngParams& P, Cursor& c, int cw, int lane) {
  c.u = c.u1 = 0;
  if (c.op >= P.n_ops) return;
  const EngOp& op = P.ops ? P.ops[c.op] : P.inl[c.op];
  if (!has_weights(op.kind)) return;
  const Geo g = geo_of(op);
  const Plan pl = plan_of(op, g, cw);
  c.u = pl.u0;
  c.u1 = pl.u1;
  c.nslab = g.nslab;
  c.grp = pl.u0 / g.nslab;
  c.s = pl.u0 - c.grp * g.nslab;
  c.r_lo = pl.r_lo;
  c.r_hi = pl.r_hi;
  c.w0 = op.w[0];
  c.w1 = op.w[1];
  c.w2 = op.w[2];
  c.se0 = op.nseg > 1 ? (int)op.seg_end[0] : 0x7fffffff;
  c.se1 = op.nseg > 2 ? (int)op.seg_end[1] : 0x7fffffff;
  c.row_bytes = g.bpr * g.blk;
  c.bpr = g.bpr;
  c.q8 = g.q8;
  c.pair = g.pair;
  if (c.u < c.u1) cursor_slot(c, lane);
}

__device__ __forceinline__ bool cursor_settle(const EngParams& P, Cursor& c, int cw, int lane) {
  while (c.op < P.n_ops && c.u >= c.u1) {
    ++c.op;
    cursor_load(P, c, cw, lane);
  }
  return c.op < P.n_ops;
}

__device__ __forceinline__ void cursor_advance(const EngParams& P, Cursor& c, int cw, int lane) {
  ++c.u;
  if (c.u >= c.u1) {
    cursor_settle(P, c, cw, lane);
    return;
  }
  if (++c.s < c.nslab) {
    // next slab of the same rows: only the offset and, for the last slab, the length change
    const int slab = c.q8 ? kQ8SlabBlocks : kQ4SlabBlocks;
    const int blk = c.q8 ? 34 : 144;
    if (c.src) c.src += slab * blk;
    c.nch = min(slab, c.bpr - c.s * slab) * blk / 16;
  } else {
    c.s = 0;
    ++c.grp;
    cursor_slot(c, lane);
  }
}

FAK_DEV void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

// The whole warp copies one stage into `buf` and commits one cp.async group.
// Lane l copies row slot l / kLanesPerSlot, 16-byte chunks t, t + kLanesPerSlot, ...
// (t = l % kLanesPerSlot), so per-lane addresses advance by constants.
__device__ __forceinline__ void issue_stage(const Cursor& c, int lane, uint8_t* buf) {
  const int r = lane / kLanesPerSlot, t = lane % kLanesPerSlot;
  if (c.src) {
    uint8_t* dst = buf + r * (c.q8 ? kQ8StageRow : kQ4StageRow);
#pragma unroll
    for (int i = 0; i < (72 + kLanesPerSlot - 1) / kLanesPerSlot; ++i) {
      const int ch = t + kLanesPerSlot * i;
      if (ch < c.nch) cp_async16(dst + 16 * ch, c.src + 16 * ch);
    }
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
}

// Warm L2 with a stage's rows (the first lane of each row slot).
__device__ __forceinline__ void prefetch_stage_l2(const Cursor& c, int lane) {
  if (lane % kLanesPerSlot == 0 && c.src)
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(c.src), "r"((uint32_t)(c.nch * 16)) : "memory");
}

// ------------------------------------------------------------------ x preparation
// Quantize x (optionally RMS-normalized) into the limb records in shared memory.
constexpr int kMaxSbPerWarp = (kMaxSuper + kNumConsumerWarps - 1) / kNumConsumerWarps;
constexpr int kSbBatch = 2;  // super-blocks whose loads are in flight together

// An untagged x (the caller's vector, or a step after a grid-wide wait) is read
// with L1-cached loads: in a multi-step launch they follow the grid-wide
// acquire, so no line of an earlier step's x can be served stale.  A tagged x
// (F_TAGIN) is read from L2 and polled until every value carries the expected
// version tag; a poll that outlasts the timeout records FAK_ERR_TIMEOUT and
// returns false.  One pass over x: every load is issued first, then each
// super-block is quantized and the warp's share of sum(x^2) is left in
// red[cw].  The RMSNorm factor is a common scale of the whole vector, so it is
// applied to the row results in the epilogue instead (the per-super-block
// power-of-two scales keep the same relative precision either way).
template <bool I8>
__device__ bool prepare_x(const EngOp& op, const EngParams& P, uint8_t* smem, float* red, int cw, int lane,
                          volatile int* abort) {
  // int8 activations (the variant of the pages' int8-SDOT decode GEMV) for Q4_K steps only
  const bool i8 = I8 && op.kind != OP_Q8;
  const float* x = op.x;
  const int nsb = op.K / 256;
  uint8_t* xq = smem + kOffX;
  float* xS = reinterpret_cast<float*>(smem + kOffS);
  float* xsc = reinterpret_cast<float*>(smem + kOffScale);
  float ss = 0.0f;
  const bool tagged = op.flags & F_TAGIN;
  const uint32_t want = tag_in_par(op.tags) ^ ((P.flip >> tag_in_buf(op.tags)) & 1u);
  // the later batches' lines, all requested from L2 now so that their loads hit L1
  if (!tagged) {
#pragma unroll
    for (int k = kSbBatch; k < kMaxSbPerWarp; ++k) {
      const int sb = cw + k * kNumConsumerWarps;
      if (sb < nsb) asm volatile("prefetch.global.L1 [%0];" ::"l"(x + sb * 256 + lane * 8));
    }
  }
#pragma unroll 1
  for (int k0 = 0; k0 < kMaxSbPerWarp; k0 += kSbBatch) {
  float4 va[kSbBatch], vb[kSbBatch];
#pragma unroll
  for (int k = 0; k < kSbBatch; ++k) {
    const int sb = cw + (k0 + k) * kNumConsumerWarps;
    if (sb < nsb) {
      const float* src = x + sb * 256 + lane * 8;
      if (tagged) {
        va[k] = ld_relaxed_f4(src);
        vb[k] = ld_relaxed_f4(src + 4);
      } else {
        va[k] = __ldca(reinterpret_cast<const float4*>(src));
        vb[k] = __ldca(reinterpret_cast<const float4*>(src + 4));
      }
    }
  }
  if (tagged) {
    // poll the super-blocks that still hold an older version until all carry the expected tag
    uint64_t t0 = 0;
    for (uint32_t it = 0;; ++it) {
      bool all = true;
#pragma unroll
      for (int k = 0; k < kSbBatch; ++k) {
        const int sb = cw + (k0 + k) * kNumConsumerWarps;
        if (sb < nsb && !__all_sync(0xffffffffu, stale8(va[k], vb[k], want) == 0u)) {
          all = false;
          const float* src = x + sb * 256 + lane * 8;
          va[k] = ld_relaxed_f4(src);
          vb[k] = ld_relaxed_f4(src + 4);
        }
      }
      if (all) {
#pragma unroll
        for (int k = 0; k < kSbBatch; ++k) {
          va[k] = untag4(va[k]);
          vb[k] = untag4(vb[k]);
        }
        break;
      }
      if (*abort) return false;
      if (it == 0) {
        t0 = globaltimer_ns();
      } else if (globaltimer_ns() - t0 > P.timeout_ns) {
        set_error(P, FAK_ERR_TIMEOUT, abort);
        return false;
      }
      __nanosleep(64);
    }
  }
#pragma unroll
  for (int k = 0; k < kSbBatch; ++k) {
    const int sb = cw + (k0 + k) * kNumConsumerWarps;
    if (sb >= nsb) break;
    const float v[8] = {va[k].x, va[k].y, va[k].z, va[k].w, vb[k].x, vb[k].y, vb[k].z, vb[k].w};
    if (i8) {
      // per 32-element sub-block (four lanes): d = max|x| / 127, X = rint(x * (127 / max|x|)),
      // one signed byte each; the dot then sums q * X exactly and scales by d
      float am8 = 0.0f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        am8 = fmaxf(am8, fabsf(v[i]));
        ss = fmaf(v[i], v[i], ss);
      }
      am8 = fmaxf(am8, __shfl_xor_sync(0xffffffffu, am8, 1));
      am8 = fmaxf(am8, __shfl_xor_sync(0xffffffffu, am8, 2));
      const float qs = am8 > 0.0f ? 127.0f / am8 : 0.0f;
      const float dsub = am8 / 127.0f;
      int Xi[8], xs = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        Xi[i] = max(-127, min(127, __float2int_rn(v[i] * qs)));
        xs += Xi[i];
      }
      const uint32_t w0 = __byte_perm(__byte_perm(Xi[0], Xi[1], 0x0040), __byte_perm(Xi[2], Xi[3], 0x0040), 0x5410);
      const uint32_t w1 = __byte_perm(__byte_perm(Xi[4], Xi[5], 0x0040), __byte_perm(Xi[6], Xi[7], 0x0040), 0x5410);
      const int j = lane >> 2;  // sub-block
      uint8_t* grec = xq + sb * kSuperBytes + (j >> 1) * kGroupRec;
      *reinterpret_cast<uint2*>(grec + (j & 1) * 96 + (lane & 3) * 8) = make_uint2(w0, w1);
      xs += __shfl_xor_sync(0xffffffffu, xs, 1);
      xs += __shfl_xor_sync(0xffffffffu, xs, 2);
      if ((lane & 3) == 0) {
        reinterpret_cast<float*>(grec + 32)[j & 1] = dsub;  // the second limb's slot is free here
        xS[sb * 8 + j] = dsub * (float)xs;
      }
      continue;
    }
    float am = 0.0f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      am = fmaxf(am, fabsf(v[i]));
      ss = fmaf(v[i], v[i], ss);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, o));
    const uint32_t eb = (__float_as_uint(am) >> 23) & 0xFF;  // am in [2^(eb-127), 2^(eb-126))
    float f = 0.0f, sx = 0.0f;
    if (eb >= 22) {
      f = __uint_as_float((275u - eb) << 23);  // 2^(148-eb): |v*f| < 2^22
      sx = __uint_as_float((eb - 21u) << 23);  // 1/f
    }
    // X = rint(v * f) from one FMA: v * f is exact (f is a power of two) and
    // |v * f| < 2^22, so v * f + 1.5 * 2^23 lands in [2^23, 2^24), where floats
    // are the integers, rounded to nearest even once; its bits are
    // X + 0x4B400000.  Bytes 0 and 1 of the bits are X's; byte 2 is X's signed
    // top byte plus 64.
    uint32_t B[8];
    uint32_t bsum = 0;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      B[i] = __float_as_uint(fmaf(v[i], f, 12582912.0f));
      bsum += B[i];
    }
    const int xsum_own = (int)(bsum - 8u * 0x4B400000u);  // exact: |sum X| < 2^25
    uint32_t p0[2], p1[2], p2[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint32_t* b4 = B + 4 * h;
      const uint32_t t01 = __byte_perm(b4[0], b4[1], 0x5140), t23 = __byte_perm(b4[2], b4[3], 0x5140);
      p0[h] = __byte_perm(t01, t23, 0x5410);
      p1[h] = __byte_perm(t01, t23, 0x7632);
      const uint32_t u = __byte_perm(__byte_perm(b4[0], b4[1], 0x0062), __byte_perm(b4[2], b4[3], 0x0062), 0x5410);
      // per byte: (X >> 16) + 64 in [0, 128) -> X >> 16 as a two's-complement byte
      const uint32_t y = u ^ 0x40404040u;
      p2[h] = y | ((y << 1) & 0x80808080u);
    }
    int xsum = xsum_own;
    const int j = lane >> 2;  // sub-block
    uint8_t* rec = xq + sb * kSuperBytes + (j >> 1) * kGroupRec + (j & 1) * 96 + (lane & 3) * 8;
    *reinterpret_cast<uint2*>(rec) = make_uint2(p0[0], p0[1]);
    *reinterpret_cast<uint2*>(rec + 32) = make_uint2(p1[0], p1[1]);
    *reinterpret_cast<uint2*>(rec + 64) = make_uint2(p2[0], p2[1]);
    xsum += __shfl_xor_sync(0xffffffffu, xsum, 1);
    xsum += __shfl_xor_sync(0xffffffffu, xsum, 2);
    if ((lane & 3) == 0) xS[sb * 8 + (lane >> 2)] = sx * (float)xsum;
    if (lane == 0) xsc[sb] = sx;
  }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  if (lane == 0) red[cw] = ss;
  return true;
}

// The RMSNorm factor from the warps' partial sums (same order in every thread
// of every CTA, so every CTA gets the bitwise same factor).
__device__ __forceinline__ float norm_factor(const EngOp& op, const float* red) {
  if (!(op.flags & F_NORM)) return 1.0f;
  float tot = 0.0f;
#pragma unroll
  for (int w = 0; w < kNumConsumerWarps; ++w) tot += red[w];
  return 1.0f / sqrtf(tot / (float)op.K + op.eps);
}

// ------------------------------------------------------------------ Q4_K slab
// One stage: up to 8 row slots x up to 8 blocks.  Lane (b, g) = (lane/4, lane%4)
// covers block b of the slab and its 64-weight group g (sub-blocks 2g, 2g+1).
// Row slots are computed in pairs without branches (slots past the valid rows
// hold stale bytes; their sums are never written).
struct XRegs {
  uint32_t A0[8], A1[8], A2[8], B0[8], B1[8], B2[8];
  float SA, SB, sx16;
};

// The x limbs of block jb, 64-weight group g, from the shared-memory records.
__device__ __forceinline__ void load_xregs(const uint8_t* smem, int jb, int g, XRegs& x) {
  const uint8_t* rec = smem + kOffX + jb * kSuperBytes + g * kGroupRec;
  const uint4* r0 = reinterpret_cast<const uint4*>(rec);
  const uint4* r1 = reinterpret_cast<const uint4*>(rec + 96);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint4 t;
    t = r0[0 + h]; x.A0[4 * h] = t.x; x.A0[4 * h + 1] = t.y; x.A0[4 * h + 2] = t.z; x.A0[4 * h + 3] = t.w;
    t = r0[2 + h]; x.A1[4 * h] = t.x; x.A1[4 * h + 1] = t.y; x.A1[4 * h + 2] = t.z; x.A1[4 * h + 3] = t.w;
    t = r0[4 + h]; x.A2[4 * h] = t.x; x.A2[4 * h + 1] = t.y; x.A2[4 * h + 2] = t.z; x.A2[4 * h + 3] = t.w;
    t = r1[0 + h]; x.B0[4 * h] = t.x; x.B0[4 * h + 1] = t.y; x.B0[4 * h + 2] = t.z; x.B0[4 * h + 3] = t.w;
    t = r1[2 + h]; x.B1[4 * h] = t.x; x.B1[4 * h + 1] = t.y; x.B1[4 * h + 2] = t.z; x.B1[4 * h + 3] = t.w;
    t = r1[4 + h]; x.B2[4 * h] = t.x; x.B2[4 * h + 1] = t.y; x.B2[4 * h + 2] = t.z; x.B2[4 * h + 3] = t.w;
  }
  const float* xS = reinterpret_cast<const float*>(smem + kOffS);
  x.SA = xS[jb * 8 + 2 * g];
  x.SB = xS[jb * 8 + 2 * g + 1];
  x.sx16 = reinterpret_cast<const float*>(smem + kOffScale)[jb] * 0.0625f;
}

// R consecutive row slots starting at `base` (a block of the first slot), one
// 64-weight group g of that block, accumulated into acc[0..R).
template <int R>
__device__ __forceinline__ void q4k_rows(const uint8_t* base, int g, const XRegs& x, float (&acc)[R]) {
  const uint32_t sel = (uint32_t)(2 * g) | ((uint32_t)(2 * g + 1) << 4);
  // all row slots at once: 6R independent DP4A chains per quant word
  uint4 h[R], qa[R], qb[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    h[r] = *reinterpret_cast<const uint4*>(base + r * kQ4StageRow);
    qa[r] = *reinterpret_cast<const uint4*>(base + r * kQ4StageRow + 16 + 32 * g);
    qb[r] = *reinterpret_cast<const uint4*>(base + r * kQ4StageRow + 32 + 32 * g);
  }
  uint32_t a0[R], a1[R], b0[R], b1[R];
  int a2[R], b2[R];
#pragma unroll
  for (int r = 0; r < R; ++r) a0[r] = a1[r] = b0[r] = b1[r] = 0, a2[r] = b2[r] = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint32_t w = u < 4 ? (u == 0 ? qa[r].x : u == 1 ? qa[r].y : u == 2 ? qa[r].z : qa[r].w)
                               : (u == 4 ? qb[r].x : u == 5 ? qb[r].y : u == 6 ? qb[r].z : qb[r].w);
      const uint32_t lo = w & 0x0F0F0F0Fu, hi = w & 0xF0F0F0F0u;
      a0[r] = dp4a_uu(lo, x.A0[u], a0[r]);
      a1[r] = dp4a_uu(lo, x.A1[u], a1[r]);
      a2[r] = dp4a_us(lo, x.A2[u], a2[r]);
      b0[r] = dp4a_uu(hi, x.B0[u], b0[r]);
      b1[r] = dp4a_uu(hi, x.B1[u], b1[r]);
      b2[r] = dp4a_us(hi, x.B2[u], b2[r]);
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint32_t sc_lo = h[r].y & 0x3F3F3F3Fu;
    const uint32_t m_lo = h[r].z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (h[r].w & 0x0F0F0F0Fu) | ((h[r].y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((h[r].w >> 4) & 0x0F0F0F0Fu) | ((h[r].z >> 2) & 0x30303030u);
    const uint32_t scp = prmt(sc_lo, sc_hi, sel);
    const uint32_t mp = prmt(m_lo, m_hi, sel);
    const int scA16 = (int)(scp & 0xFF) << 4, scB = (int)((scp >> 8) & 0xFF);
    const float mA = (float)(mp & 0xFF), mB = (float)((mp >> 8) & 0xFF);
    const float d = half_bits_to_float(h[r].x & 0xFFFF), dmin = half_bits_to_float(h[r].x >> 16);
    const int J0 = (int)a0[r] * scA16 + (int)b0[r] * scB;
    const int J1 = (int)a1[r] * scA16 + (int)b1[r] * scB;
    const int J2 = a2[r] * scA16 + b2[r] * scB;
    const float Jf = fmaf((float)J2, 65536.0f, fmaf((float)J1, 256.0f, (float)J0));
    const float mterm = fmaf(mA, x.SA, mB * x.SB);
    acc[r] = fmaf(d * x.sx16, Jf, fmaf(-dmin, mterm, acc[r]));
  }
}

// int8-activation form: the x bytes of sub-blocks 2g and 2g+1, their scales and sums.
struct XRegs8 {
  uint32_t A[8], B[8];
  float dA, dB, SA, SB;
};

__device__ __forceinline__ void load_xregs8(const uint8_t* smem, int jb, int g, XRegs8& x) {
  const uint8_t* rec = smem + kOffX + jb * kSuperBytes + g * kGroupRec;
  const uint4* r0 = reinterpret_cast<const uint4*>(rec);
  const uint4* r1 = reinterpret_cast<const uint4*>(rec + 96);
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint4 t = r0[h];
    x.A[4 * h] = t.x; x.A[4 * h + 1] = t.y; x.A[4 * h + 2] = t.z; x.A[4 * h + 3] = t.w;
    t = r1[h];
    x.B[4 * h] = t.x; x.B[4 * h + 1] = t.y; x.B[4 * h + 2] = t.z; x.B[4 * h + 3] = t.w;
  }
  const float2 dd = *reinterpret_cast<const float2*>(rec + 32);
  x.dA = dd.x;
  x.dB = dd.y;
  const float* xS = reinterpret_cast<const float*>(smem + kOffS);
  x.SA = xS[jb * 8 + 2 * g];
  x.SB = xS[jb * 8 + 2 * g + 1];
}

template <int R>
__device__ __forceinline__ void q4k_rows8(const uint8_t* base, int g, const XRegs8& x, float (&acc)[R]) {
  const uint32_t sel = (uint32_t)(2 * g) | ((uint32_t)(2 * g + 1) << 4);
  uint4 h[R], qa[R], qb[R];
#pragma unroll
  for (int r = 0; r < R; ++r) {
    h[r] = *reinterpret_cast<const uint4*>(base + r * kQ4StageRow);
    qa[r] = *reinterpret_cast<const uint4*>(base + r * kQ4StageRow + 16 + 32 * g);
    qb[r] = *reinterpret_cast<const uint4*>(base + r * kQ4StageRow + 32 + 32 * g);
  }
  int a[R], b[R];
#pragma unroll
  for (int r = 0; r < R; ++r) a[r] = b[r] = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const uint32_t w = u < 4 ? (u == 0 ? qa[r].x : u == 1 ? qa[r].y : u == 2 ? qa[r].z : qa[r].w)
                               : (u == 4 ? qb[r].x : u == 5 ? qb[r].y : u == 6 ? qb[r].z : qb[r].w);
      a[r] = dp4a_us(w & 0x0F0F0F0Fu, x.A[u], a[r]);
      b[r] = dp4a_us(w & 0xF0F0F0F0u, x.B[u], b[r]);  // 16 q: the scale below divides by 16
    }
  }
#pragma unroll
  for (int r = 0; r < R; ++r) {
    const uint32_t sc_lo = h[r].y & 0x3F3F3F3Fu;
    const uint32_t m_lo = h[r].z & 0x3F3F3F3Fu;
    const uint32_t sc_hi = (h[r].w & 0x0F0F0F0Fu) | ((h[r].y >> 2) & 0x30303030u);
    const uint32_t m_hi = ((h[r].w >> 4) & 0x0F0F0F0Fu) | ((h[r].z >> 2) & 0x30303030u);
    const uint32_t scp = prmt(sc_lo, sc_hi, sel);
    const uint32_t mp = prmt(m_lo, m_hi, sel);
    const int scA16 = (int)(scp & 0xFF) << 4, scB = (int)((scp >> 8) & 0xFF);
    const float mA = (float)(mp & 0xFF), mB = (float)((mp >> 8) & 0xFF);
    const float d = half_bits_to_float(h[r].x & 0xFFFF), dmin = half_bits_to_float(h[r].x >> 16);
    const float Jf = fmaf((float)(a[r] * scA16), x.dA, (float)(b[r] * scB) * x.dB);
    const float mterm = fmaf(mA, x.SA, mB * x.SB);
    acc[r] = fmaf(d * 0.0625f, Jf, fmaf(-dmin, mterm, acc[r]));
  }
}

__device__ __forceinline__ void q4k_slab8(const uint8_t* stage, const uint8_t* smem, int jb0, int nb, int lane,
                                          float (&acc)[kSlots]) {
  const int g = lane & 3;
  XRegs8 x;
  if (nb > kQ4SlabBlocks / 2) {
    const int b = lane >> 2;
    if (b >= nb) return;
    load_xregs8(smem, jb0 + b, g, x);
    q4k_rows8<kSlots>(stage + b * 144, g, x, acc);
  } else {
    const int b = (lane >> 2) & 3, hr = lane >> 4;
    if (b >= nb) return;
    load_xregs8(smem, jb0 + b, g, x);
    float t[2] = {hr ? acc[2] : acc[0], hr ? acc[3] : acc[1]};
    q4k_rows8<2>(stage + b * 144 + 2 * hr * kQ4StageRow, g, x, t);
    acc[0] = hr ? acc[0] : t[0];
    acc[1] = hr ? acc[1] : t[1];
    acc[2] = hr ? t[0] : acc[2];
    acc[3] = hr ? t[1] : acc[3];
  }
}

// A slab of more than four blocks: lane (b, g) = (lane/4, lane%4) takes its
// (block, group) pair for all four row slots.  A slab of at most four blocks
// (the last slab of a row whose length is not a multiple of eight blocks) has
// only 16 pairs, so the upper half-warp takes row slots 2 and 3 of the same
// pairs and each lane computes two rows: such a slab costs half a full one
// instead of a full one with half the lanes idle.  Row slots past the valid
// rows hold stale bytes; their sums are never written.
__device__ __forceinline__ void q4k_slab(const uint8_t* stage, const uint8_t* smem, int jb0, int nb, int lane,
                                         float (&acc)[kSlots]) {
  const int g = lane & 3;
  XRegs x;
  if (nb > kQ4SlabBlocks / 2) {
    const int b = lane >> 2;
    if (b >= nb) return;
    load_xregs(smem, jb0 + b, g, x);
    q4k_rows<kSlots>(stage + b * 144, g, x, acc);
  } else {
    const int b = (lane >> 2) & 3, hr = lane >> 4;
    if (b >= nb) return;
    load_xregs(smem, jb0 + b, g, x);
    float t[2] = {hr ? acc[2] : acc[0], hr ? acc[3] : acc[1]};
    q4k_rows<2>(stage + b * 144 + 2 * hr * kQ4StageRow, g, x, t);
    acc[0] = hr ? acc[0] : t[0];
    acc[1] = hr ? acc[1] : t[1];
    acc[2] = hr ? t[0] : acc[2];
    acc[3] = hr ? t[1] : acc[3];
  }
}

// ------------------------------------------------------------------ Q8_0 slab
// One stage: up to 8 row slots x up to 32 blocks; lane l covers block l.
__device__ __forceinline__ float q8_row(const uint8_t* rowbase, int lane, const uint32_t (&P0)[8],
                                        const uint32_t (&P1)[8], const uint32_t (&P2)[8], float sx, uint32_t sel,
                                        int odd, float acc) {
  const uint32_t* wp = reinterpret_cast<const uint32_t*>(rowbase + ((34 * lane) & ~3));
  uint32_t w[9];
#pragma unroll
  for (int u = 0; u < 9; ++u) w[u] = wp[u];
  const float d = half_bits_to_float(odd ? (w[0] >> 16) : (w[0] & 0xFFFF));
  int i0 = 0, i1 = 0, i2 = 0;
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    const uint32_t q = prmt(w[u], w[u + 1], sel);
    i0 = dp4a_su(q, P0[u], i0);
    i1 = dp4a_su(q, P1[u], i1);
    i2 = dp4a_ss(q, P2[u], i2);
  }
  const float Jf = fmaf((float)i2, 65536.0f, fmaf((float)i1, 256.0f, (float)i0));
  return fmaf(d * sx, Jf, acc);
}

__device__ __forceinline__ void q8_slab(const uint8_t* stage, const uint8_t* smem, int cb0, int nb, int nslots,
                                        int lane, float acc[kSlots]) {
  if (lane >= nb) return;
  const int cb = cb0 + lane;
  const uint4* rec = reinterpret_cast<const uint4*>(smem + kOffX + (cb >> 3) * kSuperBytes +
                                                    ((cb & 7) >> 1) * kGroupRec + (cb & 1) * 96);
  uint32_t P0[8], P1[8], P2[8];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint4 t;
    t = rec[0 + h]; P0[4 * h] = t.x; P0[4 * h + 1] = t.y; P0[4 * h + 2] = t.z; P0[4 * h + 3] = t.w;
    t = rec[2 + h]; P1[4 * h] = t.x; P1[4 * h + 1] = t.y; P1[4 * h + 2] = t.z; P1[4 * h + 3] = t.w;
    t = rec[4 + h]; P2[4 * h] = t.x; P2[4 * h + 1] = t.y; P2[4 * h + 2] = t.z; P2[4 * h + 3] = t.w;
  }
  const float sx = reinterpret_cast<const float*>(smem + kOffScale)[cb >> 3];
  const int odd = lane & 1;  // 34*lane % 4 == 2*odd: odd lanes have aligned quants
  const uint32_t sel = odd ? 0x7654u : 0x5432u;
#pragma unroll
  for (int rp = 0; rp < kSlots / 2; ++rp) {
    if (2 * rp >= nslots) break;
    acc[2 * rp] = q8_row(stage + (2 * rp) * kQ8StageRow, lane, P0, P1, P2, sx, sel, odd, acc[2 * rp]);
    acc[2 * rp + 1] = q8_row(stage + (2 * rp + 1) * kQ8StageRow, lane, P0, P1, P2, sx, sel, odd, acc[2 * rp + 1]);
  }
}

__device__ __forceinline__ void better(float v, int idx, float& bv, int& bi) {
  if (idx < 0 || v != v) return;
  if (bi < 0 || v > bv || (v == bv && idx < bi)) {
    bv = v;
    bi = idx;
  }
}

// The step's output fields, cached in registers once per step.
struct EmitInfo {
  float* y0;
  float* y1;
  float* y2;
  int se0, se1;  // segment row ends
  int flags;
  float rn;      // RMSNorm factor (1 without F_NORM)
  uint32_t tg;   // F_TAGOUT: the version tag of segment s in bit s
  bool pair;
};

__device__ __forceinline__ EmitInfo emit_info(const EngOp& op, float rn, unsigned flip) {
  EmitInfo E;
  E.y0 = op.y[0];
  E.y1 = op.y[1];
  E.y2 = op.y[2];
  E.se0 = op.nseg > 1 ? (int)op.seg_end[0] : 0x7fffffff;
  E.se1 = op.nseg > 2 ? (int)op.seg_end[1] : 0x7fffffff;
  E.flags = op.flags;
  E.rn = rn;
  E.tg = 0;
#pragma unroll
  for (int sgi = 0; sgi < 3; ++sgi)
    E.tg |= (tag_out_par(op.tags, sgi) ^ ((flip >> tag_out_buf(op.tags, sgi)) & 1u)) << sgi;
  E.pair = op.kind == OP_Q4K_SWIGLU;
  return E;
}

// Final value of output row `row`: RMSNorm factor, then the SwiGLU pair
// (gate v, up v_up), or residual add + store, or logits + argmax candidate.
__device__ __forceinline__ float* out_ptr(const EmitInfo& E, int row) {
  return row < E.se0 ? E.y0 + row : (row < E.se1 ? E.y1 + (row - E.se0) : E.y2 + (row - E.se1));
}

// The residual of output row `row` (0 without F_RESID): a tagged output is read back untagged.
__device__ __forceinline__ float resid_load(const EmitInfo& E, int row) {
  if (!(E.flags & F_RESID)) return 0.0f;
  const float r = ld_cg_f(out_ptr(E, row));
  return (E.flags & F_TAGOUT) ? untag(r) : r;
}

// The residual as loaded (still tagged where the buffer is), for a load issued well before its use:
// nothing touches the value until resid_ready, so the load's round trip overlaps the step's compute.
__device__ __forceinline__ float resid_load_raw(const EmitInfo& E, int row) {
  return (E.flags & F_RESID) ? ld_cg_f(out_ptr(E, row)) : 0.0f;
}
__device__ __forceinline__ float resid_ready(const EmitInfo& E, float raw) {
  return (E.flags & F_TAGOUT) ? untag(raw) : raw;
}

__device__ __forceinline__ void emit(const EmitInfo& E, const EngParams& P, int row, float v, float v_up, float& wbv,
                                     int& wbi, float res) {
  if (E.pair) {
    const float gt = v * E.rn, up = v_up * E.rn;
    const float a = gt / (1.0f + expf(-gt)) * up;
    if (E.flags & F_TAGOUT)
      st_tagged(E.y0 + row, a, E.tg & 1u);
    else
      E.y0[row] = a;
    return;
  }
  float* yp = out_ptr(E, row);
  const float val = v * E.rn + res;
  if (E.flags & F_ARGMAX) {
    if (P.logits) P.logits[row] = val;
    better(val, row, wbv, wbi);
  } else if (E.flags & F_TAGOUT) {
    const int sgi = row < E.se0 ? 0 : (row < E.se1 ? 1 : 2);
    st_tagged(yp, val, (E.tg >> sgi) & 1u);
  } else {
    *yp = val;
  }
}

// Sum the four row slots' partial sums over the warp with a fixed 6-shuffle
// transpose: afterwards lanes 8r..8r+7 hold row r's total (lane 8r's value is
// the one used, so results are bitwise reproducible).
__device__ __forceinline__ float reduce4(const float (&acc)[kSlots], int lane) {
  const bool h16 = lane & 16, h8 = lane & 8;
  float k0 = h16 ? acc[2] : acc[0], k1 = h16 ? acc[3] : acc[1];
  const float s0 = h16 ? acc[0] : acc[2], s1 = h16 ? acc[1] : acc[3];
  k0 += __shfl_xor_sync(0xffffffffu, s0, 16);
  k1 += __shfl_xor_sync(0xffffffffu, s1, 16);
  float keep = h8 ? k1 : k0;
  const float send = h8 ? k0 : k1;
  keep += __shfl_xor_sync(0xffffffffu, send, 8);
  keep += __shfl_xor_sync(0xffffffffu, keep, 4);
  keep += __shfl_xor_sync(0xffffffffu, keep, 2);
  keep += __shfl_xor_sync(0xffffffffu, keep, 1);
  return keep;
}

// ------------------------------------------------------------------ mixer steps
// One CTA per head; the other CTAs go straight on to the next step (which polls
// this step's tagged output).  384 threads.  Scratch in the x-record area of
// shared memory (free between the previous step's last CTA barrier and the next
// step's x preparation).

// Up to N tagged values at once: every load is in flight together, then only the stale ones are
// read again until all carry their expected tag (bounded like every wait).  use[k] false: slot k
// is skipped and v[k] left as it is.
template <int N>
__device__ __forceinline__ bool poll_n(const float* const (&p)[N], const uint32_t (&want)[N], const bool (&use)[N],
                                       float (&v)[N], const EngParams& P, volatile int* abort) {
  uint32_t stale = 0;
#pragma unroll
  for (int k = 0; k < N; ++k)
    if (use[k]) v[k] = ld_relaxed_f(p[k]);
#pragma unroll
  for (int k = 0; k < N; ++k)
    if (use[k] && (__float_as_uint(v[k]) & 1u) != want[k]) stale |= 1u << k;
  uint64_t t0 = 0;
  for (uint32_t it = 0; stale; ++it) {
    if (*abort) return false;
    if (it == 0) {
      t0 = globaltimer_ns();
    } else if (globaltimer_ns() - t0 > P.timeout_ns) {
      set_error(P, FAK_ERR_TIMEOUT, abort);
      return false;
    }
    __nanosleep(64);
#pragma unroll
    for (int k = 0; k < N; ++k)
      if ((stale >> k) & 1u) v[k] = ld_relaxed_f(p[k]);
#pragma unroll
    for (int k = 0; k < N; ++k)
      if (((stale >> k) & 1u) && (__float_as_uint(v[k]) & 1u) == want[k]) stale &= ~(1u << k);
  }
#pragma unroll
  for (int k = 0; k < N; ++k)
    if (use[k]) v[k] = untag(v[k]);
  return true;
}

// Sum over the first `nw` warps' values of `v` (block-wide; every thread gets the same sum,
// summed in warp order).  scratch: at least nw floats; the caller's threads all call it.
__device__ __forceinline__ float block_sum(float v, int nw, float* scratch, int ctid) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((ctid & 31) == 0 && (ctid >> 5) < nw) scratch[ctid >> 5] = v;
  named_bar_sync(1, kConsumerThreads);
  float t = 0.0f;
  for (int w = 0; w < nw; ++w) t += scratch[w];
  named_bar_sync(1, kConsumerThreads);
  return t;
}

__device__ __forceinline__ float silu_f(float x) { return x / (1.0f + expf(-x)); }

// Gated DeltaNet step of value head h = blockIdx.x: the causal conv of its q, k, v channels,
// the L2 norms, the gates, the delta-rule update of S_h (dk x dv = 128 x 128, three threads per
// column, 43 rows each) and the gated RMSNorm of o_h.
__device__ void gdn_step(const EngParams& P, const EngOp& op, uint8_t* smem, int ctid, volatile int* abort) {
  const MixDesc& M = *reinterpret_cast<const MixDesc*>(op.x);
  const int h = blockIdx.x;
  const int nv = M.nv, nk = M.nk;
  if (h >= nv) return;
  const int ratio = nv / nk, kh = h / ratio;
  const int conv_dim = 2 * nk * 128 + nv * 128;
  const uint32_t want = tag_in_par(op.tags) ^ ((P.flip >> tag_in_buf(op.tags)) & 1u);
  const uint32_t otag = tag_out_par(op.tags, 0) ^ ((P.flip >> tag_out_buf(op.tags, 0)) & 1u);
  const int par = (P.flip >> 8) & 1;
  float* y = reinterpret_cast<float*>(smem + kOffX);  // [384] conv outputs: q | k | v
  float* zs = y + 384;                                 // [128] silu(z)
  float* part = zs + 128;                              // [3][128]
  float* scr = part + 384;                             // [16] reductions
  float* gates = scr + 16;                             // [2] beta, alpha
  // conv channel of this thread: q (key head kh), k (key head kh), v (value head h)
  const int c = ctid < 128 ? kh * 128 + ctid
                           : (ctid < 256 ? nk * 128 + kh * 128 + (ctid - 128) : 2 * nk * 128 + h * 128 + (ctid - 256));
  // What does not depend on this token's input is requested first, so that its latency overlaps
  // the wait for the in_proj output: the head's state (64 KB, written by the previous token and
  // long evicted from L2) is prefetched into L2; this thread's conv channel state and taps, the
  // gate parameters and the norm gain are loaded.
  const int j = ctid & 127, r = ctid >> 7;
  float* Sh = M.S + (size_t)h * 128 * 128;
  for (int line = ctid; line < 128 * 128 * 4 / 128; line += kConsumerThreads)
    asm volatile("prefetch.global.L2 [%0];" ::"l"(Sh + line * 32));
  const float* so = M.conv_state + ((size_t)par * conv_dim + c) * 3;
  const float4 w = *reinterpret_cast<const float4*>(M.conv_w + (size_t)c * 4);
  const float s0 = so[0], s1 = so[1], s2 = so[2];
  const float dtb = ctid == 0 ? M.dt_bias[h] : 0.0f, alog = ctid == 0 ? M.a_log[h] : 0.0f;
  const float nwj = ctid < 128 ? M.norm_w[j] : 0.0f;
  // the step's inputs, all in flight at once: the conv channel, z (warps 0-3), b and a (thread 0)
  const float* const pin[4] = {M.t + c, M.t + conv_dim + h * 128 + (ctid & 127), M.t + conv_dim + nv * 128 + h,
                               M.t + conv_dim + nv * 128 + nv + h};
  const uint32_t wants[4] = {want, want, want, want};
  const bool use[4] = {true, ctid < 128, ctid == 0, ctid == 0};
  float vin[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  poll_n<4>(pin, wants, use, vin, P, abort);
  const float xin = vin[0], zv = vin[1], bv = vin[2], av = vin[3];
  named_bar_sync(1, kConsumerThreads);
  if (*abort) return;
  {
    float* sn = M.conv_state + ((size_t)(par ^ 1) * conv_dim + c) * 3;
    const float acc = fmaf(w.w, xin, fmaf(w.z, s2, fmaf(w.y, s1, w.x * s0)));
    y[ctid] = silu_f(acc);
    // the q and k channels are shared by `ratio` value heads: the first one writes their new state
    if (ctid >= 256 || h % ratio == 0) {
      sn[0] = s1;
      sn[1] = s2;
      sn[2] = xin;
    }
    if (ctid < 128) zs[ctid] = silu_f(zv);
    if (ctid == 0) {
      gates[0] = 1.0f / (1.0f + expf(-bv));
      const float sp = av + dtb;
      const float soft = sp > 20.0f ? sp : log1pf(expf(sp));
      gates[1] = expf(-expf(alog) * soft);
    }
  }
  named_bar_sync(1, kConsumerThreads);
  // L2 norms of q (warps 0-3) and k (warps 4-7)
  const float yv = y[ctid];
  float sq = (ctid < 256) ? yv * yv : 0.0f;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sq += __shfl_xor_sync(0xffffffffu, sq, o);
  if ((ctid & 31) == 0) scr[ctid >> 5] = sq;
  named_bar_sync(1, kConsumerThreads);
  const float qq = (scr[0] + scr[1]) + (scr[2] + scr[3]);
  const float kk = (scr[4] + scr[5]) + (scr[6] + scr[7]);
  const float rq = 1.0f / sqrtf(qq + M.eps) / sqrtf(128.0f), rk = 1.0f / sqrtf(kk + M.eps);
  const float beta = gates[0], alpha = gates[1];
  // state update: column j, rows [43 r, 43 r + 43)
  float sreg[43];
  float kv = 0.0f;
#pragma unroll
  for (int ii = 0; ii < 43; ++ii) {
    const int i = 43 * r + ii;
    if (i < 128) {
      sreg[ii] = alpha * Sh[i * 128 + j];
      kv = fmaf(sreg[ii], y[128 + i] * rk, kv);
    }
  }
  part[r * 128 + j] = kv;
  named_bar_sync(1, kConsumerThreads);
  const float kvj = (part[j] + part[128 + j]) + part[256 + j];
  const float delta = beta * (y[256 + j] - kvj);
  named_bar_sync(1, kConsumerThreads);  // every thread has read part[] before it is reused
  float o = 0.0f;
#pragma unroll
  for (int ii = 0; ii < 43; ++ii) {
    const int i = 43 * r + ii;
    if (i < 128) {
      const float sv = fmaf(y[128 + i] * rk, delta, sreg[ii]);
      Sh[i * 128 + j] = sv;
      o = fmaf(sv, y[i] * rq, o);
    }
  }
  part[r * 128 + j] = o;
  named_bar_sync(1, kConsumerThreads);
  const float oj = (part[j] + part[128 + j]) + part[256 + j];
  // gated RMSNorm over the head (warps 0-3 hold the 128 columns)
  const float ss = block_sum(ctid < 128 ? oj * oj : 0.0f, 4, scr + 8, ctid);
  if (ctid < 128) {
    const float rn = 1.0f / sqrtf(ss / 128.0f + M.eps);
    st_tagged(M.out + h * 128 + j, oj * rn * nwj * zs[j], otag);
  }
}

// q, k, v, gate (4 x 256), reduction scratch (32) and the scores (max_ctx <= 8192) fit in the x-limb
// region the step reuses
static_assert((4 * 256 + 32 + 8192) * 4 <= kMaxSuper * kSuperBytes, "attention scratch exceeds the x-limb region");

// Gated attention step of query head h = blockIdx.x at position *P.pos: qk-norm, RoPE, the
// KV-cache append (by the first query head of each KV group), softmax over positions 0..pos
// and the sigmoid output gate.
__device__ void attn_step(const EngParams& P, const EngOp& op, uint8_t* smem, int ctid, volatile int* abort) {
  const MixDesc& M = *reinterpret_cast<const MixDesc*>(op.x);
  const int h = blockIdx.x;
  if (h >= M.nq) return;
  const int grp = M.nq / M.nkv, g = h / grp;
  const int pos = *P.pos;
  const uint32_t want = tag_in_par(op.tags) ^ ((P.flip >> tag_in_buf(op.tags)) & 1u);
  const uint32_t want_kv = 1u ^ ((P.flip >> 3) & 1u);  // every k / v slice: version 1 of its token
  const uint32_t otag = tag_out_par(op.tags, 0) ^ ((P.flip >> tag_out_buf(op.tags, 0)) & 1u);
  if (pos < 0 || pos >= M.max_ctx) {
    // past the cache: record the error, and still hand the next step a (zero) output so that the
    // token ends at once instead of in the readers' timeout; nothing is written to the cache
    if (ctid == 0) atomicCAS(P.err ? P.err : &g_fak_status, 0, FAK_ERR_DEVICE);
    if (ctid < 256) st_tagged(M.out + h * 256 + ctid, 0.0f, otag);
    return;
  }
  float* qs = reinterpret_cast<float*>(smem + kOffX);  // [256] normed, rotated q
  float* ks = qs + 256;                                // [256] normed, rotated k of this position
  float* vs = ks + 256;                                // [256]
  float* gs = vs + 256;                                // [256] sigmoid(gate)
  float* scr = gs + 256;                               // [32]
  float* sc = scr + 32;                                // [max_ctx] scores, then weights
  const int d = ctid;
  // q, gate, k and v of this position, all in flight at once
  const int dd = d & 255;
  const float* const pin[4] = {M.t + h * 512 + dd, M.t + h * 512 + 256 + dd, M.kin + g * 256 + dd,
                               M.vin + g * 256 + dd};
  const uint32_t wants[4] = {want, want, want_kv, want_kv};
  const bool use[4] = {d < 256, d < 256, d < 256, d < 256};
  float vin[4] = {0.0f, 0.0f, 0.0f, 0.0f};
  poll_n<4>(pin, wants, use, vin, P, abort);
  const float qv = vin[0], gv = vin[1], kv = vin[2], vv = vin[3];
  named_bar_sync(1, kConsumerThreads);
  if (*abort) return;
  const float sq = block_sum(d < 256 ? qv * qv : 0.0f, 8, scr, ctid);
  const float sk = block_sum(d < 256 ? kv * kv : 0.0f, 8, scr + 8, ctid);
  if (d < 256) {
    qs[d] = qv / sqrtf(sq / 256.0f + M.eps) * M.q_norm_w[d];
    ks[d] = kv / sqrtf(sk / 256.0f + M.eps) * M.k_norm_w[d];
    vs[d] = vv;
    gs[d] = 1.0f / (1.0f + expf(-gv));
  }
  named_bar_sync(1, kConsumerThreads);
  const int half = M.rot / 2;
  if (d < half) {
    // the angle pos * theta^(-2d/rot) in double precision (it reaches thousands of radians),
    // reduced modulo 2 pi in double; sine and cosine of the reduced angle in single precision
    const double ang = (double)pos * M.inv_freq[d];
    const double red = ang - 6.283185307179586 * rint(ang * 0.15915494309189535);
    float s, c;
    sincosf((float)red, &s, &c);
    const float q1 = qs[d], q2 = qs[d + half], k1 = ks[d], k2 = ks[d + half];
    qs[d] = q1 * c - q2 * s;
    qs[d + half] = q2 * c + q1 * s;
    ks[d] = k1 * c - k2 * s;
    ks[d + half] = k2 * c + k1 * s;
  }
  named_bar_sync(1, kConsumerThreads);
  float* kcp = M.kc + (size_t)g * M.max_ctx * 256;
  float* vcp = M.vc + (size_t)g * M.max_ctx * 256;
  if (h % grp == 0 && d < 256) {
    kcp[(size_t)pos * 256 + d] = ks[d];
    vcp[(size_t)pos * 256 + d] = vs[d];
  }
  // scores: warp w takes positions w, w + 12, ... (two at a time, their key rows loaded as two
  // float4 per lane); lane l dims 8l..8l+7; the current position's key comes from shared memory
  const int w = ctid >> 5, lane = ctid & 31;
#pragma unroll 2
  for (int sidx = w; sidx < pos; sidx += kNumConsumerWarps) {
    const float4* kr = reinterpret_cast<const float4*>(kcp + (size_t)sidx * 256 + lane * 8);
    const float4 k0 = __ldcg(kr), k1 = __ldcg(kr + 1);
    const float kk[8] = {k0.x, k0.y, k0.z, k0.w, k1.x, k1.y, k1.z, k1.w};
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc = fmaf(qs[lane * 8 + e], kk[e], acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) sc[sidx] = acc * 0.0625f;  // 1 / sqrt(256)
  }
  if (w == pos % kNumConsumerWarps) {
    float acc = 0.0f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc = fmaf(qs[lane * 8 + e], ks[lane * 8 + e], acc);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
    if (lane == 0) sc[pos] = acc * 0.0625f;
  }
  named_bar_sync(1, kConsumerThreads);
  float mx = -INFINITY;
  for (int sidx = ctid; sidx <= pos; sidx += kConsumerThreads) mx = fmaxf(mx, sc[sidx]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  if (lane == 0) scr[16 + w] = mx;
  named_bar_sync(1, kConsumerThreads);
  mx = scr[16];
  for (int ww = 1; ww < kNumConsumerWarps; ++ww) mx = fmaxf(mx, scr[16 + ww]);
  named_bar_sync(1, kConsumerThreads);
  float se = 0.0f;
  for (int sidx = ctid; sidx <= pos; sidx += kConsumerThreads) {
    const float e = expf(sc[sidx] - mx);
    sc[sidx] = e;
    se += e;
  }
  const float sum = block_sum(se, kNumConsumerWarps, scr, ctid);
  if (d < 256) {
    // the cached positions in order, sixteen loads in flight, then this position's own value
    float acc = 0.0f;
#pragma unroll 16
    for (int sidx = 0; sidx < pos; ++sidx) acc = fmaf(sc[sidx], __ldcg(vcp + (size_t)sidx * 256 + d), acc);
    acc = fmaf(sc[pos], vs[d], acc);
    st_tagged(M.out + h * 256 + d, acc / sum * gs[d], otag);
  }
}

// ------------------------------------------------------------------ the steps
// I8X: Q4_K steps take int8 activations (one scale per 32-element sub-block)
// instead of the exact three-limb form; Q8_0 steps are the same in both.
template <bool I8X>
__global__ void __launch_bounds__(kThreads, 1) engine_kernel(const __grid_constant__ EngParams P) {
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  const int ctid = threadIdx.x;
  const int cw = ctid >> 5, lane = ctid & 31;
  float* red = reinterpret_cast<float*>(smem + kOffMisc);          // [16]
  float* bestv = red + 16;                                          // [16]
  int* besti = reinterpret_cast<int*>(red + 32);                    // [16]
  volatile int* abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 192);
  int* wend = reinterpret_cast<int*>(smem + kOffMisc + 200);        // [12] each warp's last unit (split mode)
  if (ctid == 0) *abort = 0;
  uint8_t* mybuf = smem + kOffRing + (kBuffers * cw) * kStageBytes;
  const unsigned G = gridDim.x;

  // the warp's stream of weight stages, one stage ahead of the compute (the
  // step descriptors are written once by the host, never by a kernel)
  Cursor ic;
  ic.op = 0;
  cursor_load(P, ic, cw, lane);
  bool ic_ok = cursor_settle(P, ic, cw, lane);
  // Launched as a programmatic dependent of the previous kernel on the stream
  // (standalone and per-matmul launches), this grid may start while that
  // kernel drains.  It lets the next launch be scheduled at once, warms L2
  // with its first weight stages (L2 is coherent, so this is right even if the
  // previous kernel writes the weights), and touches nothing else in global
  // memory until the previous grid has completed.  The griddepcontrol
  // instructions are no-ops for an ordinary or cooperative launch.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (!P.sync) {
    Cursor pc = ic;
    for (int k = 0; k < kWarmStages && pc.op < P.n_ops; ++k) {
      prefetch_stage_l2(pc, lane);
      cursor_advance(P, pc, cw, lane);
    }
  }
  asm volatile("griddepcontrol.wait;" ::: "memory");
  // two stages in flight before the first compute; every later iteration
  // commits exactly one (possibly empty) group, so "wait_group 2" always
  // means "this iteration's stage has landed"
  for (int b = 0; b < kBuffers - 1; ++b) {
    if (ic_ok) {
      issue_stage(ic, lane, mybuf + b * kStageBytes);
      cursor_advance(P, ic, cw, lane);
      ic_ok = ic.op < P.n_ops;
    } else {
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
  }
  int j = 0;  // stages computed by this warp
  // set when the warp issued its next stage early, at the end of its previous step
  // (three copies in flight through the grid-wide wait); the next unit then skips
  // its own issue, so "wait_group 2" still means "this unit's stage has landed"
  bool ahead = false;
  bool ahead_due = false;  // warp 0: the early issue waits for the step's release
  // Step descriptors are read from shared memory: warp 0 copies step 0's now and, during
  // step i, loads step i+1's (one word per lane), storing it before the step's last CTA
  // barrier.  Read from global memory after a grid-wide handover, each dependent field
  // load would be an L2 round trip.
  uint32_t* sdesc = reinterpret_cast<uint32_t*>(smem + kOffDesc);
  if (P.ops && cw == 0) sdesc[lane] = __ldcg(reinterpret_cast<const uint32_t*>(P.ops) + lane);
  __syncthreads();

  for (int i = 0; i < P.n_ops; ++i) {
    const EngOp& op = P.ops ? *reinterpret_cast<const EngOp*>(smem + kOffDesc + (i & 1) * 128) : P.inl[i];
    uint32_t next_desc = 0;
    if (P.ops && cw == 0 && i + 1 < P.n_ops)
      next_desc = __ldcg(reinterpret_cast<const uint32_t*>(P.ops + i + 1) + lane);
    if (P.ops && lane < 2 && i + 1 + lane < P.n_ops)  // the copy cursor reads them next
      asm volatile("prefetch.global.L1 [%0];" ::"l"(P.ops + i + 1 + lane));
    // does thread 0 signal this step's end on the grid-wide counter?
    const bool arrives = P.sync && !(op.flags & F_NOARRIVE);
    // -- wait for the earlier steps of this launch to finish on every CTA
    if (ctid == 0 && P.sync && (op.flags & F_WAIT) && (i > 0 || P.first_wait) && !*abort) {
      const unsigned target = (unsigned)op.wait_target * G + (unsigned)op.wait_extra;
      if (ld_acquire_gpu(&P.sync[0]) < target) {
        const uint64_t t0 = globaltimer_ns();
        for (uint32_t it = 1; ld_acquire_gpu(&P.sync[0]) < target; ++it) {
          if ((it & 255) == 0 && globaltimer_ns() - t0 > P.timeout_ns) {
            set_error(P, FAK_ERR_TIMEOUT, abort);
            break;
          }
        }
      }
    }
    named_bar_sync(1, kConsumerThreads);
    if (*abort) break;

    if (op.kind == OP_EMBED) {
      int tok = P.tok_in ? *P.tok_in : 0;
      if (tok < 0 || tok >= op.vocab) {
        if (ctid == 0) atomicCAS(P.err ? P.err : &g_fak_status, 0, FAK_ERR_DEVICE);
        tok = 0;
      }
      const int64_t D = op.K, c = blockIdx.x;
      const int64_t a = D * c / G, b = D * (c + 1) / G;
      if (op.flags & F_TAGOUT) {
        const uint32_t tg = tag_out_par(op.tags, 0) ^ ((P.flip >> tag_out_buf(op.tags, 0)) & 1u);
        for (int64_t k = a + ctid; k < b; k += kConsumerThreads) st_tagged(op.y[0] + k, op.x[(int64_t)tok * D + k], tg);
      } else {
        for (int64_t k = a + ctid; k < b; k += kConsumerThreads) op.y[0][k] = op.x[(int64_t)tok * D + k];
      }
    } else if (op.kind == OP_ARGMAX_REDUCE) {
      if (blockIdx.x == 0 && cw == 0) {
        float bv = 0.0f;
        int bi = -1;
        for (unsigned c = lane; c < G; c += 32) better(ld_cg_f(P.cand_val + c), ld_cg_i(P.cand_idx + c), bv, bi);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
          better(ov, oi, bv, bi);
        }
        if (lane == 0 && P.tok_out) *P.tok_out = bi < 0 ? 0 : bi;
        if (lane == 0 && P.pos) *P.pos += 1;  // the next token's position
      }
    } else if (op.kind == OP_GDN) {
      gdn_step(P, op, smem, ctid, abort);
      named_bar_sync(1, kConsumerThreads);
      if (*abort) break;
    } else if (op.kind == OP_ATTN) {
      attn_step(P, op, smem, ctid, abort);
      named_bar_sync(1, kConsumerThreads);
      if (*abort) break;
    } else {
      // the work split depends on the descriptor only: worked out while x is still arriving
      const Geo g = geo_of(op);
      const Plan pl = plan_of(op, g, cw);
      prepare_x<I8X>(op, P, smem, red, cw, lane, abort);
      named_bar_sync(1, kConsumerThreads);
      if (*abort) break;
      const float rn = norm_factor(op, red);
      const EmitInfo E = emit_info(op, rn, P.flip);
      // split mode with a residual: the combine's first pass gives thread t output row slot t, whose
      // residual (written by this CTA in an earlier step) is loaded now, under the step's compute
      float res_pre = 0.0f;
      if (pl.split && (E.flags & F_RESID) && ctid < pl.ngroups * kSlots) {
        const int r0 = pl.r_lo + (ctid / kSlots) * g.U, r = ctid % kSlots;
        if (r < (g.pair ? kSlots / 2 : kSlots) && r < min(g.U, pl.r_hi - r0)) res_pre = resid_load_raw(E, r0 + r);
      }
      float* part = reinterpret_cast<float*>(smem + kOffPart);
      const int nout = g.pair ? kSlots / 2 : kSlots;  // output rows per group slot set
      float wbv = 0.0f;
      int wbi = -1;
      int grp = pl.u0 / g.nslab, s = pl.u0 - grp * g.nslab;
      float acc[kSlots];
#pragma unroll
      for (int r = 0; r < kSlots; ++r) acc[r] = 0.0f;
      for (int u = pl.u0; u < pl.u1; ++u) {
        const int r0 = pl.r_lo + grp * g.U;
        const int nr = min(g.U, pl.r_hi - r0);
        const int nslots = g.pair ? kSlots : nr;
        if (ahead) {
          ahead = false;
        } else if (ic_ok) {
          issue_stage(ic, lane, mybuf + ((j + kBuffers - 1) % kBuffers) * kStageBytes);
          cursor_advance(P, ic, cw, lane);
          ic_ok = ic.op < P.n_ops;
        } else {
          asm volatile("cp.async.commit_group;" ::: "memory");
        }
        asm volatile("cp.async.wait_group 2;" ::: "memory");
        __syncwarp();
        const uint8_t* stage = mybuf + (j % kBuffers) * kStageBytes;
        const int nb = min(g.slab, g.bpr - s * g.slab);
        if (g.q8)
          q8_slab(stage, smem, s * g.slab, nb, nslots, lane, acc);
        else if (I8X)
          q4k_slab8(stage, smem, s * g.slab, nb, lane, acc);
        else
          q4k_slab(stage, smem, s * g.slab, nb, lane, acc);
        __syncwarp();
        ++j;
        if (s == g.nslab - 1 || u == pl.u1 - 1) {
          // end of a segment
          const float v = reduce4(acc, lane);
          const int rs = lane >> 3;  // the row slot this lane's value belongs to
          if (pl.split) {
            if ((lane & 7) == 0) part[u * kSlots + rs] = v;
          } else {
            const float up = __shfl_down_sync(0xffffffffu, v, 16);  // pair: up rows sit 16 lanes higher
            if ((lane & 7) == 0 && rs < nout && rs < nr)
              emit(E, P, r0 + rs, v, up, wbv, wbi, resid_load(E, r0 + rs));
          }
#pragma unroll
          for (int r = 0; r < kSlots; ++r) acc[r] = 0.0f;
        }
        if (++s == g.nslab) {
          s = 0;
          ++grp;
        }
      }
      // the warp is done with this step's stages: the buffer of its last one is free, so
      // the next step's third stage starts loading at the end of this step, once the
      // CTA's outputs are written (issuing it, with the copy cursor entering the next
      // step, would otherwise delay them) and after thread 0's arrival where there is
      // one (a release fence waits for copies in flight)
      ahead_due = !ahead && ic_ok && pl.u1 > pl.u0;
      if (pl.split) {
        // sum each row's segments in slab order (the ends of warp runs inside its group, then the
        // group end), one thread per (group, output row slot), and write the row; each warp
        // publishes where its run ends, so the combining threads need no divisions
        if (lane == 0) wend[cw] = pl.u1 - 1;
        named_bar_sync(1, kConsumerThreads);
        for (int t = ctid; t < pl.ngroups * kSlots; t += kConsumerThreads) {
          const int gi = t / kSlots, r = t % kSlots;
          const int r0 = pl.r_lo + gi * g.U;
          if (r >= nout || r >= min(g.U, pl.r_hi - r0)) continue;
          const int ru = (r + kSlots / 2) % kSlots;  // the paired up row's slot (SwiGLU steps)
          const float res = t == ctid ? resid_ready(E, res_pre) : resid_load(E, r0 + r);
          const int b0 = gi * g.nslab, e = b0 + g.nslab - 1;
          float v = 0.0f, vu = 0.0f;
          int last = -1;
          int bws[kNumConsumerWarps - 1];
#pragma unroll
          for (int w = 0; w < kNumConsumerWarps - 1; ++w) bws[w] = wend[w];
#pragma unroll
          for (int w = 0; w < kNumConsumerWarps - 1; ++w) {
            const int bw = bws[w];
            if (bw >= b0 && bw < e && bw > last) {
              v += part[bw * kSlots + r];
              vu += part[bw * kSlots + ru];
              last = bw;
            }
          }
          v += part[e * kSlots + r];
          vu += part[e * kSlots + ru];
          emit(E, P, r0 + r, v, vu, wbv, wbi, res);
        }
      }
      if (op.flags & F_ARGMAX) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
          const float ov = __shfl_xor_sync(0xffffffffu, wbv, o);
          const int oi = __shfl_xor_sync(0xffffffffu, wbi, o);
          better(ov, oi, wbv, wbi);
        }
        if (lane == 0) {
          bestv[cw] = wbv;
          besti[cw] = wbi;
        }
        named_bar_sync(1, kConsumerThreads);
        if (ctid == 0) {
          float bv = 0.0f;
          int bi = -1;
          for (int w = 0; w < kNumConsumerWarps; ++w) better(bestv[w], besti[w], bv, bi);
          P.cand_val[blockIdx.x] = bv;
          P.cand_idx[blockIdx.x] = bi;
        }
      }
    }
    // -- this CTA finished step i
    if (P.ops && cw == 0 && i + 1 < P.n_ops) sdesc[((i + 1) & 1) * 32 + lane] = next_desc;
    named_bar_sync(1, kConsumerThreads);
    if (ctid == 0 && arrives) red_release_gpu_add(&P.sync[0], 1u);
    if (ahead_due) {
      __syncwarp();
      issue_stage(ic, lane, mybuf + ((j + kBuffers - 1) % kBuffers) * kStageBytes);
      cursor_advance(P, ic, cw, lane);
      ic_ok = ic.op < P.n_ops;
      ahead = true;
      ahead_due = false;
    }
  }
  // nothing may still be landing in shared memory when the CTA exits
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncthreads();
  if (threadIdx.x == 0 && P.sync) {
    __threadfence();
    const unsigned prev = atomicAdd(&P.sync[1], 1u);
    if (prev == gridDim.x - 1) {
      atomicExch(&P.sync[0], 0u);
      atomicExch(&P.sync[1], 0u);
    }
  }
}

// ------------------------------------------------------------------ host side
struct DeviceInfo {
  int sms = 0;
  bool ok = false;
  bool attr_set = false;
};
std::mutex g_mu;
DeviceInfo g_dev[64];

int device_setup(int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return fak_cuda_status(cudaErrorInvalidDevice);
  std::lock_guard<std::mutex> lk(g_mu);
  DeviceInfo& di = g_dev[dev];
  if (!di.attr_set) {
    int major = 0, minor = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&di.sms, cudaDevAttrMultiProcessorCount, dev);
    if (major != 10 || minor != 3) return FAK_ERR_UNSUPPORTED;
    cudaError_t e = cudaFuncSetAttribute(engine_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return fak_cuda_status(e);
    e = cudaFuncSetAttribute(engine_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return fak_cuda_status(e);
    di.attr_set = true;
    di.ok = true;
  }
  *sms = di.sms;
  return FAK_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

EngOp make_matvec(int kind, const void* W, int64_t N, int64_t K, const float* x, float* y, int flags) {
  EngOp op;
  memset(&op, 0, sizeof(op));
  op.kind = kind;
  op.flags = flags;
  op.K = (int)K;
  op.nseg = 1;
  op.nrows = N;
  op.seg_end[0] = N;
  op.w[0] = static_cast<const uint8_t*>(W);
  op.y[0] = y;
  op.x = x;
  op.eps = 1e-6f;
  return op;
}

int launch_engine(const EngParams& P, int grid, bool cooperative, cudaStream_t s, bool i8x = false) {
  void (*kern)(EngParams) = i8x ? engine_kernel<true> : engine_kernel<false>;
  cudaError_t e;
  if (cooperative) {
    void* args[] = {const_cast<EngParams*>(&P)};
    e = cudaLaunchCooperativeKernel((const void*)kern, dim3(grid), dim3(kThreads), args, kSmemAlloc, s);
  } else {
    // programmatic stream serialization: this grid's launch overlaps the end of
    // the previous kernel, whose completion it still waits for on the device
    cudaLaunchConfig_t cfg;
    memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemAlloc;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, P);
  }
  return fak_cuda_status(e);
}

EngParams base_params() {
  EngParams P;
  memset(&P, 0, sizeof(P));
  P.timeout_ns = 1000000000ull;
  return P;
}

int single_matvec(int kind, const void* W, int64_t N, int64_t K, const float* x, float* y, cudaStream_t s,
                  bool i8x = false) {
  if (!W || !x || !y) return FAK_ERR_INVALID_ARG;
  if (N < 1 || N > 0x7fffffffLL || K < 256 || K % 256 != 0 || K > FAK_ENGINE_MAX_K) return FAK_ERR_SHAPE;
  if (!aligned16(W) || !aligned16(x)) return FAK_ERR_ALIGN;
  int sms = 0;
  int st = device_setup(&sms);
  if (st != FAK_OK) return st;
  EngParams P = base_params();
  P.inl[0] = make_matvec(kind, W, N, K, x, y, 0);
  P.n_ops = 1;
  const int64_t groups = (N + kRowsPerGroup - 1) / kRowsPerGroup;
  const int grid = (int)std::min<int64_t>(groups, sms);
  return launch_engine(P, grid, false, s, i8x);
}

}  // namespace

// ================================================================== C ABI
extern "C" const char* fak_strerror(int status) {
  switch (status) {
    case FAK_OK: return "ok";
    case FAK_ERR_INVALID_ARG: return "invalid argument (null pointer or bad enum)";
    case FAK_ERR_SHAPE: return "dimension out of the supported range";
    case FAK_ERR_ALIGN: return "pointer not 16-byte aligned";
    case FAK_ERR_CUDA: return "CUDA runtime error";
    case FAK_ERR_TIMEOUT: return "bounded device-side wait timed out";
    case FAK_ERR_NOMEM: return "device allocation failed";
    case FAK_ERR_DEVICE: return "device rejected an input (token id out of range)";
    case FAK_ERR_UNSUPPORTED: return "current device is not sm_103";
    default: return "unknown status";
  }
}

cudaError_t fak_scratch_alloc(void** p, size_t bytes, cudaStream_t s) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(s, &cs);
  if (e != cudaSuccess) return e;
  if (cs != cudaStreamCaptureStatusNone) return cudaMallocAsync(p, bytes, s);
  int dev = 0;
  e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  static std::mutex mu;
  static cudaMemPool_t pools[64];
  cudaMemPool_t pool;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!pools[dev]) {
      cudaMemPoolProps props;
      memset(&props, 0, sizeof(props));
      props.allocType = cudaMemAllocationTypePinned;
      props.location.type = cudaMemLocationTypeDevice;
      props.location.id = dev;
      e = cudaMemPoolCreate(&pools[dev], &props);
      if (e != cudaSuccess) {
        pools[dev] = nullptr;
        return e;
      }
      uint64_t keep = ~0ull;  // never hand memory back between calls
      cudaMemPoolSetAttribute(pools[dev], cudaMemPoolAttrReleaseThreshold, &keep);
    }
    pool = pools[dev];
  }
  return cudaMallocFromPoolAsync(p, bytes, pool, s);
}

extern "C" const char* fak_version(void) { return "fak-q4k-gb300 0.1 (sm_103a)"; }

extern "C" int fak_q4k_gemv(const void* Wq, int64_t N, int64_t K, const float* x, float* y, fak_stream_t stream) {
  return single_matvec(OP_Q4K, Wq, N, K, x, y, (cudaStream_t)stream);
}

extern "C" int fak_q4k_gemv_i8x(const void* Wq, int64_t N, int64_t K, const float* x, float* y,
                                fak_stream_t stream) {
  return single_matvec(OP_Q4K, Wq, N, K, x, y, (cudaStream_t)stream, true);
}

extern "C" int fak_q8_0_gemv(const void* Wq, int64_t N, int64_t K, const float* x, float* y, fak_stream_t stream) {
  return single_matvec(OP_Q8, Wq, N, K, x, y, (cudaStream_t)stream);
}

extern "C" int fak_device_status(fak_stream_t stream) {
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return fak_cuda_status(e);
  int v = 0, zero = 0;
  e = cudaMemcpyFromSymbol(&v, g_fak_status, sizeof(int));
  if (e != cudaSuccess) return fak_cuda_status(e);
  cudaMemcpyToSymbol(g_fak_status, &zero, sizeof(int));
  const int g = fak_gemm_take_status();
  const int b = fak_bgemv_take_status();
  return v != 0 ? v : (g != 0 ? g : b);
}

// ------------------------------------------------------------------ MLP decode
extern "C" size_t fak_mlp_workspace_bytes(int64_t d_ff) {
  if (d_ff <= 0) return 0;
  return 256 + (size_t)((d_ff * 4 + 255) / 256 * 256);
}

extern "C" int fak_mlp_decode(const void* Wgate, const void* Wup, const void* Wdown, int64_t d_model, int64_t d_ff,
                              const float* x, float eps, float* y, void* workspace, size_t workspace_bytes,
                              fak_stream_t stream) {
  if (!Wgate || !Wup || !Wdown || !x || !y || !workspace) return FAK_ERR_INVALID_ARG;
  if (d_model < 256 || d_model % 256 || d_model > FAK_ENGINE_MAX_K || d_ff < 256 || d_ff % 256 ||
      d_ff > FAK_ENGINE_MAX_K)
    return FAK_ERR_SHAPE;
  if (workspace_bytes < fak_mlp_workspace_bytes(d_ff)) return FAK_ERR_SHAPE;
  if (!aligned16(Wgate) || !aligned16(Wup) || !aligned16(Wdown) || !aligned16(x) ||
      (reinterpret_cast<uintptr_t>(workspace) & 255))
    return FAK_ERR_ALIGN;
  int sms = 0;
  int st = device_setup(&sms);
  if (st != FAK_OK) return st;
  unsigned* sync = static_cast<unsigned*>(workspace);
  float* a = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + 256);
  EngParams P = base_params();
  P.inl[0] = make_matvec(OP_Q4K_SWIGLU, Wgate, d_ff, d_model, x, a, F_NORM);
  P.inl[0].w[1] = static_cast<const uint8_t*>(Wup);
  P.inl[0].eps = eps;
  P.inl[1] = make_matvec(OP_Q4K, Wdown, d_model, d_ff, a, y, F_WAIT);
  P.inl[1].wait_target = 1;  // the gate / up step's arrival on every CTA
  P.n_ops = 2;
  P.sync = sync;
  cudaError_t e = cudaMemsetAsync(sync, 0, 2 * sizeof(unsigned), (cudaStream_t)stream);
  if (e != cudaSuccess) return fak_cuda_status(e);
  return launch_engine(P, sms, true, (cudaStream_t)stream);
}

// ------------------------------------------------------------------ MLP decode, no allocation
// Some callers may not allocate device memory at call time: code running
// under a memory planner that owns every byte of the device, code inside a
// region where an allocation's implicit synchronization is not allowed, or a
// host that simply has no allocator handle to pass in.  For them the batch-1
// MLP has a variant whose scratch (two grid-sync counters and the SwiGLU
// output) lives in this file-scope array, sized for d_ff up to
// FAK_MLP_NOALLOC_MAX_FF.  Every GPU that loads the library holds it until the
// process exits.  In host code the symbol is only a stand-in, so its device
// address is looked up once per device (cudaGetSymbolAddress, with that device
// current) and passed to the kernel.
static __device__ __align__(256) uint8_t g_mlp_noalloc_scratch[256 + 4 * FAK_MLP_NOALLOC_MAX_FF];

namespace {
std::mutex g_noalloc_mu;
void* g_noalloc_ptr[64] = {};
}  // namespace

extern "C" int fak_mlp_decode_noalloc(const void* Wgate, const void* Wup, const void* Wdown, int64_t d_model,
                                      int64_t d_ff, const float* x, float eps, float* y, fak_stream_t stream) {
  if (!Wgate || !Wup || !Wdown || !x || !y) return FAK_ERR_INVALID_ARG;
  if (d_model < 256 || d_model % 256 || d_model > FAK_ENGINE_MAX_K || d_ff < 256 || d_ff % 256 ||
      d_ff > FAK_MLP_NOALLOC_MAX_FF)
    return FAK_ERR_SHAPE;
  if (!aligned16(Wgate) || !aligned16(Wup) || !aligned16(Wdown) || !aligned16(x)) return FAK_ERR_ALIGN;
  int sms = 0;
  int st = device_setup(&sms);
  if (st != FAK_OK) return st;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fak_cuda_status(e);
  if (dev < 0 || dev >= 64) return FAK_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      e = cudaGetSymbolAddress(&g_noalloc_ptr[dev], g_mlp_noalloc_scratch);
      if (e != cudaSuccess) {
        g_noalloc_ptr[dev] = nullptr;
        return fak_cuda_status(e);
      }
    }
    scratch = g_noalloc_ptr[dev];
  }
  unsigned* sync = static_cast<unsigned*>(scratch);
  float* a = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + 256);
  EngParams P = base_params();
  P.inl[0] = make_matvec(OP_Q4K_SWIGLU, Wgate, d_ff, d_model, x, a, F_NORM);
  P.inl[0].w[1] = static_cast<const uint8_t*>(Wup);
  P.inl[0].eps = eps;
  P.inl[1] = make_matvec(OP_Q4K, Wdown, d_model, d_ff, a, y, F_WAIT);
  P.inl[1].wait_target = 1;  // the gate / up step's arrival on every CTA
  P.n_ops = 2;
  P.sync = sync;
  // the counters must start at zero; the SwiGLU output is fully overwritten
  e = cudaMemsetAsync(sync, 0, 2 * sizeof(unsigned), (cudaStream_t)stream);
  if (e != cudaSuccess) return fak_cuda_status(e);
  return launch_engine(P, sms, true, (cudaStream_t)stream);
}

// ------------------------------------------------------------------ decode context
struct fak_decode {
  fak_decode_desc desc;
  std::vector<fak_layer_desc> layers;
  int sms = 0;
  int mode = 0;    // FAK_DECODE_ONE_LAUNCH or FAK_DECODE_PER_MATMUL
  bool i8x = false;  // int8 activations for the Q4_K steps
  bool host_wait = false;  // per-matmul launches, each waited on by the host
  int n_ops = 0;
  int n_fa = 0;
  EngOp* d_ops = nullptr;
  std::vector<EngOp> h_ops;
  float* h = nullptr;
  float* t = nullptr;
  float* kv = nullptr;
  float* a = nullptr;
  float* cand_val = nullptr;
  int* cand_idx = nullptr;
  unsigned* sync = nullptr;
  int* err = nullptr;
  unsigned long long timeout_ns = 1000000000ull;
  int debug_op = -1;
  // version tags (see the engine kernel): tokens stepped since the buffers were last zeroed, and
  // the writes per token of each tagged buffer (0 h, 1 t, 2 a, 3 the k / v outputs, 4 mix, 5 t2)
  uint64_t token = 0;
  uint32_t writes_per_token[6] = {0, 0, 0, 0, 0, 0};
  // the mixer bodies (desc.mixer set): their output, the recurrent state and the position
  bool mixer = false;
  fak_mixer_desc mdesc;
  std::vector<fak_mixer_layer> mlayers;
  float* mix = nullptr;          // [n_mix]
  // The FA layers' q+gate output, apart from the GDN layers' in_proj output in t: with the mixer
  // bodies, their readers take parts of it (one head each), and a one-bit version tag is only
  // sound when every version of a buffer overwrites every element its readers read.
  float* t2 = nullptr;           // [fa_qg]
  float* mstate = nullptr;       // per GDN layer: conv state [2][conv_dim][3], then S [nv][128][128]
  size_t mstate_floats = 0;
  float* kvcache = nullptr;      // per FA layer: k cache, v cache [nkv][max_ctx][256]
  size_t kvcache_floats = 0;
  int* pos = nullptr;
  MixDesc* d_mix = nullptr;      // per layer
};

namespace {
void free_ctx(fak_decode* c) {
  if (!c) return;
  cudaFree(c->d_ops);
  cudaFree(c->h);
  cudaFree(c->t);
  cudaFree(c->kv);
  cudaFree(c->a);
  cudaFree(c->cand_val);
  cudaFree(c->cand_idx);
  cudaFree(c->sync);
  cudaFree(c->err);
  cudaFree(c->mix);
  cudaFree(c->t2);
  cudaFree(c->mstate);
  cudaFree(c->kvcache);
  cudaFree(c->pos);
  cudaFree(c->d_mix);
  delete c;
}

int upload_ops(fak_decode* c) {
  std::vector<EngOp> ops = c->h_ops;
  for (auto& o : ops) o.wait_extra = 0;
  if (c->debug_op >= 0 && c->debug_op < (int)ops.size()) {
    EngOp& o = ops[c->debug_op];
    if (o.flags & F_TAGIN)
      o.tags ^= 1 << 3;   // wait for a version parity the input never carries
    else
      o.wait_extra = 1;   // wait for one more arrival than the grid provides
  }
  return fak_cuda_status(cudaMemcpy(c->d_ops, ops.data(), sizeof(EngOp) * ops.size(), cudaMemcpyHostToDevice));
}

// Zeroes the tagged buffers (version 0, tag 0) and restarts the token count.
int reset_tags(fak_decode* c, cudaStream_t s) {
  const int64_t D = c->desc.d_model, F = c->desc.d_ff;
  const int64_t tmax = std::max<int64_t>(c->desc.gdn_in, c->desc.fa_qg);
  const int64_t nkv = std::max<int64_t>(1, 2LL * c->n_fa * c->desc.fa_kv);
  cudaError_t e = cudaMemsetAsync(c->h, 0, D * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->t, 0, tmax * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->a, 0, F * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->kv, 0, nkv * 4, s);
  if (e == cudaSuccess && c->mix) e = cudaMemsetAsync(c->mix, 0, (size_t)c->desc.n_mix * 4, s);
  if (e == cudaSuccess && c->t2) e = cudaMemsetAsync(c->t2, 0, (size_t)c->desc.fa_qg * 4, s);
  c->token = 0;
  return fak_cuda_status(e);
}

// Zeroes the mixer bodies' state (conv states, S, KV caches) and the position.
int reset_mixer_state(fak_decode* c, cudaStream_t s) {
  if (!c->mixer) return FAK_OK;
  cudaError_t e = cudaSuccess;
  if (c->mstate_floats) e = cudaMemsetAsync(c->mstate, 0, c->mstate_floats * 4, s);
  if (e == cudaSuccess && c->kvcache_floats) e = cudaMemsetAsync(c->kvcache, 0, c->kvcache_floats * 4, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(c->pos, 0, sizeof(int), s);
  return fak_cuda_status(e);
}

unsigned tag_flip(const fak_decode* c) {
  unsigned f = 0;
  for (int b = 0; b < 6; ++b) f |= (unsigned)((c->token * c->writes_per_token[b]) & 1u) << b;
  return f | (unsigned)(c->token & 1u) << 8;
}
}  // namespace

extern "C" int fak_decode_create(const fak_decode_desc* d, fak_decode** out) {
  if (!d || !out || !d->layers || !d->lm_head || !d->embedding) return FAK_ERR_INVALID_ARG;
  *out = nullptr;
  if (d->mode < FAK_DECODE_ONE_LAUNCH || d->mode > FAK_DECODE_PER_MATMUL_HOST_WAIT) return FAK_ERR_INVALID_ARG;
  auto okdim = [](int64_t v) { return v >= 256 && v % 256 == 0 && v <= FAK_ENGINE_MAX_K; };
  if (d->n_layers < 0 || !okdim(d->d_model) || !okdim(d->d_ff) || !okdim(d->n_mix) || d->vocab < 1 ||
      d->gdn_in < 1 || d->fa_qg < 1 || d->fa_kv < 1)
    return FAK_ERR_SHAPE;
  int n_fa = 0;
  for (int l = 0; l < d->n_layers; ++l) {
    const fak_layer_desc& L = d->layers[l];
    if (L.kind != FAK_LAYER_GDN && L.kind != FAK_LAYER_FA) return FAK_ERR_INVALID_ARG;
    if (!L.w_in || !L.w_out || !L.w_gate || !L.w_up || !L.w_down) return FAK_ERR_INVALID_ARG;
    if (L.kind == FAK_LAYER_FA && (!L.w_k || !L.w_v)) return FAK_ERR_INVALID_ARG;
    if (d->n_mix > (L.kind == FAK_LAYER_GDN ? d->gdn_in : d->fa_qg)) return FAK_ERR_SHAPE;
    const void* ps[] = {L.w_in, L.w_k, L.w_v, L.w_out, L.w_gate, L.w_up, L.w_down};
    for (const void* p : ps)
      if (p && !aligned16(p)) return FAK_ERR_ALIGN;
    n_fa += L.kind == FAK_LAYER_FA;
  }
  if (!aligned16(d->lm_head) || !aligned16(d->embedding)) return FAK_ERR_ALIGN;
  int sms = 0;
  int st = device_setup(&sms);
  if (st != FAK_OK) return st;
  if (d->mixer) {
    const fak_mixer_desc& m = *d->mixer;
    if (!m.layers) return FAK_ERR_INVALID_ARG;
    if (m.gdn_dk != 128 || m.gdn_dv != 128 || m.fa_dh != 256 || m.gdn_nk < 1 || m.gdn_nv < 1 ||
        m.gdn_nv % m.gdn_nk || m.gdn_nv > sms || m.fa_nq < 1 || m.fa_nkv < 1 || m.fa_nq % m.fa_nkv ||
        m.fa_nq > sms || m.fa_rot < 2 || m.fa_rot % 2 || m.fa_rot > 256 || m.max_ctx < 1 || m.max_ctx > 8192 ||
        !(m.eps >= 0.0f) || !(m.rope_theta > 0.0f))
      return FAK_ERR_SHAPE;
    if ((int64_t)m.gdn_nv * 128 != d->n_mix || (int64_t)m.fa_nq * 256 != d->n_mix ||
        d->gdn_in != 2 * m.gdn_nk * 128 + 2 * m.gdn_nv * 128 + 2 * m.gdn_nv || d->fa_qg != 2 * m.fa_nq * 256 ||
        d->fa_kv != m.fa_nkv * 256)
      return FAK_ERR_SHAPE;
    for (int l = 0; l < d->n_layers; ++l) {
      const fak_mixer_layer& M = m.layers[l];
      if (d->layers[l].kind == FAK_LAYER_GDN) {
        if (!M.conv_w || !M.a_log || !M.dt_bias || !M.norm_w) return FAK_ERR_INVALID_ARG;
        if (!aligned16(M.conv_w)) return FAK_ERR_ALIGN;
      } else if (!M.q_norm_w || !M.k_norm_w) {
        return FAK_ERR_INVALID_ARG;
      }
    }
  }
  fak_decode* c = new fak_decode();
  c->desc = *d;
  c->layers.assign(d->layers, d->layers + d->n_layers);
  c->desc.layers = c->layers.data();
  c->sms = sms;
  // the _I8X modes are the two launch shapes with int8 activations; HOST_WAIT is PER_MATMUL with a
  // host wait after every launch
  c->host_wait = d->mode == FAK_DECODE_PER_MATMUL_HOST_WAIT;
  c->mode = c->host_wait ? FAK_DECODE_PER_MATMUL : (d->mode & 1);
  c->i8x = d->mode == FAK_DECODE_ONE_LAUNCH_I8X || d->mode == FAK_DECODE_PER_MATMUL_I8X;
  c->n_fa = n_fa;
  if (c->mode == FAK_DECODE_ONE_LAUNCH) {
    int dev = 0, coop = 0, per_sm = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev);
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, engine_kernel<false>, kThreads, kSmemAlloc);
    if (!coop || per_sm < 1) {
      delete c;
      return FAK_ERR_UNSUPPORTED;
    }
  }
  const int64_t D = d->d_model, F = d->d_ff;
  const int64_t tmax = std::max<int64_t>(d->gdn_in, d->fa_qg);
  bool okm = cudaMalloc(&c->h, D * 4) == cudaSuccess && cudaMalloc(&c->t, tmax * 4) == cudaSuccess &&
             cudaMalloc(&c->kv, std::max<int64_t>(1, 2LL * n_fa * d->fa_kv) * 4) == cudaSuccess &&
             cudaMalloc(&c->a, F * 4) == cudaSuccess && cudaMalloc(&c->cand_val, sms * 4) == cudaSuccess &&
             cudaMalloc(&c->cand_idx, sms * 4) == cudaSuccess && cudaMalloc(&c->sync, 64) == cudaSuccess &&
             cudaMalloc(&c->err, 64) == cudaSuccess;
  if (!okm) {
    (void)cudaGetLastError();
    free_ctx(c);
    return FAK_ERR_NOMEM;
  }
  cudaMemset(c->sync, 0, 64);
  cudaMemset(c->err, 0, 64);
  cudaMemset(c->kv, 0, std::max<int64_t>(1, 2LL * n_fa * d->fa_kv) * 4);
  // the tagged buffers start at version 0 (tag 0): no step can mistake them for its input
  cudaMemset(c->h, 0, D * 4);
  cudaMemset(c->t, 0, tmax * 4);
  cudaMemset(c->a, 0, F * 4);
  // the mixer bodies: output buffer, recurrent state, KV caches, position, step operands
  std::vector<MixDesc> mds;
  if (d->mixer) {
    c->mixer = true;
    c->mdesc = *d->mixer;
    c->mlayers.assign(d->mixer->layers, d->mixer->layers + d->n_layers);
    c->mdesc.layers = c->mlayers.data();
    const fak_mixer_desc& m = c->mdesc;
    const int64_t conv_dim = 2LL * m.gdn_nk * 128 + (int64_t)m.gdn_nv * 128;
    const size_t gdn_floats = (size_t)(2 * conv_dim * 3 + (int64_t)m.gdn_nv * 128 * 128);
    const size_t fa_floats = (size_t)2 * m.fa_nkv * m.max_ctx * 256;
    c->mstate_floats = gdn_floats * (size_t)(d->n_layers - n_fa);
    c->kvcache_floats = fa_floats * (size_t)n_fa;
    bool okx = cudaMalloc(&c->mix, (size_t)d->n_mix * 4) == cudaSuccess &&
               cudaMalloc(&c->t2, (size_t)d->fa_qg * 4) == cudaSuccess &&
               cudaMalloc(&c->pos, sizeof(int)) == cudaSuccess &&
               cudaMalloc(&c->d_mix, sizeof(MixDesc) * std::max(1, d->n_layers)) == cudaSuccess &&
               (!c->mstate_floats || cudaMalloc(&c->mstate, c->mstate_floats * 4) == cudaSuccess) &&
               (!c->kvcache_floats || cudaMalloc(&c->kvcache, c->kvcache_floats * 4) == cudaSuccess);
    if (!okx) {
      (void)cudaGetLastError();
      free_ctx(c);
      return FAK_ERR_NOMEM;
    }
    cudaMemset(c->mix, 0, (size_t)d->n_mix * 4);
    cudaMemset(c->t2, 0, (size_t)d->fa_qg * 4);
    if (reset_mixer_state(c, 0) != FAK_OK || cudaDeviceSynchronize() != cudaSuccess) {
      free_ctx(c);
      return FAK_ERR_CUDA;
    }
    size_t gi = 0, fi = 0;
    int fa_l = 0;
    for (int l = 0; l < d->n_layers; ++l) {
      MixDesc md;
      memset(&md, 0, sizeof(md));
      const fak_mixer_layer& M = m.layers[l];
      md.t = d->layers[l].kind == FAK_LAYER_GDN ? c->t : c->t2;
      md.out = c->mix;
      md.nk = m.gdn_nk;
      md.nv = m.gdn_nv;
      md.nq = m.fa_nq;
      md.nkv = m.fa_nkv;
      md.rot = m.fa_rot;
      md.max_ctx = m.max_ctx;
      md.theta = m.rope_theta;
      for (int i = 0; i < m.fa_rot / 2; ++i)
        md.inv_freq[i] = std::pow((double)m.rope_theta, -2.0 * (double)i / (double)m.fa_rot);
      md.eps = m.eps;
      if (d->layers[l].kind == FAK_LAYER_GDN) {
        md.conv_w = M.conv_w;
        md.a_log = M.a_log;
        md.dt_bias = M.dt_bias;
        md.norm_w = M.norm_w;
        md.conv_state = c->mstate + gi;
        md.S = c->mstate + gi + 2 * conv_dim * 3;
        gi += gdn_floats;
      } else {
        md.kin = c->kv + (2LL * fa_l) * d->fa_kv;
        md.vin = c->kv + (2LL * fa_l + 1) * d->fa_kv;
        md.q_norm_w = M.q_norm_w;
        md.k_norm_w = M.k_norm_w;
        md.kc = c->kvcache + fi;
        md.vc = c->kvcache + fi + fa_floats / 2;
        fi += fa_floats;
        ++fa_l;
      }
      mds.push_back(md);
    }
    if (cudaMemcpy(c->d_mix, mds.data(), sizeof(MixDesc) * mds.size(), cudaMemcpyHostToDevice) != cudaSuccess) {
      free_ctx(c);
      return FAK_ERR_CUDA;
    }
  }

  // the op list: embed, per layer 4 matvec steps, lm_head + argmax, argmax reduce.  Each step
  // hands its output to the next through version tags (no grid-wide wait); only the argmax
  // reduce waits on the arrival counter, for the lm_head step's per-CTA candidates.
  enum { B_H = 0, B_T = 1, B_A = 2, B_KV = 3, B_MIX = 4, B_T2 = 5 };
  uint32_t ver[6] = {0, 0, 0, 0, 0, 0};  // versions written so far in a token
  auto tag_in = [&](int b) { return (int32_t)(b | (int)(ver[b] & 1u) << 3); };
  auto tag_out = [&](int sgi, int b) {
    const uint32_t v = b == B_KV ? 1u : ++ver[b];  // every k / v slice is written once per token
    return (int32_t)((b | (int)(v & 1u) << 3) << (4 + 4 * sgi));
  };
  const int kTagged = F_TAGIN | F_TAGOUT | F_NOARRIVE;
  std::vector<EngOp>& ops = c->h_ops;
  EngOp e;
  memset(&e, 0, sizeof(e));
  e.kind = OP_EMBED;
  e.flags = F_TAGOUT | F_NOARRIVE;
  e.K = (int)D;
  e.vocab = d->vocab;
  e.x = d->embedding;
  e.y[0] = c->h;
  e.nseg = 1;
  e.tags = tag_out(0, B_H);
  ops.push_back(e);
  int fa_i = 0;
  for (int l = 0; l < d->n_layers; ++l) {
    const fak_layer_desc& L = c->layers[l];
    const bool fa_t2 = c->mixer && L.kind == FAK_LAYER_FA;  // q+gate in its own buffer (see t2)
    EngOp in = make_matvec(OP_Q4K, L.w_in, L.kind == FAK_LAYER_GDN ? d->gdn_in : d->fa_qg, D, c->h,
                           fa_t2 ? c->t2 : c->t, F_NORM | kTagged);
    in.eps = d->eps;
    in.tags = tag_in(B_H) | tag_out(0, fa_t2 ? B_T2 : B_T);
    if (L.kind == FAK_LAYER_FA) {
      in.nseg = 3;
      in.seg_end[0] = d->fa_qg;
      in.seg_end[1] = d->fa_qg + d->fa_kv;
      in.seg_end[2] = d->fa_qg + 2LL * d->fa_kv;
      in.nrows = in.seg_end[2];
      in.w[1] = static_cast<const uint8_t*>(L.w_k);
      in.w[2] = static_cast<const uint8_t*>(L.w_v);
      in.y[1] = c->kv + (2LL * fa_i) * d->fa_kv;
      in.y[2] = c->kv + (2LL * fa_i + 1) * d->fa_kv;
      in.tags |= tag_out(1, B_KV) | tag_out(2, B_KV);
      ++fa_i;
    }
    ops.push_back(in);
    if (c->mixer) {
      // the mixer body between the projections: reads t (and this layer's k, v), writes mix
      EngOp mx;
      memset(&mx, 0, sizeof(mx));
      mx.kind = L.kind == FAK_LAYER_GDN ? OP_GDN : OP_ATTN;
      mx.flags = kTagged;
      mx.nseg = 1;
      mx.x = reinterpret_cast<const float*>(c->d_mix + l);
      mx.tags = tag_in(fa_t2 ? B_T2 : B_T) | tag_out(0, B_MIX);
      ops.push_back(mx);
    }
    EngOp out = make_matvec(OP_Q4K, L.w_out, D, d->n_mix, c->mixer ? c->mix : c->t, c->h, F_RESID | kTagged);
    out.tags = tag_in(c->mixer ? B_MIX : B_T) | tag_out(0, B_H);
    ops.push_back(out);
    EngOp gu = make_matvec(OP_Q4K_SWIGLU, L.w_gate, F, D, c->h, c->a, F_NORM | kTagged);
    gu.w[1] = static_cast<const uint8_t*>(L.w_up);
    gu.eps = d->eps;
    gu.tags = tag_in(B_H) | tag_out(0, B_A);
    ops.push_back(gu);
    EngOp dn = make_matvec(OP_Q4K, L.w_down, D, F, c->a, c->h, F_RESID | kTagged);
    dn.tags = tag_in(B_A) | tag_out(0, B_H);
    ops.push_back(dn);
  }
  EngOp lm = make_matvec(OP_Q8, d->lm_head, d->vocab, D, c->h, nullptr, F_NORM | F_TAGIN | F_ARGMAX);
  lm.eps = d->eps;
  lm.tags = tag_in(B_H);
  ops.push_back(lm);
  EngOp am;
  memset(&am, 0, sizeof(am));
  am.kind = OP_ARGMAX_REDUCE;
  am.flags = F_WAIT;
  am.wait_target = 1;  // the lm_head step is the only one that arrives
  am.nseg = 1;
  ops.push_back(am);
  for (int b = 0; b < 6; ++b) c->writes_per_token[b] = ver[b];
  c->writes_per_token[B_KV] = 1;
  c->n_ops = (int)ops.size();
  if (cudaMalloc(&c->d_ops, sizeof(EngOp) * ops.size()) != cudaSuccess) {
    (void)cudaGetLastError();
    free_ctx(c);
    return FAK_ERR_NOMEM;
  }
  st = upload_ops(c);
  if (st != FAK_OK) {
    free_ctx(c);
    return st;
  }
  *out = c;
  return FAK_OK;
}

extern "C" int fak_decode_step(fak_decode* c, const int32_t* tok_in, int32_t* tok_out, float* logits,
                               fak_stream_t stream) {
  if (!c || !tok_in || !tok_out) return FAK_ERR_INVALID_ARG;
  cudaStream_t s = (cudaStream_t)stream;
  EngParams P = base_params();
  P.ops = c->d_ops;
  P.err = c->err;
  P.cand_val = c->cand_val;
  P.cand_idx = c->cand_idx;
  P.tok_in = tok_in;
  P.tok_out = tok_out;
  P.logits = logits;
  P.timeout_ns = c->timeout_ns;
  P.flip = tag_flip(c);
  P.pos = c->pos;
  if (c->mode == FAK_DECODE_ONE_LAUNCH) {
    P.sync = c->sync;
    P.n_ops = c->n_ops;
    P.first_wait = 0;
    const int st = launch_engine(P, c->sms, true, s, c->i8x);
    if (st == FAK_OK) ++c->token;
    return st;
  }
  for (int i = 0; i < c->n_ops; ++i) {
    P.ops = c->d_ops + i;
    P.n_ops = 1;
    P.sync = nullptr;
    int st = launch_engine(P, c->sms, false, s, c->i8x);
    if (st != FAK_OK) return st;
    if (c->host_wait) {
      st = fak_cuda_status(cudaStreamSynchronize(s));
      if (st != FAK_OK) return st;
    }
  }
  ++c->token;
  return FAK_OK;
}

extern "C" int fak_decode_status(fak_decode* c, fak_stream_t stream) {
  if (!c) return FAK_ERR_INVALID_ARG;
  cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
  if (e != cudaSuccess) return fak_cuda_status(e);
  int v = 0;
  e = cudaMemcpy(&v, c->err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return fak_cuda_status(e);
  cudaMemset(c->err, 0, sizeof(int));
  if (v != 0) {
    // an aborted step leaves the counters and the tagged buffers half-written: start over
    cudaMemset(c->sync, 0, 64);
    int st = reset_tags(c, (cudaStream_t)stream);
    if (st == FAK_OK) st = reset_mixer_state(c, (cudaStream_t)stream);
    if (st != FAK_OK) return st;
    e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return fak_cuda_status(e);
  }
  return v;
}

extern "C" int fak_decode_read_state(fak_decode* c, int which, float* dst, size_t count, fak_stream_t stream) {
  if (!c || !dst || which < 0 || which > 2) return FAK_ERR_INVALID_ARG;
  const size_t n = which == 0 ? (size_t)c->desc.d_model
                              : (which == 1 ? (size_t)2 * c->n_fa * c->desc.fa_kv : (size_t)c->desc.n_mix);
  if (count != n) return FAK_ERR_SHAPE;
  if (n == 0) return FAK_OK;
  const float* src = which == 0 ? c->h : (which == 1 ? c->kv : (c->mixer ? c->mix : c->t));
  return fak_cuda_status(cudaMemcpyAsync(dst, src, n * sizeof(float), cudaMemcpyDefault, (cudaStream_t)stream));
}

extern "C" int fak_decode_reset(fak_decode* c, fak_stream_t stream) {
  if (!c) return FAK_ERR_INVALID_ARG;
  int st = reset_tags(c, (cudaStream_t)stream);
  if (st == FAK_OK) st = reset_mixer_state(c, (cudaStream_t)stream);
  return st;
}

extern "C" int fak_decode_launches_per_step(const fak_decode* c) {
  if (!c) return 0;
  return c->mode == FAK_DECODE_ONE_LAUNCH ? 1 : c->n_ops;
}

extern "C" int fak_decode_set_timeout_ns(fak_decode* c, int64_t ns) {
  if (!c || ns <= 0) return FAK_ERR_INVALID_ARG;
  c->timeout_ns = (unsigned long long)ns;
  return FAK_OK;
}

extern "C" int fak_decode_debug_unreachable_wait(fak_decode* c, int op_index) {
  if (!c || op_index >= c->n_ops) return FAK_ERR_INVALID_ARG;
  c->debug_op = op_index;
  return upload_ops(c);
}

extern "C" void fak_decode_destroy(fak_decode* c) { free_ctx(c); }
