// pda_tc.cu -- stage 1 on the 5th-generation tensor cores (tcgen05, TMEM)
// with TMA page gathers, for sm_103a.
//
// Method: "perf(attention): run up to 8 query rows per request in the triton
// decode kernel" (FreeToken PR #900), "Changes" -- one CTA per (request,
// kv head, head block, KV chunk); the request's R query rows x q heads share
// every K/V byte; each row is masked at its own position and window; the
// chunk's partial (o, lse) goes to stage 2. The orientation is the swap-AB of
// "[Feature Request] Support q_len > 1 for FP8 decode" (hpc-ops issue #4):
// S^T = K Q^T puts 128 KV tokens on the MMA M axis and the R x heads rows
// (16..64) on N, so a decode tile fills the MMA. PV is O^T += V^T P^T with
// head_dim on M. FP8 dequantisation folds into the logit scale and the
// finalize ("Naive Support for Hopper FP8 Prefill Kernel with Per-Head
// Quantization", item 3).
//
// Operands keep the cache's own type: bf16 caches run kind::f16 (bf16) MMAs;
// OCP E4M3 caches run kind::f8f6f4 MMAs on the codes as they sit in shared
// memory (no widening pass). For E4M3 the other operand is written as E4M3
// terms: P = P1 + P2 (P2 the E4M3 residual of P1, about 8 significant bits
// together), and a bf16 query as Q * 2^a = Q1 + Q2/16 (stacked on N): a bf16
// value has 8 significant bits, Q1 holds 4 and the residual the other 4, so
// the split is exact except for residuals below E4M3's normal range (an
// absolute error under 2^-22 of the row's largest element). V is read MN-major straight
// from its [token][d] tile, so no transpose is needed on this hardware. The
// softmax denominator always sums the exact fp32 probabilities.
//
// Warp roles: warp 0 (with two more warps in the one-CTA-per-SM builds)
// issues the TMA page gathers (one 128-byte swizzled box per page and
// 128-byte column of the head) into a ring of 16 KB slots, and warp 0 owns the
// TMEM allocation; warp 1 issues the MMAs from one thread; 8 or 16 warps run
// the online softmax out of TMEM (thread = token row of S^T, a share of the
// columns), write P to shared memory and finish the output (thread = head_dim
// row of O^T). All hand-offs are mbarriers; every wait is bounded and a
// timeout sets PDA_STATUS_WAIT_TIMEOUT and unwinds without hanging.
//
// int8 caches add a TMA ring and converter warps in front of the MMA ring:
// the codes widen exactly to f16, and those builds run kind::f16 MMAs with
// an f16 query and P. The MLA latent (head_dim 576) is read twice from the
// same cache: as K over all its channels and as V over its first 512. The
// mixed-precision MLA records (E4M3 nope with a scale per token and 128
// channels, bf16 rope) keep the codes as MMA operands too: each nope block's
// S^T has TMEM columns of its own, the softmax weighs the blocks by their
// tokens' scales, and each 128-d block of V takes its own P, the weights
// times that block's scales.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "pda_internal.h"

namespace pda {
namespace {


constexpr int kTok = 128;          // KV tokens per tile (MMA M of S^T)
constexpr int kSlot = 16384;       // ring slot: [128 tokens x 128 bytes]
constexpr float kTh = 8.0f;        // lazy rescale threshold, log2 units (P <= 2^8)
constexpr float kLog2e = 1.4426950408889634f;
// running maximum before any key: finite, so a column with no visible key
// so far gives ex2(-inf - kMInit) = 0 rather than NaN
constexpr float kMInit = -1.0e30f;
constexpr float kLn2 = 0.6931471805599453f;

// ------------------------------------------------------------------ helpers
__device__ __forceinline__ uint32_t su32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// Byte offset of byte `b` (< 128) of row `r` inside a 128-byte-swizzled atom
// (rows of 128 B, 16-byte chunks XORed with the row's low 3 bits).
__device__ __forceinline__ uint32_t sw128(uint32_t r, uint32_t b) {
  return r * 128u + ((((b >> 4) ^ r) & 7u) << 4) + (b & 15u);
}

// NB bytes (a multiple of 4, packed little-endian in `w`) at byte b0 of row
// r of a 128-byte-swizzled buffer; b0 is a multiple of NB's alignment (16,
// 8 or 4), so no store crosses a 16-byte chunk.
template <int NB>
__device__ __forceinline__ void store_row(uint8_t* base, int r, int b0, const uint32_t* w) {
  if constexpr (NB % 16 == 0) {
#pragma unroll
    for (int q = 0; q < NB / 16; ++q)
      *reinterpret_cast<uint4*>(base + sw128(r, b0 + 16 * q)) =
          make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
  } else if constexpr (NB % 8 == 0) {
#pragma unroll
    for (int q = 0; q < NB / 8; ++q)
      *reinterpret_cast<uint2*>(base + sw128(r, b0 + 8 * q)) = make_uint2(w[2 * q], w[2 * q + 1]);
  } else {
#pragma unroll
    for (int q = 0; q < NB / 4; ++q) *reinterpret_cast<uint32_t*>(base + sw128(r, b0 + 4 * q)) = w[q];
  }
}

// Shared-memory matrix descriptor, 128-byte swizzle (sm_100 family format).
__device__ __forceinline__ uint64_t sdesc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor: f32 accumulate, A/B format `fmt` (kind::f16: 0 =
// f16, 1 = bf16; kind::f8f6f4: 0 = E4M3), A (B) MN-major if `a_mn` (`b_mn`),
// M = 128, N = n.
__device__ __forceinline__ uint32_t idesc(uint32_t fmt, uint32_t a_mn, uint32_t n,
                                          uint32_t b_mn = 0) {
  return (1u << 4) | (fmt << 7) | (fmt << 10) | (a_mn << 15) | (b_mn << 16) | ((n >> 3) << 17) |
         ((128u >> 4) << 24);
}

template <bool kF8>
__device__ __forceinline__ void mma(uint32_t d, uint64_t a, uint64_t b, uint32_t id, uint32_t acc) {
  if constexpr (kF8)
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0;"
                 " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p; }" ::"r"(d),
                 "l"(a), "l"(b), "r"(id), "r"(acc));
  else
    asm volatile("{ .reg .pred p; setp.ne.b32 p, %4, 0;"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p; }" ::"r"(d), "l"(a),
                 "l"(b), "r"(id), "r"(acc));
}

__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   su32(bar))
               : "memory");
}
__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Four int8 codes (byte k = element k) -> two f16 pairs, exactly: with
// u = x + 128 (the sign bit flipped), the f16 word 0x6400 | u is 1024 + u,
// and subtracting 1152 leaves x (every integer below 2048 is an f16).
__device__ __forceinline__ void i8x4_to_f16x4(uint32_t w, uint32_t& e01, uint32_t& e23) {
  const uint32_t u = w ^ 0x80808080u;
  uint32_t lo, hi;
  asm("prmt.b32 %0, %1, %2, 0x5140;" : "=r"(lo) : "r"(u), "r"(0x64646464u));
  asm("prmt.b32 %0, %1, %2, 0x7362;" : "=r"(hi) : "r"(u), "r"(0x64646464u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(e01) : "r"(lo), "r"(0x64806480u));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(e23) : "r"(hi), "r"(0x64806480u));
}

// Eight bf16 values -> eight f16 values (RNE; exact inside f16's normal range).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  auto two = [](uint32_t w) -> uint32_t {
    const __half2 h = __floats2half2_rn(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
    return *reinterpret_cast<const uint32_t*>(&h);
  };
  return make_uint4(two(v.x), two(v.y), two(v.z), two(v.w));
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float* v) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                 "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const float* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
               "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7]))
               : "memory");
}
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float* v) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st4(uint32_t taddr, const float* v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1,%2,%3,%4};" ::"r"(taddr),
               "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
               "r"(__float_as_uint(v[3]))
               : "memory");
}
template <int K>
__device__ __forceinline__ void tmem_ldk(uint32_t taddr, float* v) {
  if constexpr (K == 8) tmem_ld8(taddr, v);
  else tmem_ld4(taddr, v);
}
template <int K>
__device__ __forceinline__ void tmem_stk(uint32_t taddr, const float* v) {
  if constexpr (K == 8) tmem_st8(taddr, v);
  else tmem_st4(taddr, v);
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void bar_init(uint64_t* b, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(su32(b)), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_arrive(uint64_t* b) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(su32(b)) : "memory");
}
__device__ __forceinline__ void bar_expect_tx(uint64_t* b, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(su32(b)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ bool bar_try(uint64_t* b, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
      : "=r"(done)
      : "r"(su32(b)), "r"(parity)
      : "memory");
  return done != 0;
}
// try_wait that lets the hardware suspend the thread (up to `ns`) until the
// phase completes, so waiting warps stop competing for issue slots.
__device__ __forceinline__ bool bar_try_sleep(uint64_t* b, uint32_t parity, uint32_t ns) {
  uint32_t done;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3; selp.u32 %0, 1, "
      "0, p; }"
      : "=r"(done)
      : "r"(su32(b)), "r"(parity), "r"(ns)
      : "memory");
  return done != 0;
}
__device__ __forceinline__ uint64_t global_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Bound of a drain (a wait for copies already issued) and the default bound
// of every other pipeline wait: 2 s of wall time.
constexpr uint64_t kWaitLimitNs = 2000000000ull;
// Bounded wait: false if another role aborted or the call's wait limit
// (a.wait_limit_ns) ran out, which records PDA_STATUS_WAIT_TIMEOUT and
// aborts the CTA.
__device__ __forceinline__ bool bar_wait(uint64_t* b, uint32_t parity, volatile int* abort_flag,
                                         const DecodeArgs& a) {
  if (bar_try(b, parity)) return true;
  const uint64_t t0 = global_ns();
  for (;;) {
    if (bar_try_sleep(b, parity, 20000u)) return true;
    if (*abort_flag) return false;
    if (global_ns() - t0 > a.wait_limit_ns) {
      *abort_flag = 1;
      atomicOr(a.status, PDA_STATUS_WAIT_TIMEOUT);
      return false;
    }
  }
}
// Bounded wait that ignores the abort flag (draining work already issued).
__device__ __forceinline__ void bar_drain(uint64_t* b, uint32_t parity) {
  const uint64_t t0 = global_ns();
  while (!bar_try_sleep(b, parity, 20000u) && global_ns() - t0 < kWaitLimitNs) {
  }
}

// 4-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                         int c2, int c3, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, "
      "{%2, %3, %4, %5}], [%6];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(su32(bar))
      : "memory");
}

// 2^x by the SFU (ex2.approx.ftz): about 2 ulp, -inf -> 0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Two floats -> two E4M3 codes (RNE, saturating): low byte from `lo`.
__device__ __forceinline__ uint16_t f2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
// P of two columns as two E4M3 terms each, P = P1 + P2 (low bytes: `lo`),
// through f16x2: P <= 2^8 rounds to f16 (11 bits), P1 = E4M3(P) and the
// residual P - P1 (exact in f16) gives P2 = E4M3(P - P1).
__device__ __forceinline__ void p_terms(float lo, float hi, uint16_t& c1, uint16_t& c2) {
  uint32_t h, b, r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(h) : "f"(hi), "f"(lo));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(c1) : "r"(h));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(b) : "h"(c1));
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(r) : "r"(h), "r"(b));
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(c2) : "r"(r));
}
// Two E4M3 codes -> two floats (exact): .x from the low byte.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint16_t c) {
  uint32_t h;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h) : "h"(c));
  return __half22float2(*reinterpret_cast<__half2*>(&h));
}

// Barrier of the NT softmax threads (named barrier 1) that also ORs a predicate.
template <int NT>
__device__ __forceinline__ bool group_or(bool pred) {
  uint32_t in = pred ? 1u : 0u, out;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.red.or.pred q, 1, %2, p; selp.u32 %0, 1, "
      "0, q; }"
      : "=r"(out)
      : "r"(in), "n"(NT)
      : "memory");
  return out != 0;
}
template <int NT>
__device__ __forceinline__ void group_sync() {
  asm volatile("barrier.sync 1, %0;" ::"n"(NT) : "memory");
}
// The same over the 128 threads (4 warps) of one column group, on named
// barrier `id` (2 + the group's index).
__device__ __forceinline__ bool colgroup_or(bool pred, uint32_t id) {
  uint32_t in = pred ? 1u : 0u, out;
  asm volatile(
      "{ .reg .pred p, q; setp.ne.u32 p, %1, 0; barrier.red.or.pred q, %2, 128, p; selp.u32 %0, "
      "1, 0, q; }"
      : "=r"(out)
      : "r"(in), "r"(id)
      : "memory");
  return out != 0;
}
__device__ __forceinline__ void colgroup_sync(uint32_t id) {
  asm volatile("barrier.sync %0, 128;" ::"r"(id) : "memory");
}

// ------------------------------------------------------------ configuration
// NMAX: rows x q heads one CTA holds (16: two CTAs per SM; 64: one).
template <int D, int KVT, int QT, int SMODE, int NMAX>
struct TcCfg {
  static constexpr int kD = D;
  // MLA (D = 576): the keys are 576-channel latents, the values their first
  // 512 channels, read from the same cache
  static constexpr bool kMla = D == 576;
  static constexpr int kDv = kMla ? 512 : D;
  static constexpr int kNmax = NMAX;
  // int8 cache: TMA lands the codes in a raw ring, converter warps widen
  // them exactly to f16 into the MMA ring, and the MMAs are kind::f16 (f16
  // query, f16 P)
  static constexpr bool kI8 = KVT == PDA_INT8;
  // mixed-precision MLA records (E4M3 nope with a scale per token and 128
  // channels, bf16 rope): the nope codes are MMA operands as they are, each
  // 128-channel block's S^T in TMEM columns of its own (kind::f8f6f4, the
  // bf16 query as two E4M3 terms), the rope's S^T beside them (kind::f16,
  // bf16); the softmax weighs the blocks by their tokens' scales, and PV
  // takes one P per block (P times the block's scale), so that the block
  // scales never meet the codes in shared memory
  static constexpr bool kMix = SMODE == PDA_SCALE_MLA_BLOCK;
  static constexpr bool kConv = kI8;      // a TMA ring plus converter warps
  static constexpr bool kF16Ops = kConv;  // ... whose MMAs take f16 operands (f16 Q and P)
  // head_dim 512: a K (or V) tile alone is 64-128 KB, one CTA per SM; int8:
  // one CTA per SM holding both rings
  static constexpr int kCtasPerSm = NMAX <= 16 && D <= 256 && !kI8 ? 2 : 1;
  // softmax warps: 4 per TMEM lane quadrant when a CTA holds up to 64 columns, else 2
  static constexpr int kSmWarps = NMAX <= 16 ? 8 : 16;
  static constexpr int kSmThreads = 32 * kSmWarps;
  // TMA producer warps (warp 0, then warps after the softmax warps): one warp
  // issues a 16-row page box about every 130 cycles, too few for one CTA
  // per SM on small pages, so the 64-column build splits each chunk's
  // boxes over three warps
  static constexpr int kProducers = NMAX > 16 || kCtasPerSm == 1 ? 3 : 1;
  static constexpr int kProdThreads = 32 * kProducers;
  static constexpr int kProdWarp1 = 2 + kSmWarps;
  // int8: warps that widen the codes (after the producer warps)
  static constexpr int kConvWarps = kConv ? (NMAX <= 16 ? 8 : 4) : 0;
  static constexpr int kConvThreads = 32 * kConvWarps;
  static constexpr int kConvWarp0 = kProdWarp1 + kProducers - 1;
  static constexpr int kThreads = 64 + kSmThreads + 32 * (kProducers - 1) + kConvThreads;
  static constexpr int kColGroups = kSmWarps / 4;   // warps sharing a lane quadrant
  static constexpr bool kF8 = KVT == PDA_E4M3;  // E4M3 MMA operands
  static constexpr bool kQSplit = kF8 && QT == PDA_BF16;  // bf16 query as two E4M3 terms
  static constexpr int kQTerms = kQSplit ? 2 : 1;
  static constexpr int kElt = kF8 ? 1 : 2;            // bytes of an MMA operand element
  static constexpr int kAtom = 128 / kElt;           // elements per 128-byte row
  // chunks of a K row (MLA E4M3: the last half-filled, zeros past 576;
  // records: the last one the 64 bf16 rope channels)
  static constexpr int kChunksQK = (D + kAtom - 1) / kAtom;
  // ring slots per K tile: 16-bit V blocks take two adjacent slots, so units
  // keep an even size (MLA bf16: 9 chunks and one empty slot, never loaded)
  static constexpr int kChunks = kF8 ? kChunksQK : (kChunksQK + 1) & ~1;
  static constexpr int kChunksV = kDv / kAtom;       // ring slots per V tile
  static constexpr int kRawChunks = kI8 ? D / 128 : kChunks;  // TMA chunks per tile
  static constexpr int kTileSlots = kChunks + kChunksV;
  static constexpr int kQRows = kNmax * kQTerms;
  static constexpr int kQAtomBytes = kQRows * 128;
  static constexpr int kQBytes = kChunksQK * kQAtomBytes;
  // P^T operand of PV. K-major: rows n (bf16: two 64-token halves; E4M3: the
  // two terms' rows stacked, 16 + 16). MN-major (E4M3, up to 64 columns):
  // one 128-byte row per token holding term 1 then term 2 of every column,
  // so a thread stores its columns with wide stores, in two buffers so that
  // P of tile j + 1 need not wait for PV of tile j.
  static constexpr bool kPMn = kF8 && NMAX > 16;
  static constexpr int kPBufs = kPMn ? 2 : 1;
  static constexpr int kPAtomBytes = kNmax * 128;    // [kNmax rows x 128 B]
  static constexpr int kPBufBytes = kPMn ? kTok * 128 : 2 * kPAtomBytes;
  static constexpr int kOBlocks = kDv / 128;
  // records: one P per 128-d block of V (P times that block's scales)
  static constexpr int kPSets = kMix ? kOBlocks : 1;
  static constexpr int kPBytes = kPBufs * kPBufBytes * kPSets;
  // E4M3: one PV MMA of N = 2 x columns yields both terms' sums side by side
  static constexpr int kOCols = kF8 ? 2 * kNmax : kNmax;  // TMEM columns per O block
  // TMEM columns per S buffer (records: the 4 nope blocks' two-term sums,
  // then the rope's N columns, padded to 32)
  static constexpr int kSCols = kMix ? kOBlocks * kQRows + 32 : kQRows;
  // running maxima kept per column: one, or for records the denominator's
  // and one per 128-d block of O (each block's P carries its own scales)
  static constexpr int kFrames = kMix ? kOBlocks + 1 : 1;
  static constexpr int kTmemNeed = 2 * kSCols + kOBlocks * kOCols;
  static constexpr int kTmemCols =
      kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128 : kTmemNeed <= 256 ? 256 : 512;
  // two CTAs of an SM share its 512 columns
  // barriers (512 B), then m_used [kFrames], alpha [kFrames], colscale,
  // red [4][kFrames], linv [kPSets] (kNmax floats each)
  static constexpr int kSmallBytes = 512 + (6 * kFrames + 1 + kPSets) * kNmax * 4;
  static constexpr int kBudget = kCtasPerSm == 2 ? 228 * 1024 / 2 - 1024 : 227 * 1024;
  // the dynamic window starts 1024-byte aligned (checked at run time)
  static constexpr int kAvail = kBudget - kQBytes - kPBytes - kSmallBytes;
  // (at most 12 slots, but for the E4M3 MLA latent, whose aliased K units
  // want all the room there is)
  static constexpr int kMaxSlots = kMla && kF8 ? 16 : 12;
  static constexpr int kAvailSlots = kAvail / kSlot > kMaxSlots ? kMaxSlots : kAvail / kSlot;
  // int8: a third of the slots (at least 2) hold TMA'd codes, the rest f16
  // tiles (the MMA side needs two tiles of those to keep widening ahead)
  static constexpr int kIRing = kConv ? (kAvailSlots / 3 < 2 ? 2 : kAvailSlots / 3) : 0;
  static constexpr int kRingRaw = kAvailSlots - kIRing;
  // bf16 / f16 V blocks span two adjacent slots: keep the ring even so pairs never wrap
  static constexpr int kRing = kF8 ? kRingRaw : (kRingRaw & ~1);
  // The MMA issuer frees each slot as soon as its MMAs finish, so the ring
  // must hold one whole K (or V) tile (the softmax zeroes the tail rows of
  // the last V tile before its PV); head_dim <= 256 builds keep two tiles
  // in flight, head_dim 512 (a tile of 8 or 4 slots) as many as fit.
  // (int8: no tail zeroing, so one tile plus one widened chunk is enough)
  static constexpr bool kBuildable =
      kRing >= (kI8 ? kChunks + 2 : (D > 256 ? kChunksV : kTileSlots)) && kTmemNeed <= 512 &&
      kTmemCols * kCtasPerSm <= 512 && (!kI8 || (kIRing >= 1 && D <= 256)) &&
      !(kMla && !kMix && (kQSplit || kI8)) &&
      (!kMix || (kMla && KVT == PDA_E4M3 && QT == PDA_BF16 && NMAX == 16));
  static constexpr int kSmem = kQBytes + kPBytes + (kRing + kIRing) * kSlot + kSmallBytes;
  // E4M3 MLA latent: V is the first 512 channels of the K tile already in
  // the ring, so no V unit is loaded; each K unit stays until its PV (the
  // rope chunk goes after its S^T), and S^T runs one tile ahead instead of
  // two, which needs two K units in the ring and pays only with a few slots
  // more to load ahead (with exactly two, R = 2's 32-column build measured
  // 10 % slower; with 13 slots R = 1 is 6 % faster)
  static constexpr bool kVAlias = kMla && kF8 && kRing >= 2 * kChunks + 3;
  // barrier words in the small area's first 512 bytes
  static_assert(2 * (kRing + kIRing) + 10 + 2 <= 64, "barrier area");
};

// The MMA issuer consumes a tile's K and V units (kChunks and kChunksV ring
// slots) in the order K0, K1, then K_{j+2} followed by V_j for j = 0, 1, ...
// -- S^T of tile j + 2 is issued as soon as the softmax has read S^T of tile
// j, before PV of tile j, so the softmax never waits on a PV. The producer
// loads in the same order, so the ring is a plain FIFO.
// First ring chunk of K_j / V_j in that order, for K units of CK chunks and
// V units of CV (they differ for MLA): K_j follows K_0..K_{j-1} and
// V_0..V_{j-3}; V_j follows K_0..K_{min(j+2, n-1)} and V_0..V_{j-1}.
template <int CK, int CV>
__device__ __forceinline__ uint32_t chunk_pos_k(int j) {
  return static_cast<uint32_t>(j < 2 ? j * CK : j * CK + (j - 2) * CV);
}
template <int CK, int CV>
__device__ __forceinline__ uint32_t chunk_pos_v(int j, int n) {
  return static_cast<uint32_t>(min(j + 3, n) * CK + j * CV);
}

// The same for a configuration whose V units alias their K units (the ring
// then holds K_0, K_1, K_2, ... only).
template <class C>
__device__ __forceinline__ uint32_t unit_pos_k(int j) {
  if constexpr (C::kVAlias) return static_cast<uint32_t>(j * C::kChunks);
  else return chunk_pos_k<C::kChunks, C::kChunksV>(j);
}
template <class C>
__device__ __forceinline__ uint32_t unit_pos_v(int j, int n) {
  if constexpr (C::kVAlias) return static_cast<uint32_t>(j * C::kChunks);
  else return chunk_pos_v<C::kChunks, C::kChunksV>(j, n);
}

// Everything the softmax / epilogue warps need from the CTA prologue.
struct SoftmaxCtx {
  uint8_t* p_s;
  uint8_t* ring;
  uint64_t* full;
  uint64_t* s_full;
  uint64_t* s_free;
  uint64_t* p_full;
  uint64_t* pv_done;
  volatile int* abort_flag;
  float* m_used;
  float* alpha;
  float* colscale;
  float* red;
  float* linv;
  const int32_t* ptab;
  uint32_t tmem;
  int q0, R, L, W, P, hpc, M, head0, hkv, split, t_begin, t_end, ntiles;
  bool single;
};

// Online softmax over S^T in TMEM, P^T to shared memory, then the epilogue.
// Two warps share each TMEM lane quadrant: a thread owns one KV token of the
// tile (one head_dim row of O^T in the epilogue) and one half of the N
// columns. NCH = N / 16 is a compile-time constant so that every
// per-column loop has an exact trip count.
template <class C, int SMODE, int NCH>
__device__ __forceinline__ void softmax_role(const DecodeArgs& a, const SoftmaxCtx& x, int warp,
                                             int lane, int tid) {
  constexpr int N = NCH * 16;
  constexpr int NT = C::kSmThreads;
  constexpr int NH = N / C::kColGroups;  // columns of this thread
  constexpr int KC = NH % 8 == 0 ? 8 : 4; // TMEM load width
  constexpr int NCK = NH / KC;
  constexpr int R_ = C::kRing;
  constexpr bool kF8 = C::kF8;
  const int st = tid - 64;       // 0..NT-1
  const int qd = warp & 3;       // TMEM lane quadrant of this warp
  const int r = qd * 32 + lane;  // token row of S^T / d row of O^T
  const int sw = (warp - 2) & 3; // warp index within the column group
  const int c0 = ((warp - 2) >> 2) * NH;  // first column of this thread
  const uint32_t bar_id = 2u + static_cast<uint32_t>((warp - 2) >> 2);  // column group's barrier
  const int gi = sw * 32 + lane;          // thread index within the column group
  const uint32_t tl = x.tmem + (static_cast<uint32_t>(qd * 32) << 16);
  const uint32_t tl_o = tl + 2 * C::kSCols;
  const int M = x.M, hpc = x.hpc, R = x.R;

  float qk_scale = a.sm_scale * kLog2e;  // logits in log2 units
  if constexpr (C::kQSplit) qk_scale *= x.colscale[0];  // the query's 2^-a
  float v_final = 1.f;
  if constexpr (SMODE == PDA_SCALE_TENSOR) {
    qk_scale *= __ldg(a.k_scale);
    v_final = __ldg(a.v_scale);
  }
  const int p_first = x.L - R;                   // position of row 0
  const int all_hi = min(p_first, x.t_end - 1);  // every real row sees keys <= all_hi
  const int all_lo = x.W > 0 ? x.L - x.W : 0;    // ... and >= all_lo

  float lsum[NH];
#pragma unroll
  for (int i = 0; i < NH; ++i) lsum[i] = 0.f;
  bool alive = true;

  // per-token scales of this thread's key: the page id is loaded three tiles
  // ahead and the scales two tiles ahead (a tile takes about one loaded HBM
  // latency), so the loop never waits on a load. The key's page index and
  // slot advance by (kTok / P, kTok % P) per tile: no division in the loop.
  const int sP = x.P;
  const int dq = kTok / sP, dr = kTok % sP;
  const int64_t s_page = static_cast<int64_t>(sP) * a.hkv;  // scales per page
  int cur_pi = (x.t_begin + r) / sP, cur_ps = (x.t_begin + r) % sP, cur_j = 0;
  // page id of tile cur_j (-1: past the chunk), then the cursor moves on
  auto next_page = [&](int& slot) -> int {
    const int tok = x.t_begin + cur_j * kTok + r;
    const int pg = (cur_j < x.ntiles && tok < x.t_end) ? __ldg(x.ptab + cur_pi) : -1;
    slot = cur_ps;
    ++cur_j;
    cur_pi += dq;
    cur_ps += dr;
    if (cur_ps >= sP) {
      cur_ps -= sP;
      ++cur_pi;
    }
    return pg;
  };
  auto scales_for = [&](int page, int slot, float& ks, float& vs) {
    ks = 0.f;
    vs = 1.f;
    if (page >= 0 && page < a.num_pages) {
      const int64_t sidx = page * s_page + slot * a.hkv + x.hkv;
      ks = __ldg(a.k_scale + sidx);
      vs = __ldg(a.v_scale + sidx);
    }
  };
  float ks_a = 0.f, vs_a = 1.f, ks_b = 0.f, vs_b = 1.f;  // scales of tiles j and j + 1
  int pg_c = -1, sl_c = 0;                               // page and slot of tile j + 2
  if constexpr (SMODE == PDA_SCALE_TOKEN_HEAD) {
    int sl0, sl1;
    const int pg0 = next_page(sl0), pg1 = next_page(sl1);
    pg_c = next_page(sl_c);
    scales_for(pg0, sl0, ks_a, vs_a);
    scales_for(pg1, sl1, ks_b, vs_b);
  }
  for (int j = 0; j < x.ntiles; ++j) {
    const int tok = x.t_begin + j * kTok + r;
    float row_scale = qk_scale, log2_vs = 0.f, inv_vs = 1.f;
    if constexpr (SMODE == PDA_SCALE_TOKEN_HEAD) {
      const float ks = ks_a;
      float vs = vs_a;
      ks_a = ks_b;
      vs_a = vs_b;
      scales_for(pg_c, sl_c, ks_b, vs_b);
      pg_c = next_page(sl_c);
      row_scale *= ks;
      vs = vs > 0.f ? vs : 1.f;
      log2_vs = __log2f(vs);
      inv_vs = __frcp_rn(vs);
    }
    // columns this key is visible to: rows i with lo_i <= tok <= pos_i
    int n_lo = M, n_hi = 0;  // empty
    if (tok < x.t_end) {
      const int i_lo = max(0, tok - p_first);
      const int i_hi = x.W > 0 ? min(R - 1, tok + x.W - 1 - p_first) : R - 1;
      if (i_lo <= i_hi) {
        n_lo = i_lo * hpc;
        n_hi = (i_hi + 1) * hpc;
      }
    }
    const int tile0 = x.t_begin + j * kTok;
    // every real row sees every key of the tile: no mask (padding columns
    // past M then hold finite values that are never written out)
    const bool full = tile0 >= all_lo && tile0 + kTok - 1 <= all_hi;

    if (alive) alive = bar_wait(x.s_full + (j & 1), (j >> 1) & 1, x.abort_flag, a);
    alive = __all_sync(0xffffffffu, alive);
    fence_after();
    float s[NH];
    if (alive) {
      const uint32_t scol = tl + (j & 1) * C::kSCols + c0;
#pragma unroll
      for (int ch = 0; ch < NCK; ++ch) {
        float v[KC];
        tmem_ldk<KC>(scol + ch * KC, v);
        if constexpr (C::kQSplit) {
          float v2[KC];
          tmem_ldk<KC>(scol + N + ch * KC, v2);
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < KC; ++e) s[ch * KC + e] = fmaf(v2[e], 0.0625f, v[e]);
        } else {
          tmem_wait_ld();
#pragma unroll
          for (int e = 0; e < KC; ++e) s[ch * KC + e] = v[e];
        }
      }
    }
    fence_before();
    bar_arrive(x.s_free + (j & 1));

    // scale, mask, and the lazy-rescale vote against this thread's running
    // maxima (vector loads; they change only when a vote fires)
    auto load_mu = [&](float* mu) {
#pragma unroll
      for (int i = 0; i < NH; i += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(x.m_used + c0 + i);
        mu[i] = m4.x;
        mu[i + 1] = m4.y;
        mu[i + 2] = m4.z;
        mu[i + 3] = m4.w;
      }
    };
    float dmax = -INFINITY;
    {
      float mu[NH];
      load_mu(mu);
      if (full) {
#pragma unroll
        for (int i = 0; i < NH; ++i) {
          s[i] = fmaf(s[i], row_scale, log2_vs);
          dmax = fmaxf(dmax, s[i] - mu[i]);
        }
      } else {
#pragma unroll
        for (int i = 0; i < NH; ++i) {
          const int n = c0 + i;
          const float v = fmaf(s[i], row_scale, log2_vs);
          s[i] = (n >= n_lo && n < n_hi) ? v : -INFINITY;
          dmax = fmaxf(dmax, s[i] - mu[i]);
        }
      }
    }
    const bool trig = dmax > kTh;
    // One barrier reduction per tile among the 4 warps that share these
    // columns (their maxima and O columns are theirs alone): the vote also
    // carries failures, and a second reduction (only when the first fired)
    // tells them apart, so the group takes one branch. Groups meet again
    // on p_full and in the epilogue; a group that aborts is followed by the
    // others at their next vote (the abort flag is shared).
    const bool fired = colgroup_or(trig || !alive || *x.abort_flag != 0, bar_id);
    if (fired && colgroup_or(!alive || *x.abort_flag != 0, bar_id)) {
      alive = false;
      break;
    }
    if (fired) {
      // exact column maxima over the tile's 128 keys
#pragma unroll
      for (int i = 0; i < NH; ++i) {
        float v = s[i];
#pragma unroll
        for (int off = 16; off; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
        if (lane == 0) x.red[sw * C::kNmax + c0 + i] = v;
      }
      colgroup_sync(bar_id);
      if (gi < NH) {
        const int c = c0 + gi;
        const float mx = fmaxf(fmaxf(x.red[c], x.red[C::kNmax + c]),
                               fmaxf(x.red[2 * C::kNmax + c], x.red[3 * C::kNmax + c]));
        const float mo = x.m_used[c];
        const float mn = fmaxf(mo, mx);  // finite: kMInit bounds it below
        x.alpha[c] = ex2(mo - mn);
        x.m_used[c] = mn;
      }
      colgroup_sync(bar_id);
#pragma unroll
      for (int i = 0; i < NH; ++i) lsum[i] *= x.alpha[c0 + i];
    }
    // probabilities (<= 2^kTh; masked keys -> 0); the denominator sums them exactly
    {
      float mu[NH];
      load_mu(mu);
#pragma unroll
      for (int i = 0; i < NH; ++i) {
        s[i] = ex2(s[i] - mu[i]);
        lsum[i] += s[i] * inv_vs;
      }
    }
    // this tile's P buffer is free once PV of tile j - kPBufs has finished;
    // O (rescaled when the vote fired) once PV of tile j - 1 has. A commit
    // covers every earlier MMA, and no barrier can run a phase ahead: the
    // next PV on it needs the P this thread has not written yet.
    {
      const int need = fired ? j - 1 : j - C::kPBufs;
      if (need >= 0)
        alive = bar_wait(x.pv_done + (need & 1), (need >> 1) & 1, x.abort_flag, a);
    }
    alive = __all_sync(0xffffffffu, alive);
    fence_after();
    if (alive && fired && j >= 1) {
      // rescale O^T (this thread's d row) by alpha per column (E4M3: both terms)
#pragma unroll
      for (int blk = 0; blk < C::kOBlocks; ++blk) {
#pragma unroll
        for (int half = 0; half < (kF8 ? 2 : 1); ++half) {
#pragma unroll
          for (int ch = 0; ch < NCK; ++ch) {
            const uint32_t col = tl_o + blk * C::kOCols + half * N + c0 + ch * KC;
            float v[KC];
            tmem_ldk<KC>(col, v);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < KC; ++e) v[e] *= x.alpha[c0 + ch * KC + e];
            tmem_stk<KC>(col, v);
          }
        }
      }
      tmem_wait_st();
    }
    // last tile: rows past the chunk's end may hold stale or poisoned V
    // (int8 codes are always finite, so their zero P suffices)
    if (!C::kI8 && alive && c0 == 0 && tile0 + kTok > x.t_end && tok >= x.t_end) {
      const uint32_t gv = unit_pos_v<C>(j, x.ntiles);
      for (int c = 0; c < C::kChunksV && alive; ++c) {
        const uint32_t slot = (gv + c) % R_;
        alive = bar_wait(x.full + slot, ((gv + c) / R_) & 1u, x.abort_flag, a);
        uint4* row = reinterpret_cast<uint4*>(x.ring + slot * kSlot + r * 128);
#pragma unroll
        for (int e = 0; e < 8; ++e) row[e] = make_uint4(0, 0, 0, 0);
      }
    }
    // write P^T (128-byte swizzle)
    uint8_t* pb = x.p_s + (j % C::kPBufs) * C::kPBufBytes;
    if constexpr (kF8) {
      // P = P1 + P2 in E4M3 (P2 the rounding residual of P1)
      uint32_t w1[NH / 4], w2[NH / 4];
#pragma unroll
      for (int i = 0; i < NH; i += 2) {
        uint16_t c1, c2;
        p_terms(s[i], s[i + 1], c1, c2);
        if constexpr (C::kPMn) {
          if ((i & 2) == 0) {
            w1[i >> 2] = c1;
            w2[i >> 2] = c2;
          } else {
            w1[i >> 2] |= static_cast<uint32_t>(c1) << 16;
            w2[i >> 2] |= static_cast<uint32_t>(c2) << 16;
          }
        } else {
          // K-major: term t of column n in row t * N + n, this token's byte
          const int n = c0 + i;
          pb[sw128(n, r)] = static_cast<uint8_t>(c1 & 0xFF);
          pb[sw128(n + 1, r)] = static_cast<uint8_t>(c1 >> 8);
          pb[N * 128 + sw128(n, r)] = static_cast<uint8_t>(c2 & 0xFF);
          pb[N * 128 + sw128(n + 1, r)] = static_cast<uint8_t>(c2 >> 8);
        }
      }
      if constexpr (C::kPMn) {
        // MN-major: this token's row, term 1 at byte c0, term 2 at byte N + c0
        store_row<NH>(pb, r, c0, w1);
        store_row<NH>(pb, r, N + c0, w2);
      }
    } else {
      uint8_t* pbase = pb + (r >> 6) * C::kPAtomBytes;
      const uint32_t byte = static_cast<uint32_t>(r & 63) * 2u;
#pragma unroll
      for (int i = 0; i < NH; ++i) {
        if constexpr (C::kF16Ops)
          *reinterpret_cast<__half*>(pbase + sw128(c0 + i, byte)) = __float2half_rn(s[i]);
        else
          *reinterpret_cast<__nv_bfloat16*>(pbase + sw128(c0 + i, byte)) = __float2bfloat16_rn(s[i]);
      }
    }
    fence_async_smem();
    fence_before();
    bar_arrive(x.p_full + (j & 1));
  }
  // ---------------------------------------------------------- epilogue
  if (alive && x.ntiles > 0)
    alive = bar_wait(x.pv_done + ((x.ntiles - 1) & 1), ((x.ntiles - 1) >> 1) & 1, x.abort_flag,
                     a);
  fence_after();
  if (group_or<NT>(!alive)) return;
  // column sums of the per-token partial denominators
#pragma unroll
  for (int i = 0; i < NH; ++i) {
    float v = lsum[i];
#pragma unroll
    for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) x.red[sw * C::kNmax + c0 + i] = v;
  }
  group_sync<NT>();
  if (st < M) {
    const float lt = x.red[st] + x.red[C::kNmax + st] + x.red[2 * C::kNmax + st] + x.red[3 * C::kNmax + st];
    x.linv[st] = lt > 0.f ? v_final / lt : 0.f;
    const float lse2 = lt > 0.f ? x.m_used[st] + __log2f(lt) : -INFINITY;
    const int64_t row = x.q0 + st / hpc;
    const int head = x.head0 + st % hpc;
    if (x.single) {
      if (a.lse) a.lse[row * a.hq + head] = lse2 * kLn2;
    } else {
      a.part_lse[((int64_t)x.split * a.rows_cap + row) * a.hq + head] = lse2;
    }
  }
  group_sync<NT>();
  // O^T out of TMEM (thread = one d row of each 128-row block, its columns),
  // times 1/l. Where the idle ring holds the whole [M][Dv] fp32 tile, it is
  // staged there first, so that every (row, head) output row leaves as
  // 16-byte stores of consecutive channels with one index computation per 4
  // channels; otherwise each element is stored straight from its thread.
  constexpr bool kStage = C::kNmax * C::kDv * 4 <= C::kRing * kSlot;
  float* ostage = reinterpret_cast<float*>(x.ring);
#pragma unroll
  for (int blk = 0; blk < C::kOBlocks; ++blk) {
    const int d = blk * 128 + r;
#pragma unroll
    for (int ch = 0; ch < NCK; ++ch) {
      float v[KC];
      tmem_ldk<KC>(tl_o + blk * C::kOCols + c0 + ch * KC, v);
      if constexpr (kF8) {
        float v2[KC];
        tmem_ldk<KC>(tl_o + blk * C::kOCols + N + c0 + ch * KC, v2);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < KC; ++e) v[e] += v2[e];
      } else {
        tmem_wait_ld();
      }
#pragma unroll
      for (int e = 0; e < KC; ++e) {
        const int n = c0 + ch * KC + e;
        if (n < M) {
          const float o = v[e] * x.linv[n];
          if constexpr (kStage) {
            ostage[n * C::kDv + d] = o;
          } else {
            const int64_t row = x.q0 + n / hpc;
            const int head = x.head0 + n % hpc;
            if (x.single) {
              static_cast<__nv_bfloat16*>(a.out)[(row * a.hq + head) * C::kDv + d] = __float2bfloat16_rn(o);
            } else {
              a.part_o[(((int64_t)x.split * a.rows_cap + row) * a.hq + head) * C::kDv + d] = o;
            }
          }
        }
      }
    }
  }
  if constexpr (kStage) {
    group_sync<NT>();
    constexpr int kQ = C::kDv / 4;  // 4-channel groups of one output row
    for (int q = st; q < M * kQ; q += NT) {
      const int n = q / kQ, c4 = q % kQ;
      const float4 o = reinterpret_cast<const float4*>(ostage)[q];
      const int64_t row = x.q0 + n / hpc;
      const int head = x.head0 + n % hpc;
      if (x.single) {
        const __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(o.z, o.w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + (row * a.hq + head) * C::kDv +
                                  4 * c4) = pk;
      } else {
        *reinterpret_cast<float4*>(a.part_o + (((int64_t)x.split * a.rows_cap + row) * a.hq + head) *
                                                  C::kDv + 4 * c4) = o;
      }
    }
  }
}

// Online softmax of the mixed-precision MLA records (the 16-column build).
// A token's logit is the rope's S^T plus, over the 4 nope blocks, the
// token's block scale times that block's S^T (both query terms). The
// denominator sums the plain weights 2^(y - m_0); block b's P holds the
// weights times the token's scale of block b, 2^(y + log2 s_b - m_b), so
// that PV of the block's raw codes yields that block of the output. Each of
// the five sums runs against a running maximum of its own (frame 0: the
// denominator's, frame 1 + b: block b's), so every P stays <= 2^kTh however
// the scales range; the epilogue brings each O block into frame 0.
template <class C>
__device__ __forceinline__ void softmax_rec(const DecodeArgs& a, const SoftmaxCtx& x, int warp,
                                            int lane, int tid) {
  constexpr int N = 16;                  // columns (rows x heads, padded)
  constexpr int NT = C::kSmThreads;
  constexpr int NH = N / C::kColGroups;  // columns of this thread
  constexpr int NB = C::kOBlocks;        // nope blocks
  constexpr int NF = C::kFrames;         // NB + 1 running maxima per column
  constexpr int NM = C::kNmax;
  constexpr int R_ = C::kRing;
  static_assert(NH == 8 && NM == N && NF == NB + 1 && C::kPBufs == 1, "one 16-column records build");
  const int st = tid - 64;       // 0..NT-1
  const int qd = warp & 3;       // TMEM lane quadrant of this warp
  const int r = qd * 32 + lane;  // token row of S^T / d row of O^T
  const int sw = (warp - 2) & 3; // warp index within the column group
  const int c0 = ((warp - 2) >> 2) * NH;  // first column of this thread
  const uint32_t bar_id = 2u + static_cast<uint32_t>((warp - 2) >> 2);
  const int gi = sw * 32 + lane;          // thread index within the column group
  const uint32_t tl = x.tmem + (static_cast<uint32_t>(qd * 32) << 16);
  const uint32_t tl_o = tl + 2 * C::kSCols;
  const int M = x.M, hpc = x.hpc, R = x.R;

  const float qk = a.sm_scale * kLog2e;        // logits in log2 units
  const float qk_nope = qk * x.colscale[0];    // ... of the nope terms (the query's 2^-a)
  const int p_first = x.L - R;                   // position of row 0
  const int all_hi = min(p_first, x.t_end - 1);  // every real row sees keys <= all_hi
  const int all_lo = x.W > 0 ? x.L - x.W : 0;    // ... and >= all_lo

  float lsum[NH];
#pragma unroll
  for (int i = 0; i < NH; ++i) lsum[i] = 0.f;
  bool alive = true;

  // block scales of this thread's key: page ids three tiles ahead, scales
  // two (the cursor advances by (kTok / P, kTok % P) per tile)
  const int sP = x.P;
  const int dq = kTok / sP, dr = kTok % sP;
  int cur_pi = (x.t_begin + r) / sP, cur_ps = (x.t_begin + r) % sP, cur_j = 0;
  auto next_page = [&](int& slot) -> int {
    const int tok = x.t_begin + cur_j * kTok + r;
    const int pg = (cur_j < x.ntiles && tok < x.t_end) ? __ldg(x.ptab + cur_pi) : -1;
    slot = cur_ps;
    ++cur_j;
    cur_pi += dq;
    cur_ps += dr;
    if (cur_ps >= sP) {
      cur_ps -= sP;
      ++cur_pi;
    }
    return pg;
  };
  auto scales_for = [&](int page, int slot) -> float4 {
    if (page < 0 || page >= a.num_pages) return make_float4(0.f, 0.f, 0.f, 0.f);
    return __ldg(reinterpret_cast<const float4*>(a.k_scale) +
                 ((int64_t)page * sP + slot) * a.hkv + x.hkv);
  };
  int sl0, sl1, sl_c;
  const int pg0 = next_page(sl0), pg1 = next_page(sl1);
  int pg_c = next_page(sl_c);
  float4 sc_a = scales_for(pg0, sl0), sc_b = scales_for(pg1, sl1);

  // this thread's running maxima (they change only when a vote fires)
  float mu[NF][NH];
  auto load_mu = [&]() {
#pragma unroll
    for (int f = 0; f < NF; ++f)
#pragma unroll
      for (int i = 0; i < NH; i += 4) {
        const float4 m4 = *reinterpret_cast<const float4*>(x.m_used + f * NM + c0 + i);
        mu[f][i] = m4.x;
        mu[f][i + 1] = m4.y;
        mu[f][i + 2] = m4.z;
        mu[f][i + 3] = m4.w;
      }
  };
  load_mu();

  for (int j = 0; j < x.ntiles; ++j) {
    const int tok = x.t_begin + j * kTok + r;
    const float4 sc = sc_a;
    sc_a = sc_b;
    sc_b = scales_for(pg_c, sl_c);
    pg_c = next_page(sl_c);
    const float sb[NB] = {sc.x, sc.y, sc.z, sc.w};
    // columns this key is visible to: rows i with lo_i <= tok <= pos_i
    int n_lo = M, n_hi = 0;  // empty
    if (tok < x.t_end) {
      const int i_lo = max(0, tok - p_first);
      const int i_hi = x.W > 0 ? min(R - 1, tok + x.W - 1 - p_first) : R - 1;
      if (i_lo <= i_hi) {
        n_lo = i_lo * hpc;
        n_hi = (i_hi + 1) * hpc;
      }
    }
    const int tile0 = x.t_begin + j * kTok;
    const bool full = tile0 >= all_lo && tile0 + kTok - 1 <= all_hi;

    if (alive) alive = bar_wait(x.s_full + (j & 1), (j >> 1) & 1, x.abort_flag, a);
    alive = __all_sync(0xffffffffu, alive);
    fence_after();
    float y[NH];
#pragma unroll
    for (int i = 0; i < NH; ++i) y[i] = 0.f;
    if (alive) {
      const uint32_t scol = tl + (j & 1) * C::kSCols + c0;
      float v[NB][2][NH], vr[NH];
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        tmem_ld8(scol + b * C::kQRows, v[b][0]);
        tmem_ld8(scol + b * C::kQRows + N, v[b][1]);
      }
      tmem_ld8(scol + NB * C::kQRows, vr);
      tmem_wait_ld();
#pragma unroll
      for (int b = 0; b < NB; ++b) {
        const float w = qk_nope * sb[b];
#pragma unroll
        for (int i = 0; i < NH; ++i) y[i] = fmaf(fmaf(v[b][1][i], 0.0625f, v[b][0][i]), w, y[i]);
      }
#pragma unroll
      for (int i = 0; i < NH; ++i) y[i] = fmaf(vr[i], qk, y[i]);
    }
    fence_before();
    bar_arrive(x.s_free + (j & 1));
    if (!full) {
#pragma unroll
      for (int i = 0; i < NH; ++i) {
        const int n = c0 + i;
        if (n < n_lo || n >= n_hi) y[i] = -INFINITY;
      }
    }
    // log2 of the block scales (a zero scale: the block adds nothing)
    float ls[NB];
#pragma unroll
    for (int b = 0; b < NB; ++b) ls[b] = sb[b] > 0.f ? __log2f(sb[b]) : -INFINITY;

    // the lazy-rescale vote over all five frames (as in the other builds)
    float dmax = -INFINITY;
#pragma unroll
    for (int i = 0; i < NH; ++i) {
      dmax = fmaxf(dmax, y[i] - mu[0][i]);
#pragma unroll
      for (int b = 0; b < NB; ++b) dmax = fmaxf(dmax, y[i] + ls[b] - mu[1 + b][i]);
    }
    const bool fired = colgroup_or(dmax > kTh || !alive || *x.abort_flag != 0, bar_id);
    if (fired && colgroup_or(!alive || *x.abort_flag != 0, bar_id)) {
      alive = false;
      break;
    }
    if (fired) {
      // exact maxima of every frame over the tile's 128 keys
#pragma unroll
      for (int f = 0; f < NF; ++f)
#pragma unroll
        for (int i = 0; i < NH; ++i) {
          float v = f == 0 ? y[i] : y[i] + ls[f - 1];
#pragma unroll
          for (int off = 16; off; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
          if (lane == 0) x.red[(f * 4 + sw) * NM + c0 + i] = v;
        }
      colgroup_sync(bar_id);
      if (gi < NF * NH) {  // one (frame, column) per thread
        const int f = gi / NH, c = c0 + gi % NH;
        const float* rd = x.red + f * 4 * NM + c;
        const float mx = fmaxf(fmaxf(rd[0], rd[NM]), fmaxf(rd[2 * NM], rd[3 * NM]));
        const float mo = x.m_used[f * NM + c];
        const float mn = fmaxf(mo, mx);  // finite: kMInit bounds it below
        x.alpha[f * NM + c] = ex2(mo - mn);
        x.m_used[f * NM + c] = mn;
      }
      colgroup_sync(bar_id);
#pragma unroll
      for (int i = 0; i < NH; ++i) lsum[i] *= x.alpha[c0 + i];
      load_mu();
    }
#pragma unroll
    for (int i = 0; i < NH; ++i) lsum[i] += ex2(y[i] - mu[0][i]);
    // the P buffers and O are free once PV of tile j - 1 has finished
    if (j >= 1) alive = bar_wait(x.pv_done + ((j - 1) & 1), ((j - 1) >> 1) & 1, x.abort_flag, a);
    alive = __all_sync(0xffffffffu, alive);
    fence_after();
    if (alive && fired && j >= 1) {
      // rescale each O^T block (this thread's d row, both terms) by its frame's alpha
#pragma unroll
      for (int blk = 0; blk < NB; ++blk) {
        float al[NH];
#pragma unroll
        for (int i = 0; i < NH; ++i) al[i] = x.alpha[(1 + blk) * NM + c0 + i];
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t col = tl_o + blk * C::kOCols + half * N + c0;
          float v[NH];
          tmem_ld8(col, v);
          tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < NH; ++i) v[i] *= al[i];
          tmem_st8(col, v);
        }
      }
      tmem_wait_st();
    }
    // last tile: rows past the chunk's end may hold stale or poisoned codes
    if (alive && c0 == 0 && tile0 + kTok > x.t_end && tok >= x.t_end) {
      const uint32_t gv = unit_pos_v<C>(j, x.ntiles);
      for (int c = 0; c < C::kChunksV && alive; ++c) {
        const uint32_t slot = (gv + c) % R_;
        alive = bar_wait(x.full + slot, ((gv + c) / R_) & 1u, x.abort_flag, a);
        uint4* row = reinterpret_cast<uint4*>(x.ring + slot * kSlot + r * 128);
#pragma unroll
        for (int e = 0; e < 8; ++e) row[e] = make_uint4(0, 0, 0, 0);
      }
    }
    // P^T of each block (K-major, two E4M3 terms: term t of column n in row t * N + n)
#pragma unroll
    for (int b = 0; b < NB; ++b) {
      uint8_t* pb = x.p_s + b * C::kPBufBytes;
#pragma unroll
      for (int i = 0; i < NH; i += 2) {
        uint16_t c1, c2;
        p_terms(ex2(y[i] + ls[b] - mu[1 + b][i]), ex2(y[i + 1] + ls[b] - mu[1 + b][i + 1]), c1, c2);
        const int n = c0 + i;
        pb[sw128(n, r)] = static_cast<uint8_t>(c1 & 0xFF);
        pb[sw128(n + 1, r)] = static_cast<uint8_t>(c1 >> 8);
        pb[N * 128 + sw128(n, r)] = static_cast<uint8_t>(c2 & 0xFF);
        pb[N * 128 + sw128(n + 1, r)] = static_cast<uint8_t>(c2 >> 8);
      }
    }
    fence_async_smem();
    fence_before();
    bar_arrive(x.p_full + (j & 1));
  }
  // ---------------------------------------------------------- epilogue
  if (alive && x.ntiles > 0)
    alive = bar_wait(x.pv_done + ((x.ntiles - 1) & 1), ((x.ntiles - 1) >> 1) & 1, x.abort_flag,
                     a);
  fence_after();
  if (group_or<NT>(!alive)) return;
  // column sums of the per-token partial denominators
#pragma unroll
  for (int i = 0; i < NH; ++i) {
    float v = lsum[i];
#pragma unroll
    for (int off = 16; off; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) x.red[sw * NM + c0 + i] = v;
  }
  group_sync<NT>();
  if (st < M) {
    const float lt = x.red[st] + x.red[NM + st] + x.red[2 * NM + st] + x.red[3 * NM + st];
    const float m0 = x.m_used[st];
    // block b's O is in frame 1 + b: 2^(m_b - m_0) brings it to the denominator's
#pragma unroll
    for (int b = 0; b < NB; ++b)
      x.linv[b * NM + st] = lt > 0.f ? ex2(x.m_used[(1 + b) * NM + st] - m0) / lt : 0.f;
    const float lse2 = lt > 0.f ? m0 + __log2f(lt) : -INFINITY;
    const int64_t row = x.q0 + st / hpc;
    const int head = x.head0 + st % hpc;
    if (x.single) {
      if (a.lse) a.lse[row * a.hq + head] = lse2 * kLn2;
    } else {
      a.part_lse[((int64_t)x.split * a.rows_cap + row) * a.hq + head] = lse2;
    }
  }
  group_sync<NT>();
  // O^T out of TMEM (thread = one d row of each block, its columns) through
  // the idle ring, so that every (row, head) output row leaves as 16-byte
  // stores of consecutive channels
  static_assert(NM * C::kDv * 4 <= C::kRing * kSlot, "the ring stages the output");
  float* ostage = reinterpret_cast<float*>(x.ring);
#pragma unroll
  for (int blk = 0; blk < NB; ++blk) {
    const int d = blk * 128 + r;
    float v[NH], v2[NH];
    tmem_ld8(tl_o + blk * C::kOCols + c0, v);
    tmem_ld8(tl_o + blk * C::kOCols + N + c0, v2);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < NH; ++i) {
      const int n = c0 + i;
      if (n < M) ostage[n * C::kDv + d] = (v[i] + v2[i]) * x.linv[blk * NM + n];
    }
  }
  group_sync<NT>();
  constexpr int kQ = C::kDv / 4;  // 4-channel groups of one output row
  for (int q = st; q < M * kQ; q += NT) {
    const int n = q / kQ, c4 = q % kQ;
    const float4 o = reinterpret_cast<const float4*>(ostage)[q];
    const int64_t row = x.q0 + n / hpc;
    const int head = x.head0 + n % hpc;
    if (x.single) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(o.z, o.w);
      uint2 pk;
      pk.x = *reinterpret_cast<const uint32_t*>(&lo);
      pk.y = *reinterpret_cast<const uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(static_cast<__nv_bfloat16*>(a.out) + (row * a.hq + head) * C::kDv +
                                4 * c4) = pk;
    } else {
      *reinterpret_cast<float4*>(a.part_o + (((int64_t)x.split * a.rows_cap + row) * a.hq + head) *
                                                C::kDv + 4 * c4) = o;
    }
  }
}

template <int D, int KVT, int QT, int SMODE, int NMAX>
__global__ void __launch_bounds__(TcCfg<D, KVT, QT, SMODE, NMAX>::kThreads,
                                  TcCfg<D, KVT, QT, SMODE, NMAX>::kCtasPerSm)
    stage1_tc(const __grid_constant__ DecodeArgs a, const __grid_constant__ CUtensorMap tmk,
              const __grid_constant__ CUtensorMap tmv) {
  using C = TcCfg<D, KVT, QT, SMODE, NMAX>;
  constexpr bool kF8 = C::kF8;
  constexpr int R_ = C::kRing;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // swizzled TMA boxes and MMA operands need 1024-byte alignment; the sizes
  // above assume the window provides it, so a CTA without it does nothing
  if ((su32(smem_raw) & 1023u) != 0) {
    if (threadIdx.x == 0) atomicOr(a.status, PDA_STATUS_SMEM_MISALIGNED);
    return;
  }
  uint8_t* smem = smem_raw;
  uint8_t* q_s = smem;
  uint8_t* p_s = q_s + C::kQBytes;
  uint8_t* ring = p_s + C::kPBytes;
  uint8_t* iring = ring + R_ * kSlot;  // int8: the TMA'd codes (kIRing slots)
  uint8_t* small = iring + C::kIRing * kSlot;
  uint64_t* full = reinterpret_cast<uint64_t*>(small);
  uint64_t* empty = full + R_;
  uint64_t* i_full = empty + R_;           // [kIRing] int8 codes landed
  uint64_t* i_empty = i_full + C::kIRing;  // [kIRing] ... widened, slot free
  uint64_t* s_full = i_empty + C::kIRing;
  uint64_t* s_free = s_full + 2;
  uint64_t* p_full = s_free + 2;   // [2]: P of tile j complete, by j & 1
  uint64_t* pv_done = p_full + 2;  // [2]: PV of tile j complete, by j & 1
  uint64_t* q_ready = pv_done + 2;
  uint64_t* drain = q_ready + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* m_used = reinterpret_cast<float*>(small + 512);  // [kFrames][kNmax]
  float* alpha = m_used + C::kFrames * C::kNmax;          // [kFrames][kNmax]
  float* colscale = alpha + C::kFrames * C::kNmax;
  float* red = colscale + C::kNmax;  // [4][kFrames][kNmax]
  float* linv = red + 4 * C::kFrames * C::kNmax;  // [kPSets][kNmax]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- which work item (uniform per CTA; exits before any barrier)
  WorkItem wi;
  if (!work_item(a, blockIdx.x, wi)) return;
  const int hb = wi.hb, split = wi.split, hkv = wi.hkv, b = wi.b;
  // the request's scalars, loaded together (one round trip)
  const int q0 = a.qo_indptr[b];
  const int q1 = a.qo_indptr[b + 1];
  const int L = a.kv_len[b];
  const int W = a.window ? a.window[b] : 0;
  const int kv0 = a.kv_indptr[b];
  const int R = q1 - q0;
  if (R <= 0 || R > a.max_q_len || L < R || L > a.max_kv_len || q0 + R > a.rows_cap) {
    if (tid == 0 && split == 0 && hb == 0 && hkv == 0) {
      uint32_t bits = 0;
      if (R < 0 || R > a.max_q_len) bits |= PDA_STATUS_ROWS_GT_MAX;
      else if (R > 0 && L < R) bits |= PDA_STATUS_KV_LEN_LT_ROWS;
      else if (R > 0 && L > a.max_kv_len) bits |= PDA_STATUS_KV_LEN_GT_MAX;
      else if (R > 0 && q0 + R > a.rows_cap) bits |= PDA_STATUS_ROWS_GT_CAP;
      if (bits) atomicOr(a.status, bits);
    }
    return;
  }
  const int hpc = a.hpc[R];
  if (hb >= a.group / hpc) return;
  const int P = a.page_size;
  const SplitRange sr = split_range(L, R, W, P, chunk_for(a, b));
  if (split >= sr.num_splits) return;
  const int chunk = chunk_for(a, b);
  const int page_begin = sr.lo_page + split * chunk;
  const int page_end = min(page_begin + chunk, sr.num_pages);
  const int t_begin = page_begin * P;
  const int t_end = min(page_end * P, L);
  const int ntiles = (t_end - t_begin + kTok - 1) / kTok;
  const int M = R * hpc;
  const int N = (M + 15) & ~15;   // MMA N of PV (and of each Q term)
  const int Nq = N * C::kQTerms;  // MMA N of S^T
  const int head0 = hkv * a.group + hb * hpc;
  const int32_t* ptab = a.page_table + kv0;

  // ---- setup. The producer warps load the first page ids, then (once
  // warp 0 has initialised the barriers) start the first ring fill without
  // waiting for the rest of the CTA; the MMA warp allocates TMEM and the
  // softmax warps build the query tile meanwhile. Named barrier 7 is the
  // CTA's setup barrier: producers only arrive on it, the others wait.
  const bool producer = warp == 0 || (warp >= C::kProdWarp1 && warp < C::kProdWarp1 + C::kProducers - 1);
  const int pw = warp == 0 ? 0 : warp - C::kProdWarp1 + 1;  // producer index
  const int box_rows = P < kTok ? P : kTok;
  const int nbox = kTok / box_rows;  // <= 16 (P >= 8)
  const int bx = pw + lane * C::kProducers;  // this lane's box within a chunk
  const uint32_t box_bytes = static_cast<uint32_t>(box_rows) * 128u;
  const CUtensorMap* maps[2] = {&tmk, &tmv};
  // this lane's box of tile j: page id (loaded now, checked when used, so
  // the warp never waits on the load) and first slot; false: no box
  auto page_of = [&](int j, int& page, int& slot0) -> bool {
    const int tb = t_begin + j * kTok + bx * box_rows;
    if (j >= ntiles || bx >= nbox || tb >= t_end) return false;
    page = __ldg(ptab + tb / P);
    slot0 = tb % P;
    return true;
  };
  // page ids of tiles j .. j+3 (rotated as K_{j+2} and V_j are emitted);
  // tile j+4's is loaded two tiles before its check
  int pg0 = 0, s00 = 0, pg1 = 0, s01 = 0, pg2 = 0, s02 = 0, pg3 = 0, s03 = 0;
  bool ok0 = false, ok1 = false, ok2 = false, ok3 = false;
  if (producer) {
    if (lane == 0) {
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    ok0 = page_of(0, pg0, s00);
    ok1 = page_of(1, pg1, s01);
    ok2 = page_of(2, pg2, s02);
    ok3 = page_of(3, pg3, s03);
  }
  if (tid == 0) {
    for (int s = 0; s < R_; ++s) {
      // TMA: one arrive.expect_tx per producer warp; int8: every converter
      // thread arrives after widening its share into the slot
      bar_init(full + s, C::kConv ? C::kConvThreads : C::kProducers);
      bar_init(empty + s, 1);
    }
    for (int s = 0; s < C::kIRing; ++s) {
      bar_init(i_full + s, C::kProducers);
      bar_init(i_empty + s, C::kConvThreads);
    }
    bar_init(s_full, 1);
    bar_init(s_full + 1, 1);
    bar_init(s_free, C::kSmThreads);
    bar_init(s_free + 1, C::kSmThreads);
    bar_init(p_full, C::kSmThreads);
    bar_init(p_full + 1, C::kSmThreads);
    bar_init(pv_done, 1);
    bar_init(pv_done + 1, 1);
    bar_init(q_ready, C::kSmThreads);
    bar_init(drain, 1);
    *abort_flag = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (producer) {
    __syncwarp();  // warp 0 reconverges after the barrier setup
    // the other producer warps may use the barriers once warp 0 has made them
    if constexpr (C::kProducers > 1) {
      if (warp == 0)
        asm volatile("bar.arrive 6, %0;" ::"n"(C::kProdThreads) : "memory");
      else
        asm volatile("bar.sync 6, %0;" ::"n"(C::kProdThreads) : "memory");
    } else {
      __syncwarp();
    }
    asm volatile("bar.arrive 7, %0;" ::"n"(C::kThreads) : "memory");
  } else {
    if (warp == 1) {  // the MMA warp owns the TMEM allocation
      asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                       su32(tmem_slot)),
                   "r"(C::kTmemCols)
                   : "memory");
      asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    } else if (warp >= 2 && warp < 2 + C::kSmWarps) {
      const int st = tid - 64;  // 0..kSmThreads-1
      const int sw = warp - 2;  // softmax warp index
      if (st < C::kNmax) {
#pragma unroll
        for (int f = 0; f < C::kFrames; ++f) m_used[f * C::kNmax + st] = kMInit;
        colscale[st] = 1.f;
      }
      // ---- query operand Q^T (K-major, 128-byte swizzle), rows n < N (zero
      // past M); every load is issued before the first store, so the tile
      // costs one round trip to memory
      if constexpr (!C::kQSplit) {
        constexpr int kRowChunks = D * C::kElt / 16;  // 16-byte pieces of one query row
        constexpr int kPadChunks = C::kChunksQK * 8;  // ... of its smem rows (MLA E4M3: zeros past D)
        constexpr int kIters = (C::kNmax * kPadChunks + C::kSmThreads - 1) / C::kSmThreads;
        uint4 qv[kIters];
#pragma unroll
        for (int it = 0; it < kIters; ++it) {
          const int idx = st + it * C::kSmThreads;
          const int n = idx / kPadChunks, cch = idx % kPadChunks;
          qv[it] = make_uint4(0, 0, 0, 0);
          if (n < M && cch < kRowChunks)
            qv[it] = __ldg(reinterpret_cast<const uint4*>(
                static_cast<const uint8_t*>(a.q) +
                (((int64_t)(q0 + n / hpc) * a.hq + head0 + n % hpc) * D) * C::kElt + cch * 16));
        }
#pragma unroll
        for (int it = 0; it < kIters; ++it) {
          const int idx = st + it * C::kSmThreads;
          const int n = idx / kPadChunks, cch = idx % kPadChunks;
          if (n < N) {
            uint4 v = qv[it];
            if constexpr (C::kF16Ops) v = bf16x8_to_f16x8(v);  // f16 operands (converted caches)
            const int byte = cch * 16;
            *reinterpret_cast<uint4*>(q_s + (byte / 128) * C::kQAtomBytes + sw128(n, byte % 128)) = v;
          }
        }
      } else {
        // bf16 query -> Q * 2^a = Q1 + Q2/16 in E4M3 (rows n and N + n), with
        // one exponent a for the CTA, from its largest |Q|. A lane holds kPer
        // elements of each of its warp's rows (n = sw + k * kSmWarps).
        // (records: the 512 nope channels; the 64 rope channels stay bf16)
        constexpr int kDq = C::kMix ? C::kDv : D;
        constexpr int kPer = kDq / 32;  // elements per lane (16, 8 or 4)
        constexpr int kRowsW = C::kNmax / C::kSmWarps;
        uint32_t raw[kRowsW][kPer / 2];  // bf16 pairs, low half first
        uint4 rope[kRowsW];              // records: 8 rope channels of lanes 0-7
#pragma unroll
        for (int k = 0; k < kRowsW; ++k) {
          const int n = sw + k * C::kSmWarps;
#pragma unroll
          for (int e = 0; e < kPer / 2; ++e) raw[k][e] = 0u;
          rope[k] = make_uint4(0, 0, 0, 0);
          if constexpr (C::kMix) {
            if (n < M && lane < 8)
              rope[k] = __ldg(reinterpret_cast<const uint4*>(
                                  static_cast<const uint8_t*>(a.q) +
                                  (((int64_t)(q0 + n / hpc) * a.hq + head0 + n % hpc) * D + kDq) * 2) +
                              lane);
          }
          if (n < M) {
            const uint8_t* src = static_cast<const uint8_t*>(a.q) +
                                 (((int64_t)(q0 + n / hpc) * a.hq + head0 + n % hpc) * D +
                                  lane * kPer) * 2;
            if constexpr (kPer >= 8) {
#pragma unroll
              for (int v4 = 0; v4 < kPer / 8; ++v4) {
                const uint4 w = __ldg(reinterpret_cast<const uint4*>(src) + v4);
                raw[k][4 * v4] = w.x;
                raw[k][4 * v4 + 1] = w.y;
                raw[k][4 * v4 + 2] = w.z;
                raw[k][4 * v4 + 3] = w.w;
              }
            } else {
              const uint2 w = __ldg(reinterpret_cast<const uint2*>(src));
              raw[k][0] = w.x;
              raw[k][1] = w.y;
            }
          }
        }
        float amax = 0.f;
#pragma unroll
        for (int k = 0; k < kRowsW; ++k)
#pragma unroll
          for (int e = 0; e < kPer / 2; ++e)
            amax = fmaxf(amax, fmaxf(fabsf(__uint_as_float(raw[k][e] << 16)),
                                     fabsf(__uint_as_float(raw[k][e] & 0xFFFF0000u))));
#pragma unroll
        for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (lane == 0) red[sw] = amax;
        group_sync<C::kSmThreads>();
        amax = 0.f;
        for (int w = 0; w < C::kSmWarps; ++w) amax = fmaxf(amax, red[w]);
        int ex = 0;
        if (amax > 0.f) ex = static_cast<int>(floorf(__log2f(448.f / amax)));
        ex = ex > 126 ? 126 : ex;
        // keep the scaled maximum inside E4M3's finite range despite log2 rounding
        while (ex > -126 && amax * exp2f(static_cast<float>(ex)) > 448.f) --ex;
        const float up = exp2f(static_cast<float>(ex));
        if (st == 0) colscale[0] = 1.f / up;
#pragma unroll
        for (int k = 0; k < kRowsW; ++k) {
          const int n = sw + k * C::kSmWarps;
          if (n >= N) continue;
          uint8_t codes[2][kPer];
#pragma unroll
          for (int e = 0; e < kPer; e += 2) {
            float v0 = __uint_as_float(raw[k][e / 2] << 16) * up;
            float v1 = __uint_as_float(raw[k][e / 2] & 0xFFFF0000u) * up;
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              const uint16_t c2 = f2_to_e4m3x2(v0, v1);
              const float2 back = e4m3x2_to_f2(c2);
              codes[t][e] = static_cast<uint8_t>(c2 & 0xFF);
              codes[t][e + 1] = static_cast<uint8_t>(c2 >> 8);
              v0 = (v0 - back.x) * 16.f;
              v1 = (v1 - back.y) * 16.f;
            }
          }
          const int byte = lane * kPer;  // d of this lane's first element (1 byte each)
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            uint8_t* dst = q_s + (byte / 128) * C::kQAtomBytes + sw128(t * N + n, byte % 128);
            uint32_t w[kPer / 4];
#pragma unroll
            for (int e = 0; e < kPer / 4; ++e)
              w[e] = codes[t][4 * e] | (codes[t][4 * e + 1] << 8) | (codes[t][4 * e + 2] << 16) |
                     ((uint32_t)codes[t][4 * e + 3] << 24);
            if constexpr (kPer == 16) {
              *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
            } else if constexpr (kPer == 8) {
              *reinterpret_cast<uint2*>(dst) = make_uint2(w[0], w[1]);
            } else {
              *reinterpret_cast<uint32_t*>(dst) = w[0];
            }
          }
          // records: the rope rows n (bf16, unscaled) in the last atom
          if constexpr (C::kMix) {
            if (lane < 8)
              *reinterpret_cast<uint4*>(q_s + C::kOBlocks * C::kQAtomBytes + sw128(n, lane * 16)) =
                  rope[k];
          }
        }
      }
      fence_async_smem();
      group_sync<C::kSmThreads>();  // the query scale visible to the whole group
    }
    fence_before();
    asm volatile("bar.sync 7, %0;" ::"n"(C::kThreads) : "memory");
    fence_after();
  }
  // TMEM address (the MMA and softmax warps only; producers never use it)
  const uint32_t tmem = producer ? 0u : *tmem_slot;
  const uint32_t tmem_o = tmem + 2 * C::kSCols;
  // every warp reconverges here, before the (warp-uniform) role dispatch
  __syncwarp();

  if (warp == 0 || (warp >= C::kProdWarp1 && warp < C::kProdWarp1 + C::kProducers - 1)) {
    // ================================================ TMA producer warps
    // producer pw issues boxes pw, pw + kProducers, ... of every chunk and
    // arrives on the chunk's full barrier with its own byte count
    auto checked = [&](bool want, int page) -> bool {
      if (want && (page < 0 || page >= a.num_pages)) {
        atomicOr(a.status, PDA_STATUS_PAGE_OOB);
        return false;
      }
      return want;
    };
    ok0 = checked(ok0, pg0);
    ok1 = checked(ok1, pg1);
    uint32_t g = 0;   // chunks issued (into the MMA ring; int8: into the int8 ring)
    bool alive = true;
    // int8: chunk g into the int8 ring once the converters have widened
    // the chunk whose slot it takes
    auto emit8 = [&](int kind, bool ok, int pg, int s0) {
      constexpr uint32_t kIR = C::kIRing > 0 ? C::kIRing : 1;  // (other builds never call this)
      const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, ok));
      for (int c = 0; c < C::kRawChunks && alive; ++c, ++g) {
        const uint32_t slot = g % kIR, round = g / kIR;
        int good = 1;
        if (lane == 0) {
          good = bar_wait(i_empty + slot, (round & 1u) ^ 1u, abort_flag, a);
          if (good) bar_expect_tx(i_full + slot, nvalid * box_bytes);
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          alive = false;
          break;
        }
        if (ok) {
          const uint32_t dst = su32(iring + slot * kSlot) + bx * box_bytes;
          const int c1 = a.tma_slot_dim == 1 ? s0 : hkv;
          const int c2 = a.tma_slot_dim == 1 ? hkv : s0;
          tma_load(dst, maps[kind], c * 128, c1, c2, pg, i_full + slot);
        }
      }
    };
    auto emit = [&](int kind, bool ok, int pg, int s0) {
      if constexpr (C::kConv) {
        emit8(kind, ok, pg, s0);
        return;
      }
      const uint32_t nvalid = __popc(__ballot_sync(0xffffffffu, ok));
      const int nch = kind ? C::kChunksV : C::kChunks;
      for (int c = 0; c < nch && alive; ++c, ++g) {
        const uint32_t slot = g % R_, round = g / R_;
        const bool pad = kind == 0 && c >= C::kChunksQK;  // an even-size unit's empty slot
        int good = 1;
        if (lane == 0) {
          good = bar_wait(empty + slot, (round & 1u) ^ 1u, abort_flag, a);
          if (good) bar_expect_tx(full + slot, pad ? 0u : nvalid * box_bytes);
        }
        good = __shfl_sync(0xffffffffu, good, 0);
        if (!good) {
          alive = false;
          break;
        }
        if (ok && !pad) {
          const uint32_t dst = su32(ring + slot * kSlot) + bx * box_bytes;
          const int c1 = a.tma_slot_dim == 1 ? s0 : hkv;
          const int c2 = a.tma_slot_dim == 1 ? hkv : s0;
          if constexpr (C::kMix) {
            // records: nope chunks (K and V) from the code map, the rope
            // chunk from the bf16 map
            const bool rp = kind == 0 && c == C::kOBlocks;
            tma_load(dst, rp ? &tmv : &tmk, rp ? 0 : c * 128, c1, c2, pg, full + slot);
          } else {
            tma_load(dst, maps[kind], c * C::kAtom, c1, c2, pg, full + slot);
          }
        }
      }
    };
    // PDA_INJECT_WITHHOLD_KV (a host-set test hook): issue nothing at all,
    // so that the consumers' first waits run out with nothing in flight
    const bool withhold = (a.inject & PDA_INJECT_WITHHOLD_KV) != 0u;
    if (!withhold) {
      emit(0, ok0, pg0, s00);
      if (ntiles > 1) emit(0, ok1, pg1, s01);
    }
    for (int j = 0; j < ntiles && alive && !withhold; ++j) {
      if (j + 2 < ntiles) {
        ok2 = checked(ok2, pg2);
        emit(0, ok2, pg2, s02);                     // K_{j+2}
      }
      if constexpr (!C::kVAlias) emit(1, ok0, pg0, s00);  // V_j
      pg0 = pg1; s00 = s01; ok0 = ok1;
      pg1 = pg2; s01 = s02; ok1 = ok2;
      pg2 = pg3; s02 = s03; ok2 = ok3;
      ok3 = page_of(j + 4, pg3, s03);
    }
    if constexpr (C::kConv) {
      // drain: every box issued must have landed before the CTA can exit
      if (lane == 0) {
        const uint32_t first = g > (uint32_t)C::kIRing ? g - C::kIRing : 0u;
        for (uint32_t h = first; h < g; ++h) bar_drain(i_full + h % C::kIRing, (h / C::kIRing) & 1u);
      }
    } else {
      // drain: every box issued must have landed before the CTA can exit
      if (lane == 0) {
        const uint32_t first = g > (uint32_t)R_ ? g - R_ : 0u;
        for (uint32_t h = first; h < g; ++h) bar_drain(full + h % R_, (h / R_) & 1u);
      }
    }
  } else if (warp == 1) {
    // ===================================================== MMA issuer warp
    if (lane == 0) {
      bool alive = bar_wait(q_ready, 0, abort_flag, a);
      fence_after();
      const uint32_t fmt = kF8 || C::kF16Ops ? 0u : 1u;  // E4M3, f16 (converted caches) or bf16
      const uint32_t id_s = idesc(fmt, 0, static_cast<uint32_t>(Nq));
      // E4M3: N = both P terms' columns; bf16: N columns
      const uint32_t id_p = idesc(fmt, 1, static_cast<uint32_t>(kF8 ? 2 * N : N), C::kPMn ? 1u : 0u);
      // records: the rope chunk's S^T, bf16 x bf16 (kind::f16), N columns
      const uint32_t id_rope = idesc(1u, 0, static_cast<uint32_t>(N));
      const uint32_t q_addr = su32(q_s), p_addr = su32(p_s), ring_addr = su32(ring);
      // S^T of tile j into TMEM buffer j & 1 (the softmax has freed it)
      auto issue_s = [&](int j) -> bool {
        const int sb = j & 1;
        if (j >= 2 && !bar_wait(s_free + sb, ((j >> 1) - 1) & 1, abort_flag, a)) return false;
        fence_after();
        const uint32_t gk = unit_pos_k<C>(j);
        for (int c = 0; c < C::kChunks; ++c) {
          const uint32_t slot = (gk + c) % R_;
          if (!bar_wait(full + slot, ((gk + c) / R_) & 1u, abort_flag, a)) return false;
          fence_after();
          const uint32_t abase = ring_addr + slot * kSlot;
          const uint32_t bbase = q_addr + c * C::kQAtomBytes;
          if constexpr (C::kMix) {
            // records: nope block c into its own columns, the rope after them
            const bool rp = c == C::kOBlocks;
            const uint32_t d = tmem + sb * C::kSCols + c * C::kQRows;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t ad = sdesc(abase + kk * 32, 16, 1024), bd = sdesc(bbase + kk * 32, 16, 1024);
              if (rp) mma<false>(d, ad, bd, id_rope, kk != 0);
              else mma<true>(d, ad, bd, id_s, kk != 0);
            }
          } else if (c < C::kChunksQK) {  // (not the empty slot of an even-size unit)
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma<kF8>(tmem + sb * C::kSCols, sdesc(abase + kk * 32, 16, 1024),
                       sdesc(bbase + kk * 32, 16, 1024), id_s, (c | kk) != 0);
          }
          // the slot is free once these MMAs finish (an aliased K unit's V
          // chunks once its PV has run)
          if (!C::kVAlias || c >= C::kChunksV) mma_commit(empty + slot);
        }
        mma_commit(s_full + sb);
        return true;
      };
      // O^T += V_j^T P_j^T as soon as the softmax has written P_j
      auto issue_pv = [&](int j) -> bool {
        if (!bar_wait(p_full + (j & 1), (j >> 1) & 1, abort_flag, a)) return false;
        const uint32_t gv = unit_pos_v<C>(j, ntiles);
        constexpr int kBlkSlots = kF8 ? 1 : 2;  // ring slots of one 128-d V block
        const uint32_t pbuf = p_addr + static_cast<uint32_t>(j % C::kPBufs) * C::kPBufBytes;
#pragma unroll
        for (int blk = 0; blk < C::kOBlocks; ++blk) {
          for (int c = blk * kBlkSlots; c < (blk + 1) * kBlkSlots; ++c)
            if (!bar_wait(full + (gv + c) % R_, ((gv + c) / R_) & 1u, abort_flag, a))
              return false;
          fence_after();
          if constexpr (kF8) {
            // V block = one slot (128 d); K = 32 tokens per MMA; both P terms
            // in one MMA (B rows 0..N-1 term 1, N..2N-1 term 2)
            const uint32_t vbase = ring_addr + ((gv + blk) % R_) * kSlot;
            // (records: block blk's own P)
            const uint32_t pb = pbuf + (C::kMix ? blk * C::kPBufBytes : 0);
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t bd = C::kPMn ? sdesc(pb + kk * 4096, 16384, 1024)
                                          : sdesc(pb + kk * 32, 16, 1024);
              mma<true>(tmem_o + blk * C::kOCols, sdesc(vbase + kk * 4096, kSlot, 1024), bd,
                        id_p, !(j == 0 && kk == 0));
            }
          } else {
            // V block = two adjacent slots (2 x 64 d); K = 16 tokens per MMA
            const uint32_t vbase = ring_addr + ((gv + 2 * blk) % R_) * kSlot;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              mma<false>(tmem_o + blk * C::kOCols, sdesc(vbase + kk * 2048, kSlot, 1024),
                         sdesc(pbuf + (kk >> 2) * C::kPAtomBytes + (kk & 3) * 32, 16, 1024),
                         id_p, !(j == 0 && kk == 0));
          }
          for (int c = blk * kBlkSlots; c < (blk + 1) * kBlkSlots; ++c)
            mma_commit(empty + (gv + c) % R_);
        }
        mma_commit(pv_done + (j & 1));
        return true;
      };
      if (alive) alive = issue_s(0);
      if constexpr (C::kVAlias) {
        for (int j = 0; j < ntiles && alive; ++j) {
          // S^T of tile j + 1 (its K unit is in the ring beside K_j)
          if (j + 1 < ntiles) alive = issue_s(j + 1);
          if (alive) alive = issue_pv(j);
        }
      } else {
        if (alive && ntiles > 1) alive = issue_s(1);
        for (int j = 0; j < ntiles && alive; ++j) {
          // S^T of tile j + 2 once the softmax has read tile j's buffer
          if (j + 2 < ntiles) alive = issue_s(j + 2);
          if (alive) alive = issue_pv(j);
        }
      }
      // make sure nothing issued is still running before TMEM is released
      mma_commit(drain);
      bar_drain(drain, 0);
    }
  } else if (warp >= C::kConvWarp0) {
    // =============================== int8 converter warps (kConvWarps > 0)
    // widen TMA chunk gw (128 tokens x 128 codes) into MMA-ring chunks 2gw
    // and 2gw + 1 (64 f16 each), 16 codes per thread and step, in FIFO order
    if constexpr (C::kI8) {
      const int ct = tid - C::kConvWarp0 * 32;  // 0..kConvThreads-1
      const uint32_t total = 2u * static_cast<uint32_t>(ntiles) * C::kRawChunks;
      for (uint32_t gw = 0; gw < total; ++gw) {
        const uint32_t is = gw % C::kIRing;
        const uint32_t c0 = 2 * gw, d0 = c0 % R_, d1 = (c0 + 1) % R_;
        bool ok = bar_wait(i_full + is, (gw / C::kIRing) & 1u, abort_flag, a);
        if (ok) ok = bar_wait(empty + d0, ((c0 / R_) & 1u) ^ 1u, abort_flag, a);
        if (ok) ok = bar_wait(empty + d1, (((c0 + 1) / R_) & 1u) ^ 1u, abort_flag, a);
        if (!__all_sync(0xffffffffu, ok)) break;
        const uint8_t* src = iring + is * kSlot;
        for (int idx = ct; idx < kTok * 8; idx += C::kConvThreads) {
          const int r = idx >> 3, gl = idx & 7;  // token row, 16-code piece
          const uint4 raw = *reinterpret_cast<const uint4*>(src + r * 128 + ((gl ^ (r & 7)) << 4));
          uint4 lo, hi;
          i8x4_to_f16x4(raw.x, lo.x, lo.y);
          i8x4_to_f16x4(raw.y, lo.z, lo.w);
          i8x4_to_f16x4(raw.z, hi.x, hi.y);
          i8x4_to_f16x4(raw.w, hi.z, hi.w);
          uint8_t* dst = ring + (gl < 4 ? d0 : d1) * kSlot + r * 128;
          const int p0 = (gl & 3) * 2;  // first 16-byte piece of the f16 row
          *reinterpret_cast<uint4*>(dst + ((p0 ^ (r & 7)) << 4)) = lo;
          *reinterpret_cast<uint4*>(dst + (((p0 + 1) ^ (r & 7)) << 4)) = hi;
        }
        fence_async_smem();  // the MMAs read these through the async proxy
        bar_arrive(full + d0);
        bar_arrive(full + d1);
        bar_arrive(i_empty + is);
      }
    }
  } else {
    // ========================================= softmax / epilogue warps
    const int st = tid - 64;  // 0..kSmThreads-1
    const int sw = warp - 2;  // softmax warp index
    bar_arrive(q_ready);  // the query tile was built before the CTA-wide sync

    SoftmaxCtx x;
    x.p_s = p_s;
    x.ring = ring;
    x.full = full;
    x.s_full = s_full;
    x.s_free = s_free;
    x.p_full = p_full;
    x.pv_done = pv_done;
    x.abort_flag = abort_flag;
    x.m_used = m_used;
    x.alpha = alpha;
    x.colscale = colscale;
    x.red = red;
    x.linv = linv;
    x.ptab = ptab;
    x.tmem = tmem;
    x.q0 = q0;
    x.R = R;
    x.L = L;
    x.W = W;
    x.P = P;
    x.hpc = hpc;
    x.M = M;
    x.head0 = head0;
    x.hkv = hkv;
    x.split = split;
    x.t_begin = t_begin;
    x.t_end = t_end;
    x.ntiles = ntiles;
    x.single = sr.num_splits == 1;
    if constexpr (C::kMix) {
      softmax_rec<C>(a, x, warp, lane, tid);
    } else if constexpr (NMAX <= 16) {
      softmax_role<C, SMODE, 1>(a, x, warp, lane, tid);
    } else if constexpr (NMAX <= 32) {
      if (N <= 16) softmax_role<C, SMODE, 1>(a, x, warp, lane, tid);
      else softmax_role<C, SMODE, 2>(a, x, warp, lane, tid);
    } else {
      if constexpr (NMAX > 64) {
        switch (N >> 4) {
          case 1: softmax_role<C, SMODE, 1>(a, x, warp, lane, tid); break;
          case 2: softmax_role<C, SMODE, 2>(a, x, warp, lane, tid); break;
          case 3: softmax_role<C, SMODE, 3>(a, x, warp, lane, tid); break;
          case 4: softmax_role<C, SMODE, 4>(a, x, warp, lane, tid); break;
          case 5: softmax_role<C, SMODE, 5>(a, x, warp, lane, tid); break;
          default: softmax_role<C, SMODE, 6>(a, x, warp, lane, tid); break;
        }
      } else {
        switch (N >> 4) {
          case 1: softmax_role<C, SMODE, 1>(a, x, warp, lane, tid); break;
          case 2: softmax_role<C, SMODE, 2>(a, x, warp, lane, tid); break;
          case 3: softmax_role<C, SMODE, 3>(a, x, warp, lane, tid); break;
          default: softmax_role<C, SMODE, 4>(a, x, warp, lane, tid); break;
        }
      }
    }
  }

  // ---- teardown: everyone done with TMEM and shared memory
  __syncwarp();
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  fence_before();
  __syncthreads();
  fence_after();
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(C::kTmemCols)
                 : "memory");
}

// -------------------------------------------------------------- dispatch
using TcFn = void (*)(DecodeArgs, CUtensorMap, CUtensorMap);

template <int D, int KVT, int QT, int SMODE, int NMAX>
TcFn tc_fn() {
  if constexpr (TcCfg<D, KVT, QT, SMODE, NMAX>::kBuildable)
    return stage1_tc<D, KVT, QT, SMODE, NMAX>;
  else
    return nullptr;
}
template <int D, int KVT, int QT, int SMODE, int NMAX>
int tc_smem() {
  using C = TcCfg<D, KVT, QT, SMODE, NMAX>;
  return C::kBuildable ? C::kSmem : -1;
}

// Kernel (or shared-memory size) for the plan's dtypes, head_dim and NMAX.
template <class F>
auto tc_select(const pda_plan_t* p, int nmax, F f) {
  const int kv = p->kv_dtype, qd = p->q_dtype, sm = p->scale_mode;
#define PDA_TC_CASES(DD, NN)                                                              \
  if (kv == PDA_BF16) return f.template get<DD, PDA_BF16, PDA_BF16, PDA_SCALE_NONE, NN>(); \
  if (sm == PDA_SCALE_MLA_BLOCK)                                                          \
    return f.template get<DD, PDA_E4M3, PDA_BF16, PDA_SCALE_MLA_BLOCK, NN>();             \
  if (kv == PDA_INT8) {                                                                   \
    if (sm == PDA_SCALE_TENSOR)                                                           \
      return f.template get<DD, PDA_INT8, PDA_BF16, PDA_SCALE_TENSOR, NN>();              \
    return f.template get<DD, PDA_INT8, PDA_BF16, PDA_SCALE_TOKEN_HEAD, NN>();            \
  }                                                                                       \
  if (qd == PDA_BF16) {                                                                   \
    if (sm == PDA_SCALE_TENSOR)                                                           \
      return f.template get<DD, PDA_E4M3, PDA_BF16, PDA_SCALE_TENSOR, NN>();              \
    return f.template get<DD, PDA_E4M3, PDA_BF16, PDA_SCALE_TOKEN_HEAD, NN>();            \
  }                                                                                       \
  if (sm == PDA_SCALE_TENSOR) return f.template get<DD, PDA_E4M3, PDA_E4M3, PDA_SCALE_TENSOR, NN>(); \
  return f.template get<DD, PDA_E4M3, PDA_E4M3, PDA_SCALE_TOKEN_HEAD, NN>();
  if (p->head_dim == 128) {
    if (nmax <= 16) { PDA_TC_CASES(128, 16) }
    // bf16 caches without scales also have a 96-column build (large GQA
    // groups with several rows: fewer head blocks re-reading the same K/V)
    if (nmax > 64 && kv == PDA_BF16)
      return f.template get<128, PDA_BF16, PDA_BF16, PDA_SCALE_NONE, 96>();
    PDA_TC_CASES(128, 64)
  }
  if (p->head_dim == 512) {
    if (nmax <= 16) { PDA_TC_CASES(512, 16) }
    if (nmax <= 32) { PDA_TC_CASES(512, 32) }
    PDA_TC_CASES(512, 64)
  }
  if (p->head_dim == 576) {  // MLA latent
    if (nmax <= 16) { PDA_TC_CASES(576, 16) }
    if (nmax <= 32) { PDA_TC_CASES(576, 32) }
    PDA_TC_CASES(576, 64)
  }
  if (nmax <= 16) { PDA_TC_CASES(256, 16) }
  PDA_TC_CASES(256, 64)
#undef PDA_TC_CASES
}
struct GetFn {
  template <int D, int KVT, int QT, int SMODE, int NMAX>
  TcFn get() { return tc_fn<D, KVT, QT, SMODE, NMAX>(); }
};
struct GetSmem {
  template <int D, int KVT, int QT, int SMODE, int NMAX>
  int get() { return tc_smem<D, KVT, QT, SMODE, NMAX>(); }
};

// cuTensorMapEncodeTiled, fetched once from the driver through the runtime.
using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                              const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                              const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                              CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeFn encoder() {
  static std::once_flag once;
  static EncodeFn fn = nullptr;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeFn>(p);
    cudaGetLastError();
  });
  return fn;
}

// Tensor map over the paged cache: dims (c, slot, head, page) or
// (c, head, slot, page), ordered by stride; one box = one page's (<= 128)
// tokens x 128 bytes of one head.
// `bf16_view`: the map reads bf16 values inside one-byte-element rows (the
// rope channels of a mixed-precision MLA record).
bool make_map(CUtensorMap* m, const void* base, const pda_plan_t* p, int* slot_dim, int dim0,
              bool bf16_view = false) {
  EncodeFn enc = encoder();
  if (!enc) return false;
  const int eb = p->kv_dtype == PDA_BF16 ? 2 : 1;  // E4M3 / int8 codes: one byte (strides)
  const int ed = bf16_view ? 2 : eb;               // the mapped element
  const bool slot_first = p->kv_stride_token <= p->kv_stride_head;
  *slot_dim = slot_first ? 1 : 2;
  const cuuint32_t rows = static_cast<cuuint32_t>(p->page_size < kTok ? p->page_size : kTok);
  cuuint64_t dims[4], strides[3];
  cuuint32_t box[4], estr[4] = {1, 1, 1, 1};
  dims[0] = static_cast<cuuint64_t>(dim0);  // channels read (V of MLA: the first 512)
  box[0] = static_cast<cuuint32_t>(128 / ed);
  if (slot_first) {
    dims[1] = p->page_size;
    dims[2] = p->num_kv_heads;
    strides[0] = static_cast<cuuint64_t>(p->kv_stride_token) * eb;
    strides[1] = static_cast<cuuint64_t>(p->kv_stride_head) * eb;
    box[1] = rows;
    box[2] = 1;
  } else {
    dims[1] = p->num_kv_heads;
    dims[2] = p->page_size;
    strides[0] = static_cast<cuuint64_t>(p->kv_stride_head) * eb;
    strides[1] = static_cast<cuuint64_t>(p->kv_stride_token) * eb;
    box[1] = 1;
    box[2] = rows;
  }
  dims[3] = static_cast<cuuint64_t>(p->num_pages);
  strides[2] = static_cast<cuuint64_t>(p->kv_stride_page) * eb;
  box[3] = 1;
  const CUtensorMapDataType dt =
      ed == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
  return enc(m, dt, 4, const_cast<void*>(base), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

bool tc_supported(const pda_plan_t* p) {
  return (p->head_dim == 128 || p->head_dim == 256 || p->head_dim == 512 || p->head_dim == 576) &&
         p->page_size >= 8 && p->page_size <= 256 && (p->kv_dtype != PDA_INT8 || p->head_dim <= 256);
}

// Rows x heads a CTA may hold: 64, except head_dim 512 over an E4M3 cache,
// whose two-term S and O accumulators (2 x 2N + 4 x 2N columns) leave TMEM
// room for 32, and head_dim 128 over a bf16 cache, which has a 96-column
// build. The pages' kernel takes 16 for quantised head_dim 512
// ("perf(attention): run up to 8 query rows per request in the triton
// decode kernel"); 32 halves the head blocks that re-read the cache. A
// head block streams its kv head's whole chunk whatever its columns (a CTA's
// pace is set by its K/V bytes, not by its 16-96 columns, measured on the
// 48 / 2-head mixed batch), so fewer, wider head blocks cut the bytes the
// SMs read for a large GQA group with several rows; 96 columns is the widest
// whose softmax state fits the 96 registers a thread has at 640 threads.
int tc_rows_limit(const pda_plan_t* p) {
  // (the MLA latent's E4M3 build likewise: S 2 x N, O 4 x 2N columns; the
  // records' per-block S^T, 2 x (4 x 2N + 32) columns, leaves room for 16)
  if (p->head_dim == 128 && p->kv_dtype == PDA_BF16) return 96;
  if (p->scale_mode == PDA_SCALE_MLA_BLOCK) return 16;
  return p->head_dim >= 512 && p->kv_dtype == PDA_E4M3 ? 32 : kTcRowsPerCta;
}

// Largest N (rows x heads, rounded up to 16) a CTA of this plan can hold.
static int plan_nmax(const pda_plan_t* p) {
  int n = 16;
  for (int r = 1; r <= p->max_q_len; ++r) {
    const int m = ((r * p->heads_per_cta[r] + 15) / 16) * 16;
    n = m > n ? m : n;
  }
  return n;
}

int tc_variant_rows(const pda_plan_t* p) {
  // the smallest build that holds every CTA's columns (16: two CTAs per SM
  // up to head_dim 256; head_dim 512 also has a 32-column build, bf16
  // head_dim 128 a 96-column one)
  const int n = plan_nmax(p);
  if (n <= 16 && tc_select(p, 16, GetSmem()) > 0) return 16;
  if (p->head_dim >= 512 && n <= 32 && tc_select(p, 32, GetSmem()) > 0) return 32;
  if (n > 64 && tc_select(p, 96, GetSmem()) > 0) return 96;
  return 64;
}

int tc_smem_bytes(const pda_plan_t* p) { return tc_select(p, p->rows_per_cta, GetSmem()); }

struct GetCtasPerSm {
  template <int D, int KVT, int QT, int SMODE, int NMAX>
  int get() { return TcCfg<D, KVT, QT, SMODE, NMAX>::kCtasPerSm; }
};
int tc_ctas_per_sm(const pda_plan_t* p) { return tc_select(p, p->rows_per_cta, GetCtasPerSm()); }

struct GetThreads {
  template <int D, int KVT, int QT, int SMODE, int NMAX>
  int get() { return TcCfg<D, KVT, QT, SMODE, NMAX>::kThreads; }
};
static unsigned tc_threads(const pda_plan_t* p) {
  return static_cast<unsigned>(tc_select(p, p->rows_per_cta, GetThreads()));
}

int launch_stage1_tc(const pda_plan_t* plan, const DecodeArgs& args, cudaStream_t s) {
  DecodeArgs a = args;
  CUtensorMap mk, mv;
  int slot_dim = 1;
  const bool rec = plan->scale_mode == PDA_SCALE_MLA_BLOCK;
  // mixed MLA records: the 512 nope codes (K and V), and the 64 bf16 rope
  // channels from byte 512 on
  if (rec ? (!make_map(&mk, args.k, plan, &slot_dim, 512) ||
             !make_map(&mv, static_cast<const uint8_t*>(args.k) + 512, plan, &slot_dim, 64, true))
          : (!make_map(&mk, args.k, plan, &slot_dim, plan->head_dim) ||
             !make_map(&mv, args.v, plan, &slot_dim, plan->head_dim_v)))
    return PDA_ERR_CUDA;
  a.tma_slot_dim = slot_dim;
  TcFn k1 = tc_select(plan, plan->rows_per_cta, GetFn());
  if (!k1) return PDA_ERR_UNSUPPORTED;
  const int smem = plan->stage1_smem_bytes;
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(k1),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return PDA_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan->grid_ctas));
  cfg.blockDim = dim3(tc_threads(plan));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  if (cudaLaunchKernelEx(&cfg, k1, a, mk, mv) != cudaSuccess) {
    cudaGetLastError();
    return PDA_ERR_CUDA;
  }
  return PDA_OK;
}

}  // namespace pda
