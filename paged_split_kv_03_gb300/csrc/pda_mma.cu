// pda_mma.cu -- stage 1 (per-chunk partial attention) on the mma.sync tensor
// path, and stage 2 (per-row log-sum-exp merge), for sm_103a.
//
// Method: "perf(attention): run up to 8 query rows per request in the triton
// decode kernel" (FreeToken PR #900), "Changes". One CTA owns one
// (request, kv head, head block, KV chunk). It packs the request's R query
// rows times its q heads onto the MMA M axis (row m = i * heads + hh), so the
// kv head's K/V pages are read once for all of them; it streams the chunk's
// pages through a shared-memory ring filled by 16-byte cp.async gathers that
// follow the page table; it masks every row at its own causal position and
// window; it keeps an online softmax per row; and it writes either the final
// output (one chunk) or a normalised partial (o, lse) for stage 2.
// FP8 (OCP E4M3) and int8 caches are widened exactly to 16 bits in shared
// memory;
// per-tensor K scales fold into the logit scale and per-tensor V scales into
// the finalize step ("Naive Support for Hopper FP8 Prefill Kernel with
// Per-Head Quantization", item 3); per-(token, kv head) scales multiply the
// logit column (K) and the probability column (V) of their token.
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "pda_internal.h"

namespace pda {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = 4;
constexpr int kT = 64;  // tokens per shared-memory tile
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------- PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async gather; src_bytes 0 zero-fills the destination.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async4(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

template <bool kF16>
__device__ __forceinline__ void mma16816(float* c, const uint32_t* a, uint32_t b0, uint32_t b1) {
  if constexpr (kF16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

// Two floats -> packed 16-bit pair (low = x, high = y), RNE.
template <bool kF16>
__device__ __forceinline__ uint32_t pack2(float x, float y) {
  if constexpr (kF16) {
    __half2 h = __floats2half2_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(x, y);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Two OCP E4M3 codes (low byte = first element) -> packed f16 pair. Exact:
// every E4M3 value is an f16 normal number.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t codes) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(codes));
  return r;
}

// Two E4M3 codes -> packed value pair of the compute type (exact both ways).
template <bool kF16>
__device__ __forceinline__ uint32_t e4m3x2_to_ct(uint16_t codes) {
  uint32_t h = e4m3x2_to_f16x2(codes);
  if constexpr (kF16) {
    return h;
  } else {
    float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
    return pack2<false>(f.x, f.y);
  }
}

// Two int8 codes (low byte = first element) -> packed bf16 pair. Exact:
// every integer in [-128, 127] is a bf16 value.
__device__ __forceinline__ uint32_t int8x2_to_bf16x2(uint16_t codes) {
  const float lo = static_cast<float>(static_cast<int8_t>(codes & 0xFF));
  const float hi = static_cast<float>(static_cast<int8_t>(codes >> 8));
  return pack2<false>(lo, hi);
}

// Two one-byte cache codes (E4M3 or int8) -> packed compute-type pair.
template <int KVT, bool kF16>
__device__ __forceinline__ uint32_t widen2(uint16_t codes) {
  if constexpr (KVT == PDA_INT8)
    return int8x2_to_bf16x2(codes);
  else
    return e4m3x2_to_ct<kF16>(codes);
}

__device__ __forceinline__ float fast_exp2(float x) { return exp2f(x); }

// Swizzled byte offset of 16-byte chunk `c` of row `r` in a tile whose rows
// are `row_bytes` (a multiple of 128) long: XOR of the chunk's low 3 bits with
// the row's keeps every 8-row ldmatrix access on distinct bank groups.
__device__ __forceinline__ uint32_t swz(int r, int c, int row_bytes) {
  return static_cast<uint32_t>(r * row_bytes + ((c ^ (r & 7)) << 4));
}

// ------------------------------------------------------------ configuration
template <int D, int KVT, int QT, int SMODE>
struct Cfg {
  static constexpr bool kKvFp8 = KVT == PDA_E4M3 || KVT == PDA_INT8;  // one-byte codes, widened
  static constexpr bool kQFp8 = QT == PDA_E4M3;
  static constexpr bool kF16 = kQFp8;  // MMA operand type: f16 for E4M3 queries, else bf16
  static constexpr int kKvBytes = kKvFp8 ? 1 : 2;
  static constexpr int kTileBytes = kT * D * kKvBytes;  // one of K, V
  static constexpr int kStages = (2 * kTileBytes <= 16384) ? 4 : (2 * kTileBytes <= 32768 ? 3 : 2);
  static constexpr int kRow16 = D * 2;                  // bytes of one 16-bit row
  static constexpr int kQBytes = kMmaRowsPerCta * kRow16;
  static constexpr int kRingBytes = kStages * 2 * kTileBytes;
  static constexpr int kMergeStride = D + 8;            // fp32 words per merge row (padded)
  static constexpr int kMergeBytes = kWarps * 16 * kMergeStride * 4 + kWarps * 16 * 2 * 4;
  static constexpr int kRingOrMerge = kRingBytes > kMergeBytes ? kRingBytes : kMergeBytes;
  static constexpr int kConvBytes = kKvFp8 ? 2 * kT * kRow16 : 0;
  static constexpr int kScaleBytes = SMODE == PDA_SCALE_TOKEN_HEAD ? kStages * 2 * kT * 4 : 0;
  static constexpr int kSmem = kQBytes + kRingOrMerge + kConvBytes + kScaleBytes;
  static constexpr int kCpr = D * kKvBytes / 16;        // 16-byte chunks per cached row
  static_assert(kSmem <= 227 * 1024, "stage-1 tile does not fit shared memory");
};

struct RowInfo {
  int lo, hi;  // visible key range [lo, hi] of the row inside this chunk (empty if lo > hi)
};

// ------------------------------------------------------------------ stage 1
template <int D, int KVT, int QT, int SMODE>
__global__ void __launch_bounds__(kThreads, 1) stage1_mma(const __grid_constant__ DecodeArgs a) {
  using C = Cfg<D, KVT, QT, SMODE>;
  constexpr bool kF16 = C::kF16;
  extern __shared__ __align__(128) uint8_t smem[];
  uint8_t* q_s = smem;
  uint8_t* ring = smem + C::kQBytes;
  uint8_t* conv = ring + C::kRingOrMerge;
  float* scl = reinterpret_cast<float*>(conv + C::kConvBytes);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // ---- which work item
  WorkItem wi;
  if (!work_item(a, blockIdx.x, wi)) return;
  const int hb = wi.hb, split = wi.split, hkv = wi.hkv, b = wi.b;
  const int q0 = a.qo_indptr[b];
  const int R = a.qo_indptr[b + 1] - q0;
  const int L = a.kv_len[b];
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
  if (hb >= a.group / hpc) return;  // fewer head blocks are needed for fewer rows
  const int W = a.window ? a.window[b] : 0;
  const int P = a.page_size;
  const SplitRange sr = split_range(L, R, W, P, chunk_for(a, b));
  if (split >= sr.num_splits) return;
  const int chunk = chunk_for(a, b);
  const int page_begin = sr.lo_page + split * chunk;
  const int page_end = min(page_begin + chunk, sr.num_pages);
  const int t_begin = page_begin * P;              // first token of the chunk (tile origin)
  const int t_end = min(page_end * P, L);          // one past the chunk's last real token
  const int ntiles = (t_end - t_begin + kT - 1) / kT;
  const int M = R * hpc;
  const int head0 = hkv * a.group + hb * hpc;      // first q head of this CTA
  const int32_t* ptab = a.page_table + a.kv_indptr[b];

  // ---- scales folded into the logit scale / the finalize step
  float qk_scale = a.sm_scale * kLog2e;            // logits in log2 units
  float v_final = 1.f;
  if constexpr (SMODE == PDA_SCALE_TENSOR) {
    qk_scale *= __ldg(a.k_scale);
    v_final = __ldg(a.v_scale);
  }

  // ---- query tile: rows m < M, zero rows up to the warp tiles in use
  const int mt = (M + 15) >> 4;
  const int mt_eff = mt == 3 ? 4 : mt;
  {
    constexpr int qchunks = D * (C::kQFp8 ? 1 : 2) / 16;  // 16-byte chunks per global row
    for (int idx = tid; idx < mt_eff * 16 * qchunks; idx += kThreads) {
      const int m = idx / qchunks, c = idx % qchunks;
      if constexpr (C::kQFp8) {
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (m < M) {
          const uint8_t* src = static_cast<const uint8_t*>(a.q) +
                               ((int64_t)(q0 + m / hpc) * a.hq + head0 + m % hpc) * D + c * 16;
          raw = __ldg(reinterpret_cast<const uint4*>(src));
        }
        const uint16_t* cw = reinterpret_cast<const uint16_t*>(&raw);
        uint4 lo, hi;
        lo.x = e4m3x2_to_ct<kF16>(cw[0]); lo.y = e4m3x2_to_ct<kF16>(cw[1]);
        lo.z = e4m3x2_to_ct<kF16>(cw[2]); lo.w = e4m3x2_to_ct<kF16>(cw[3]);
        hi.x = e4m3x2_to_ct<kF16>(cw[4]); hi.y = e4m3x2_to_ct<kF16>(cw[5]);
        hi.z = e4m3x2_to_ct<kF16>(cw[6]); hi.w = e4m3x2_to_ct<kF16>(cw[7]);
        *reinterpret_cast<uint4*>(q_s + swz(m, 2 * c, C::kRow16)) = lo;
        *reinterpret_cast<uint4*>(q_s + swz(m, 2 * c + 1, C::kRow16)) = hi;
      } else {
        uint4 raw = make_uint4(0, 0, 0, 0);
        if (m < M) {
          const uint8_t* src = static_cast<const uint8_t*>(a.q) +
                               (((int64_t)(q0 + m / hpc) * a.hq + head0 + m % hpc) * D) * 2 + c * 16;
          raw = __ldg(reinterpret_cast<const uint4*>(src));
        }
        *reinterpret_cast<uint4*>(q_s + swz(m, c, C::kRow16)) = raw;
      }
    }
  }

  // ---- K/V tile gather: tile `jt` into ring stage `st`
  const uint8_t* kbase = static_cast<const uint8_t*>(a.k);
  const uint8_t* vbase = static_cast<const uint8_t*>(a.v);
  const int64_t head_off = (int64_t)hkv * a.sh;
  auto issue_tile = [&](int jt, int st) {
    if (jt < ntiles) {
      const int tok0 = t_begin + jt * kT;
      uint8_t* kst = ring + st * 2 * C::kTileBytes;
      uint8_t* vst = kst + C::kTileBytes;
      for (int idx = tid; idx < kT * C::kCpr; idx += kThreads) {
        const int r = idx / C::kCpr, c = idx % C::kCpr;
        const int tok = tok0 + r;
        int bytes = 0;
        int64_t off = 0;
        if (tok < t_end) {
          const int page = __ldg(ptab + tok / P);
          if (page >= 0 && page < a.num_pages) {
            bytes = 16;
            off = ((int64_t)page * a.sp + (int64_t)(tok % P) * a.st + head_off) * C::kKvBytes +
                  c * 16;
          } else {
            atomicOr(a.status, PDA_STATUS_PAGE_OOB);
          }
        }
        uint32_t dk, dv;
        if constexpr (C::kKvFp8) {  // raw bytes, row-major; widened later
          dk = smem_u32(kst + r * D + c * 16);
          dv = smem_u32(vst + r * D + c * 16);
        } else {
          dk = smem_u32(kst + swz(r, c, C::kRow16));
          dv = smem_u32(vst + swz(r, c, C::kRow16));
        }
        cp_async16(dk, kbase + off, bytes);
        cp_async16(dv, vbase + off, bytes);
      }
      if constexpr (SMODE == PDA_SCALE_TOKEN_HEAD) {
        if (tid < kT) {
          const int tok = tok0 + tid;
          int bytes = 0;
          int64_t sidx = 0;
          if (tok < t_end) {
            const int page = __ldg(ptab + tok / P);
            if (page >= 0 && page < a.num_pages) {
              bytes = 4;
              sidx = ((int64_t)page * P + tok % P) * a.hkv + hkv;
            }
          }
          cp_async4(smem_u32(scl + st * 2 * kT + tid), a.k_scale + sidx, bytes);
          cp_async4(smem_u32(scl + st * 2 * kT + kT + tid), a.v_scale + sidx, bytes);
        }
      }
    }
    cp_async_commit();
  };

  // ---- per-warp role: m-tile `mi`, token slice `ts` of every tile
  const int nslices = kWarps / mt_eff;
  const int mi = warp % mt_eff;
  const int ts = warp / mt_eff;
  const int blocks_per_slice = (kT / 16) / nslices;  // 16-token blocks per warp per tile
  const bool active = mi < mt;
  const int g = lane >> 2, t4 = lane & 3;
  RowInfo ri[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    const int m = mi * 16 + g + 8 * h;
    if (m < M) {
      const int pos = L - R + m / hpc;
      ri[h].lo = W > 0 ? pos - W + 1 : 0;
      ri[h].hi = min(pos, t_end - 1);
    } else {
      ri[h].lo = 1;
      ri[h].hi = 0;  // padded row: sees nothing
    }
  }
  // tokens every real row of the CTA sees: [all_lo, all_hi]
  const int all_hi = min(L - R, t_end - 1);
  const int all_lo = W > 0 ? L - 1 - W + 1 : 0;

  float o[D / 8][4];
#pragma unroll
  for (int n = 0; n < D / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float row_max[2] = {-INFINITY, -INFINITY};
  float row_sum[2] = {0.f, 0.f};

  const uint32_t q_base = smem_u32(q_s) + mi * 16 * C::kRow16;
  // ldmatrix lane roles
  const int a_row = lane & 15, a_chunk = lane >> 4;                 // Q as A (m16 x k16)
  const int bk_row = ((lane >> 4) << 3) + (lane & 7), bk_chunk = (lane >> 3) & 1;  // K as B
  const int bv_row = (lane & 7) + (((lane >> 3) & 1) << 3), bv_chunk = lane >> 4;  // V as B^T

#pragma unroll 1
  for (int s = 0; s < C::kStages - 1; ++s) issue_tile(s, s);

#pragma unroll 1
  for (int j = 0; j < ntiles; ++j) {
    const int st = j % C::kStages;
    issue_tile(j + C::kStages - 1, (j + C::kStages - 1) % C::kStages);
    cp_async_wait<C::kStages - 1>();
    __syncthreads();
    const uint8_t* kt;
    const uint8_t* vt;
    if constexpr (C::kKvFp8) {
      // widen the E4M3 / int8 tile pair to the 16-bit compute type, swizzled
      const uint8_t* kraw = ring + st * 2 * C::kTileBytes;
      const uint8_t* vraw = kraw + C::kTileBytes;
      uint8_t* k16 = conv;
      uint8_t* v16 = conv + kT * C::kRow16;
      for (int idx = tid; idx < 2 * kT * C::kCpr; idx += kThreads) {
        const int which = idx / (kT * C::kCpr);
        const int rem = idx % (kT * C::kCpr);
        const int r = rem / C::kCpr, c = rem % C::kCpr;
        const uint4 raw = *reinterpret_cast<const uint4*>((which ? vraw : kraw) + r * D + c * 16);
        const uint16_t* cw = reinterpret_cast<const uint16_t*>(&raw);
        uint4 lo, hi;
        lo.x = widen2<KVT, kF16>(cw[0]); lo.y = widen2<KVT, kF16>(cw[1]);
        lo.z = widen2<KVT, kF16>(cw[2]); lo.w = widen2<KVT, kF16>(cw[3]);
        hi.x = widen2<KVT, kF16>(cw[4]); hi.y = widen2<KVT, kF16>(cw[5]);
        hi.z = widen2<KVT, kF16>(cw[6]); hi.w = widen2<KVT, kF16>(cw[7]);
        uint8_t* dst = which ? v16 : k16;
        *reinterpret_cast<uint4*>(dst + swz(r, 2 * c, C::kRow16)) = lo;
        *reinterpret_cast<uint4*>(dst + swz(r, 2 * c + 1, C::kRow16)) = hi;
      }
      __syncthreads();
      kt = k16;
      vt = v16;
    } else {
      kt = ring + st * 2 * C::kTileBytes;
      vt = kt + C::kTileBytes;
    }
    const float* ks_t = scl + st * 2 * kT;
    const float* vs_t = ks_t + kT;
    const int tile_tok0 = t_begin + j * kT;

    if (active) {
      const uint32_t k_base = smem_u32(kt), v_base = smem_u32(vt);
#pragma unroll 1
      for (int blk = 0; blk < blocks_per_slice; ++blk) {
        const int r0 = (ts * blocks_per_slice + blk) * 16;  // first token row in the tile
        const int tok0 = tile_tok0 + r0;
        // S = Q K^T for 16 rows x 16 tokens (two n8 tiles)
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          uint32_t qa[4];
          ldsm_x4(q_base + swz(a_row, 2 * kk + a_chunk, C::kRow16), qa[0], qa[1], qa[2], qa[3]);
          uint32_t kb0, kb1, kb2, kb3;
          ldsm_x4(k_base + swz(r0 + bk_row, 2 * kk + bk_chunk, C::kRow16), kb0, kb1, kb2, kb3);
          mma16816<kF16>(sc[0], qa, kb0, kb1);
          mma16816<kF16>(sc[1], qa, kb2, kb3);
        }
        // logit scale (+ per-token K scale), causal/window mask
        const bool full = tok0 >= all_lo && tok0 + 15 <= all_hi;
#pragma unroll
        for (int n = 0; n < 2; ++n) {
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int col = n * 8 + 2 * t4 + (e & 1);
            float x = sc[n][e] * qk_scale;
            if constexpr (SMODE == PDA_SCALE_TOKEN_HEAD) x *= ks_t[r0 + col];
            if (!full) {
              const int tok = tok0 + col;
              const RowInfo& rr = ri[e >> 1];
              if (tok < rr.lo || tok > rr.hi) x = -INFINITY;
            }
            sc[n][e] = x;
          }
        }
        // online softmax per row (rows g and g+8 of the m-tile)
        float alpha[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          float mx = fmaxf(fmaxf(sc[0][2 * h], sc[0][2 * h + 1]), fmaxf(sc[1][2 * h], sc[1][2 * h + 1]));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
          const float m_new = fmaxf(row_max[h], mx);
          const float m_use = m_new == -INFINITY ? 0.f : m_new;
          alpha[h] = fast_exp2(row_max[h] - m_use);
          row_max[h] = m_new;
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            sc[n][2 * h] = fast_exp2(sc[n][2 * h] - m_use);
            sc[n][2 * h + 1] = fast_exp2(sc[n][2 * h + 1] - m_use);
          }
          row_sum[h] = row_sum[h] * alpha[h] + sc[0][2 * h] + sc[0][2 * h + 1] + sc[1][2 * h] +
                       sc[1][2 * h + 1];
        }
        if (__any_sync(0xffffffffu, alpha[0] != 1.f || alpha[1] != 1.f)) {
#pragma unroll
          for (int n = 0; n < D / 8; ++n) {
            o[n][0] *= alpha[0];
            o[n][1] *= alpha[0];
            o[n][2] *= alpha[1];
            o[n][3] *= alpha[1];
          }
        }
        if constexpr (SMODE == PDA_SCALE_TOKEN_HEAD) {
#pragma unroll
          for (int n = 0; n < 2; ++n) {
            const float v0 = vs_t[r0 + n * 8 + 2 * t4], v1 = vs_t[r0 + n * 8 + 2 * t4 + 1];
            sc[n][0] *= v0; sc[n][1] *= v1; sc[n][2] *= v0; sc[n][3] *= v1;
          }
        }
        // O += P V  (P from the S accumulators: the m16n8 C layout of two n8
        // tiles is the m16k16 A layout)
        uint32_t pa[4];
        pa[0] = pack2<kF16>(sc[0][0], sc[0][1]);
        pa[1] = pack2<kF16>(sc[0][2], sc[0][3]);
        pa[2] = pack2<kF16>(sc[1][0], sc[1][1]);
        pa[3] = pack2<kF16>(sc[1][2], sc[1][3]);
#pragma unroll
        for (int nn = 0; nn < D / 16; ++nn) {
          uint32_t vb0, vb1, vb2, vb3;
          ldsm_x4_t(v_base + swz(r0 + bv_row, 2 * nn + bv_chunk, C::kRow16), vb0, vb1, vb2, vb3);
          mma16816<kF16>(o[2 * nn], pa, vb0, vb1);
          mma16816<kF16>(o[2 * nn + 1], pa, vb2, vb3);
        }
      }
    }
    __syncthreads();  // stage `st` (and the widened tile) may be refilled now
  }
  cp_async_wait<0>();
  __syncthreads();
  // Let stage 2 start launching; it waits for this grid's memory anyway.
  asm volatile("griddepcontrol.launch_dependents;\n" ::);

  // ---- merge the token slices of each m-tile through shared memory
  float* mo = reinterpret_cast<float*>(ring);
  float* mml = mo + kWarps * 16 * C::kMergeStride;  // [warp][16][2] = (max, sum)
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    row_sum[h] += __shfl_xor_sync(0xffffffffu, row_sum[h], 1);
    row_sum[h] += __shfl_xor_sync(0xffffffffu, row_sum[h], 2);
  }
  if (active) {
#pragma unroll
    for (int n = 0; n < D / 8; ++n) {
      float* r0p = mo + (warp * 16 + g) * C::kMergeStride + n * 8 + 2 * t4;
      float* r1p = r0p + 8 * C::kMergeStride;
      *reinterpret_cast<float2*>(r0p) = make_float2(o[n][0], o[n][1]);
      *reinterpret_cast<float2*>(r1p) = make_float2(o[n][2], o[n][3]);
    }
    if (t4 == 0) {
      mml[(warp * 16 + g) * 2] = row_max[0];
      mml[(warp * 16 + g) * 2 + 1] = row_sum[0];
      mml[(warp * 16 + g + 8) * 2] = row_max[1];
      mml[(warp * 16 + g + 8) * 2 + 1] = row_sum[1];
    }
  }
  __syncthreads();

  const bool single = sr.num_splits == 1;
  constexpr int kC4 = D / 4;
  for (int idx = tid; idx < M * kC4; idx += kThreads) {
    const int m = idx / kC4, c4 = idx % kC4;
    const int mtile = m >> 4, r = m & 15;
    float mstar = -INFINITY;
    for (int s2 = 0; s2 < nslices; ++s2)
      mstar = fmaxf(mstar, mml[((s2 * mt_eff + mtile) * 16 + r) * 2]);
    float lsum = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mstar != -INFINITY) {
      for (int s2 = 0; s2 < nslices; ++s2) {
        const int w = s2 * mt_eff + mtile;
        const float ms = mml[(w * 16 + r) * 2];
        if (ms == -INFINITY) continue;
        const float f = fast_exp2(ms - mstar);
        lsum += f * mml[(w * 16 + r) * 2 + 1];
        const float4 x = *reinterpret_cast<const float4*>(mo + (w * 16 + r) * C::kMergeStride + c4 * 4);
        acc.x += f * x.x; acc.y += f * x.y; acc.z += f * x.z; acc.w += f * x.w;
      }
    }
    const float inv = lsum > 0.f ? v_final / lsum : 0.f;
    acc.x *= inv; acc.y *= inv; acc.z *= inv; acc.w *= inv;
    const float lse2 = lsum > 0.f ? mstar + __log2f(lsum) : -INFINITY;
    const int64_t row = q0 + m / hpc;
    const int head = head0 + m % hpc;
    if (single) {
      __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + (row * a.hq + head) * D + c4 * 4;
      __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 pk;
      pk.x = *reinterpret_cast<uint32_t*>(&lo);
      pk.y = *reinterpret_cast<uint32_t*>(&hi);
      *reinterpret_cast<uint2*>(dst) = pk;
      if (c4 == 0 && a.lse) a.lse[row * a.hq + head] = lse2 * kLn2;
    } else {
      const int64_t prow = ((int64_t)split * a.rows_cap + row) * a.hq + head;
      *reinterpret_cast<float4*>(a.part_o + prow * D + c4 * 4) = acc;
      if (c4 == 0) a.part_lse[prow] = lse2;
    }
  }
}

// ------------------------------------------------------------------ stage 2
// Log-sum-exp merge of the chunk partials, one output row per (request, row,
// q head) ("Stage 2 merges per row"). A warp owns a slice of 32 x VW
// consecutive floats of the row (VW = 4, or 2 at head_dim 64), so each
// partial is one coalesced vector load per lane; WPI warps per slice share
// the row's splits. Each warp merges its own splits online -- a running
// maximum of their LSEs, its sums rescaled when the maximum rises -- with all
// of a batch's loads (LSE and partial output) in flight at once, so a warp
// with at most kBatch splits waits for one round of loads; the WPI warps then
// combine their (maximum, sum, output) triples through shared memory. With
// SPLIT, a CTA holds one slice of a row (its WPI warps), so that a row of
// many splits spreads over kSlices CTAs and more warps share its splits.
template <int D, int WPI, int SPLIT = 0>
struct MergeCfg {
  static constexpr int kVW = D >= 128 ? 4 : 2;                  // floats per lane
  static constexpr int kSlices = D / (32 * kVW);                // warps across the row
  static constexpr int kSlicesCta = SPLIT ? 1 : kSlices;        // ... within one CTA
  static constexpr int kWarpsPerItem = kSlicesCta * WPI;        // <= 32
  // (row, or with SPLIT (row, slice)) units per CTA
  static constexpr int kItems = kWarpsPerItem >= 8 ? 1 : 8 / kWarpsPerItem;
  static constexpr int kThreads = kItems * kWarpsPerItem * 32;
  static constexpr int kBatch = 12;                             // partials in flight
};

template <int D, int WPI, int SPLIT>
__global__ void __launch_bounds__(MergeCfg<D, WPI, SPLIT>::kThreads)
    stage2_merge(const __grid_constant__ DecodeArgs a) {
  using M = MergeCfg<D, WPI, SPLIT>;
  constexpr int kVW = M::kVW;
  __shared__ __align__(16) float sh_acc[M::kThreads / 32][32 * kVW];
  __shared__ float sh_m[M::kThreads / 32];
  __shared__ float sh_l[M::kThreads / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int wi = warp % M::kWarpsPerItem;
  const int64_t unit = (int64_t)blockIdx.x * M::kItems + warp / M::kWarpsPerItem;
  const int sub = wi / M::kSlicesCta;
  const int slice = SPLIT ? static_cast<int>(unit % M::kSlices) : wi % M::kSlices;
  const int64_t item = a.merge_item0 + (SPLIT ? unit / M::kSlices : unit);
  const int64_t per_b = (int64_t)a.max_q_len * a.hq;
  bool valid = false;
  int n = 0;
  int64_t base = 0;
  const int b = static_cast<int>(item / per_b);
  if (b < a.batch) {
    const int rem = static_cast<int>(item % per_b);
    const int i = rem / a.hq, head = rem % a.hq;
    const int q0 = a.qo_indptr[b];
    const int R = a.qo_indptr[b + 1] - q0;
    const int L = a.kv_len[b];
    const int W = a.window ? a.window[b] : 0;
    if (i < R && R <= a.max_q_len && L >= R && L <= a.max_kv_len && q0 + R <= a.rows_cap) {
      const SplitRange sr = split_range(L, R, W, a.page_size, chunk_for(a, b));
      n = sr.num_splits;
      valid = n > 1;  // one split: stage 1 wrote the final result
      base = (int64_t)(q0 + i) * a.hq + head;
    }
  }
  // everything above overlaps stage 1's tail; its partials are read below
  asm volatile("griddepcontrol.wait;\n" ::: "memory");
  const int64_t stride = a.rows_cap * a.hq;  // partial rows per split
  const int col = slice * 32 * kVW + lane * kVW;
  float m = -INFINITY, l = 0.f;  // running maximum (log2) and sum of this warp's splits
  float acc[kVW];
#pragma unroll
  for (int e = 0; e < kVW; ++e) acc[e] = 0.f;
  if (valid) {
    for (int s0 = sub; s0 < n; s0 += M::kBatch * WPI) {
      float ls[M::kBatch];
      float x[M::kBatch][kVW];
      // issue the batch's loads first, then combine
#pragma unroll
      for (int u = 0; u < M::kBatch; ++u) {
        const int s = s0 + u * WPI;
        ls[u] = -INFINITY;
#pragma unroll
        for (int e = 0; e < kVW; ++e) x[u][e] = 0.f;
        if (s < n) {
          ls[u] = a.part_lse[s * stride + base];
          const float* src = a.part_o + (s * stride + base) * D + col;
          if constexpr (kVW == 4) {
            const float4 v = *reinterpret_cast<const float4*>(src);
            x[u][0] = v.x; x[u][1] = v.y; x[u][2] = v.z; x[u][3] = v.w;
          } else {
            const float2 v = *reinterpret_cast<const float2*>(src);
            x[u][0] = v.x; x[u][1] = v.y;
          }
        }
      }
      float bm = m;
#pragma unroll
      for (int u = 0; u < M::kBatch; ++u) bm = fmaxf(bm, ls[u]);
      if (bm > m) {  // the maximum rose: rescale what this warp has summed
        const float f = exp2f(m - bm);  // m = -inf: nothing summed yet, f = 0
        l *= f;
#pragma unroll
        for (int e = 0; e < kVW; ++e) acc[e] *= f;
        m = bm;
      }
#pragma unroll
      for (int u = 0; u < M::kBatch; ++u) {
        const float w = ls[u] == -INFINITY ? 0.f : exp2f(ls[u] - m);
        l += w;
        // an empty split's partial may hold anything: select, do not scale
#pragma unroll
        for (int e = 0; e < kVW; ++e) acc[e] = w > 0.f ? fmaf(w, x[u][e], acc[e]) : acc[e];
      }
    }
  }
  if constexpr (WPI > 1) {
#pragma unroll
    for (int e = 0; e < kVW; ++e) sh_acc[warp][lane * kVW + e] = acc[e];
    if (lane == 0) {
      sh_m[warp] = m;
      sh_l[warp] = l;
    }
    __syncthreads();
    if (sub == 0) {
      float mx = m;
      for (int k = 1; k < WPI; ++k) mx = fmaxf(mx, sh_m[warp + k * M::kSlicesCta]);
      if (mx != -INFINITY) {
        const float f0 = exp2f(m - mx);
        l *= f0;
#pragma unroll
        for (int e = 0; e < kVW; ++e) acc[e] *= f0;
        for (int k = 1; k < WPI; ++k) {
          const int w2 = warp + k * M::kSlicesCta;  // same slice, split group k
          const float mk = sh_m[w2];
          if (mk == -INFINITY) continue;
          const float f = exp2f(mk - mx);
          l = fmaf(f, sh_l[w2], l);
#pragma unroll
          for (int e = 0; e < kVW; ++e) acc[e] = fmaf(f, sh_acc[w2][lane * kVW + e], acc[e]);
        }
      }
      m = mx;
    }
  }
  if (!valid || sub != 0) return;
  const float inv = l > 0.f ? 1.f / l : 0.f;
  __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(a.out) + base * D + col;
  if constexpr (kVW == 4) {
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2] * inv, acc[3] * inv);
    uint2 pk;
    pk.x = *reinterpret_cast<uint32_t*>(&lo);
    pk.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = pk;
  } else {
    *reinterpret_cast<__nv_bfloat162*>(dst) = __floats2bfloat162_rn(acc[0] * inv, acc[1] * inv);
  }
  if (slice == 0 && lane == 0 && a.lse)
    a.lse[base] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
}

// ---------------------------------------------------------------- dispatch
using KernelFn = void (*)(DecodeArgs);

template <int D>
KernelFn pick_stage1(int kv, int qd, int sm) {
  if (kv == PDA_BF16) return stage1_mma<D, PDA_BF16, PDA_BF16, PDA_SCALE_NONE>;
  if (kv == PDA_INT8) {
    if (sm == PDA_SCALE_TENSOR) return stage1_mma<D, PDA_INT8, PDA_BF16, PDA_SCALE_TENSOR>;
    return stage1_mma<D, PDA_INT8, PDA_BF16, PDA_SCALE_TOKEN_HEAD>;
  }
  if (qd == PDA_BF16) {
    if (sm == PDA_SCALE_TENSOR) return stage1_mma<D, PDA_E4M3, PDA_BF16, PDA_SCALE_TENSOR>;
    return stage1_mma<D, PDA_E4M3, PDA_BF16, PDA_SCALE_TOKEN_HEAD>;
  }
  if (sm == PDA_SCALE_TENSOR) return stage1_mma<D, PDA_E4M3, PDA_E4M3, PDA_SCALE_TENSOR>;
  return stage1_mma<D, PDA_E4M3, PDA_E4M3, PDA_SCALE_TOKEN_HEAD>;
}

template <int D>
int smem_of(int kv, int qd, int sm) {
  if (kv == PDA_BF16) return Cfg<D, PDA_BF16, PDA_BF16, PDA_SCALE_NONE>::kSmem;
  if (kv == PDA_INT8) {
    if (sm == PDA_SCALE_TENSOR) return Cfg<D, PDA_INT8, PDA_BF16, PDA_SCALE_TENSOR>::kSmem;
    return Cfg<D, PDA_INT8, PDA_BF16, PDA_SCALE_TOKEN_HEAD>::kSmem;
  }
  if (qd == PDA_BF16) {
    if (sm == PDA_SCALE_TENSOR) return Cfg<D, PDA_E4M3, PDA_BF16, PDA_SCALE_TENSOR>::kSmem;
    return Cfg<D, PDA_E4M3, PDA_BF16, PDA_SCALE_TOKEN_HEAD>::kSmem;
  }
  if (sm == PDA_SCALE_TENSOR) return Cfg<D, PDA_E4M3, PDA_E4M3, PDA_SCALE_TENSOR>::kSmem;
  return Cfg<D, PDA_E4M3, PDA_E4M3, PDA_SCALE_TOKEN_HEAD>::kSmem;
}

KernelFn stage1_for(const pda_plan_t* p) {
  switch (p->head_dim) {
    case 64: return pick_stage1<64>(p->kv_dtype, p->q_dtype, p->scale_mode);
    case 128: return pick_stage1<128>(p->kv_dtype, p->q_dtype, p->scale_mode);
    case 256: return pick_stage1<256>(p->kv_dtype, p->q_dtype, p->scale_mode);
    default: return nullptr;  // head_dim 512: tcgen05 path only
  }
}

// Warps per slice of a merged row: one up to 12 splits, then up to 12
// splits a warp (one round of loads each), up to 8 warps (16 where each
// slice has a CTA of its own) so that a CTA of at most 512 threads keeps
// its batch of partials in registers. Rows of 512 channels with more than
// 12 splits give each slice its own CTA (SPLIT: up to 16 warps share a
// slice's splits) when the rows' slices still fit one CTA per SM -- few
// rows of many splits, as at bs 1 with 16 rows x heads (measured: head_dim
// 512 bf16 bs 1 R 1 37.6 -> 34.8 us per call); with more rows the extra CTAs
// cost more than the shorter rounds save (bs 1 R 8: +1.3 to +1.7 us), and
// at 256 channels (two slices) the call moved by less than its noise.
static int stage2_wpi(const pda_plan_t* p, bool split) {
  const int s = p->max_splits;
  const int w = s <= 12 ? 1 : s <= 24 ? 2 : s <= 48 ? 4 : s <= 96 ? 8 : 16;
  return split ? w : (w > 8 ? 8 : (p->head_dim_v == 512 && w > 4 ? 4 : w));
}
struct Stage2Launch {
  KernelFn fn;
  int units_per_cta, threads, slices;  // slices: CTAs per row (1 unless SPLIT)
};
template <int D, int WPI, int SPLIT>
Stage2Launch stage2_entry() {
  using M = MergeCfg<D, WPI, SPLIT>;
  return {stage2_merge<D, WPI, SPLIT>, M::kItems, M::kThreads, SPLIT ? M::kSlices : 1};
}
template <int D>
Stage2Launch stage2_pick(int wpi) {
  switch (wpi) {
    case 1: return stage2_entry<D, 1, 0>();
    case 2: return stage2_entry<D, 2, 0>();
    case 4: return stage2_entry<D, 4, 0>();
    default: return stage2_entry<D, (D == 512 ? 4 : 8), 0>();
  }
}
template <int D>
Stage2Launch stage2_pick_split(int wpi) {
  switch (wpi) {
    case 2: return stage2_entry<D, 2, 1>();
    case 4: return stage2_entry<D, 4, 1>();
    case 8: return stage2_entry<D, 8, 1>();
    default: return stage2_entry<D, 16, 1>();
  }
}
Stage2Launch stage2_for(const pda_plan_t* p, int64_t items) {
  // the merged rows have the value channels
  const bool split = p->head_dim_v == 512 && p->max_splits > 12 && items * 4 <= p->num_sms;
  const int wpi = stage2_wpi(p, split);
  if (split) return stage2_pick_split<512>(wpi);
  switch (p->head_dim_v) {
    case 64: return stage2_pick<64>(wpi);
    case 128: return stage2_pick<128>(wpi);
    case 256: return stage2_pick<256>(wpi);
    default: return stage2_pick<512>(wpi);
  }
}

}  // namespace

int mma_smem_bytes(const pda_plan_t* p) {
  switch (p->head_dim) {
    case 64: return smem_of<64>(p->kv_dtype, p->q_dtype, p->scale_mode);
    case 128: return smem_of<128>(p->kv_dtype, p->q_dtype, p->scale_mode);
    case 256: return smem_of<256>(p->kv_dtype, p->q_dtype, p->scale_mode);
    default: return -1;  // head_dim 512: no mma.sync build
  }
}

int mma_ctas_per_sm(const pda_plan_t* p) {
  // 228 KB of shared memory per SM, 1 KB reserved per CTA; the kernel is
  // built for at most 255 registers x 128 threads, so shared memory decides.
  const int per = mma_smem_bytes(p) + 1024;
  int n = (228 * 1024) / per;
  return n < 1 ? 1 : (n > 4 ? 4 : n);
}

int launch_stage1_mma(const pda_plan_t* plan, const DecodeArgs& args, cudaStream_t s) {
  KernelFn k1 = stage1_for(plan);
  if (!k1) return PDA_ERR_UNSUPPORTED;
  const int smem = plan->stage1_smem_bytes;
  if (cudaFuncSetAttribute(reinterpret_cast<const void*>(k1),
                           cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess) {
    cudaGetLastError();
    return PDA_ERR_CUDA;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(plan->grid_ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  if (cudaLaunchKernelEx(&cfg, k1, args) != cudaSuccess) {
    cudaGetLastError();
    return PDA_ERR_CUDA;
  }
  return PDA_OK;
}

int launch_stage2(const pda_plan_t* plan, const DecodeArgs& args, cudaStream_t s) {
  // when only the tail requests are split, the merge covers just their items
  DecodeArgs a = args;
  const int64_t per_b = (int64_t)args.max_q_len * plan->num_qo_heads;
  const int64_t b0 = plan->head_splits == 1 ? plan->tail_from : 0;
  a.merge_item0 = b0 * per_b;
  const int64_t items = (int64_t)(plan->batch - b0) * per_b;
  if (items <= 0) return PDA_OK;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t c2 = {};
  const Stage2Launch l2 = stage2_for(plan, items);
  const int64_t units = items * l2.slices;
  const int per_cta = l2.units_per_cta;
  c2.gridDim = dim3(static_cast<unsigned>((units + per_cta - 1) / per_cta));
  c2.blockDim = dim3(static_cast<unsigned>(l2.threads));
  c2.dynamicSmemBytes = 0;
  c2.stream = s;
  c2.attrs = attr;
  c2.numAttrs = 1;
  if (cudaLaunchKernelEx(&c2, l2.fn, a) != cudaSuccess) {
    cudaGetLastError();
    return PDA_ERR_CUDA;
  }
  return PDA_OK;
}

}  // namespace pda
