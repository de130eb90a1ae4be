// Quantise-on-append: the new rows' K and V into the paged cache.
//
// The step before decode reads them: the fp8_per_token_head cache of
// "perf(attention): run up to 8 query rows per request in the triton decode
// kernel" (End-to-end A/B) keeps one fp32 scale per (token, kv head); the
// "fp8 support" page (Functionality) uses symmetric per-tensor scales. One
// warp per (request, row, kv head): it loads the row's D bf16 values of K
// and of V (D / 32 per lane), takes the amax over D with warp shuffles when
// the scale is per token, and stores E4M3 or int8 codes (or the bf16
// values) into the token's page slot. MLA records ("fp8 support", the
// reviewers' 8-bit nope per 128 channels with 16-bit rope) take the latent
// alone: a scale per 128-channel block, then the rope copied. HBM-bound;
// every access is one contiguous row.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>

#include "pda.h"
#include "pda_internal.h"

namespace pda {
namespace {

struct AppendArgs {
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const int32_t* page_table;
  const int32_t* kv_indptr;
  const int32_t* kv_len;
  const int32_t* qo_indptr;
  uint8_t* k_pages;
  uint8_t* v_pages;
  float* k_scale;
  float* v_scale;
  uint32_t* status;
  int64_t sp, st, sh;  // cache strides, elements
  int batch, hkv, page_size, num_pages, max_q_len;
};

// Two floats -> two E4M3 codes (RNE, saturating to +-448): low byte from `lo`.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// Two floats -> two symmetric int8 codes (nearest, ties to even, clamped to
// +-127; NaN -> 0): low byte from `lo`.
__device__ __forceinline__ uint16_t int8x2(float lo, float hi) {
  auto one = [](float y) -> uint32_t {
    int v = isnan(y) ? 0 : __float2int_rn(y);
    v = v > 127 ? 127 : (v < -127 ? -127 : v);
    return static_cast<uint32_t>(v) & 0xFFu;
  };
  return static_cast<uint16_t>(one(lo) | (one(hi) << 8));
}

// One row (D bf16 values, kPer per lane) into the cache at byte offset `dst`
// of `pages`; per-token scale written to `scale_out` by lane 0. MODE: 0 bf16
// copy, 1 / 2 E4M3 per tensor / per token-head, 3 / 4 int8 likewise.
template <int D, int MODE>
__device__ __forceinline__ void put_row(const __nv_bfloat16* src, uint8_t* pages, int64_t elt_off,
                                        const float* scale_in, float* scale_out, int lane) {
  constexpr int kPer = D / 32;
  // load this lane's kPer bf16 values (2 * kPer bytes, aligned)
  uint32_t raw[kPer / 2];
  const uint32_t* s32 = reinterpret_cast<const uint32_t*>(src + lane * kPer);
#pragma unroll
  for (int e = 0; e < kPer / 2; ++e) raw[e] = __ldg(s32 + e);
  if constexpr (MODE == 0) {
    uint32_t* d32 = reinterpret_cast<uint32_t*>(pages + elt_off * 2 + lane * kPer * 2);
#pragma unroll
    for (int e = 0; e < kPer / 2; ++e) d32[e] = raw[e];
    return;
  } else {
    float x[kPer];
#pragma unroll
    for (int e = 0; e < kPer / 2; ++e) {
      x[2 * e] = __uint_as_float(raw[e] << 16);
      x[2 * e + 1] = __uint_as_float(raw[e] & 0xFFFF0000u);
    }
    constexpr bool kInt8 = MODE >= 3;
    float s;
    if constexpr (MODE == 1 || MODE == 3) {
      s = __ldg(scale_in);
    } else {
      float amax = 0.f;
#pragma unroll
      for (int e = 0; e < kPer; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
      for (int off = 16; off; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
      s = amax > 0.f ? __fdiv_rn(amax, kInt8 ? 127.f : 448.f) : 1.f;
      if (lane == 0) *scale_out = s;
    }
    uint16_t c[kPer / 2];
#pragma unroll
    for (int e = 0; e < kPer / 2; ++e) {
      const float y0 = __fdiv_rn(x[2 * e], s), y1 = __fdiv_rn(x[2 * e + 1], s);
      c[e] = kInt8 ? int8x2(y0, y1) : e4m3x2(y0, y1);
    }
    uint8_t* dst = pages + elt_off + lane * kPer;
    if constexpr (kPer == 2) {
      *reinterpret_cast<uint16_t*>(dst) = c[0];
    } else if constexpr (kPer == 4) {
      *reinterpret_cast<uint32_t*>(dst) = c[0] | (static_cast<uint32_t>(c[1]) << 16);
    } else if constexpr (kPer == 8) {
      *reinterpret_cast<uint2*>(dst) = make_uint2(c[0] | (static_cast<uint32_t>(c[1]) << 16),
                                                  c[2] | (static_cast<uint32_t>(c[3]) << 16));
    } else {
      *reinterpret_cast<uint4*>(dst) = make_uint4(c[0] | (static_cast<uint32_t>(c[1]) << 16),
                                                  c[2] | (static_cast<uint32_t>(c[3]) << 16),
                                                  c[4] | (static_cast<uint32_t>(c[5]) << 16),
                                                  c[6] | (static_cast<uint32_t>(c[7]) << 16));
    }
  }
}

// One MLA record (MODE 5): the row's 576 bf16 latent values -> 512 E4M3
// nope codes, each 128-channel block with its own amax / 448 scale (lane l
// holds channels 16l .. 16l + 15 of block l / 8; the block's amax is a
// shuffle over its 8 lanes), then the 64 rope values copied as bf16.
__device__ __forceinline__ void put_mla_record(const __nv_bfloat16* src, uint8_t* rec,
                                               float* scales, int lane) {
  const uint4* s4 = reinterpret_cast<const uint4*>(src + lane * 16);
  const uint4 w0 = __ldg(s4), w1 = __ldg(s4 + 1);
  const uint32_t raw[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
  float x[16];
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    x[2 * e] = __uint_as_float(raw[e] << 16);
    x[2 * e + 1] = __uint_as_float(raw[e] & 0xFFFF0000u);
  }
  float amax = 0.f;
#pragma unroll
  for (int e = 0; e < 16; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
  for (int off = 1; off < 8; off <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  // a zero block: scale 0 (no weight in the decode's sums) and zero codes
  const float sc = amax > 0.f ? __fdiv_rn(amax, 448.f) : 0.f;
  const float dv = amax > 0.f ? sc : 1.f;
  if ((lane & 7) == 0) scales[lane >> 3] = sc;
  uint32_t c[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint16_t lo = e4m3x2(__fdiv_rn(x[4 * e], dv), __fdiv_rn(x[4 * e + 1], dv));
    const uint16_t hi = e4m3x2(__fdiv_rn(x[4 * e + 2], dv), __fdiv_rn(x[4 * e + 3], dv));
    c[e] = lo | (static_cast<uint32_t>(hi) << 16);
  }
  *reinterpret_cast<uint4*>(rec + lane * 16) = make_uint4(c[0], c[1], c[2], c[3]);
  // rope: two bf16 per lane
  *reinterpret_cast<uint32_t*>(rec + 512 + lane * 4) =
      __ldg(reinterpret_cast<const uint32_t*>(src + 512) + lane);
}

template <int D, int MODE>
__global__ void __launch_bounds__(256) append_kv(const __grid_constant__ AppendArgs a) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t item = (int64_t)blockIdx.x * 8 + warp;
  const int64_t per_b = (int64_t)a.max_q_len * a.hkv;
  const int b = static_cast<int>(item / per_b);
  if (b >= a.batch) return;
  const int rem = static_cast<int>(item % per_b);
  const int i = rem / a.hkv, h = rem % a.hkv;
  const int q0 = a.qo_indptr[b];
  const int R = a.qo_indptr[b + 1] - q0;
  const int L = a.kv_len[b];
  const bool reporter = i == 0 && h == 0 && lane == 0;
  if (R < 0 || R > a.max_q_len) {
    if (reporter) atomicOr(a.status, PDA_STATUS_ROWS_GT_MAX);
    return;
  }
  if (i >= R) return;
  if (L < R) {
    if (reporter) atomicOr(a.status, PDA_STATUS_KV_LEN_LT_ROWS);
    return;
  }
  const int t = L - R + i;
  const int P = a.page_size;
  const int page = a.page_table[a.kv_indptr[b] + t / P];
  const int slot = t % P;
  if (page < 0 || page >= a.num_pages) {
    if (lane == 0) atomicOr(a.status, PDA_STATUS_PAGE_OOB);
    return;
  }
  const int64_t off = page * a.sp + slot * a.st + h * a.sh;  // elements
  const int64_t row = ((int64_t)(q0 + i) * a.hkv + h) * D;
  const int64_t sidx = ((int64_t)page * P + slot) * a.hkv + h;
  if constexpr (MODE == 5) {  // MLA record: the latent is both K and V
    put_mla_record(a.k_new + row, a.k_pages + off, a.k_scale + sidx * 4, lane);
    return;
  }
  constexpr bool kPerToken = MODE == 2 || MODE == 4;
  put_row<D, MODE>(a.k_new + row, a.k_pages, off, a.k_scale, a.k_scale + (kPerToken ? sidx : 0),
                   lane);
  put_row<D, MODE>(a.v_new + row, a.v_pages, off, a.v_scale, a.v_scale + (kPerToken ? sidx : 0),
                   lane);
}

using AppendFn = void (*)(AppendArgs);

template <int D>
AppendFn pick_mode(int mode) {
  if constexpr (D == 576) {
    return append_kv<576, 5>;  // MLA records only
  } else {
    switch (mode) {
      case 0: return append_kv<D, 0>;
      case 1: return append_kv<D, 1>;
      case 2: return append_kv<D, 2>;
      case 3: return append_kv<D, 3>;
      default: return append_kv<D, 4>;
    }
  }
}

}  // namespace
}  // namespace pda

extern "C" int pda_append_kv(const pda_plan_t* plan, const void* k_new, const void* v_new,
                             const int32_t* page_table, const int32_t* kv_indptr,
                             const int32_t* kv_len, const int32_t* qo_indptr, int32_t max_q_len,
                             void* k_pages, void* v_pages, float* k_scale, float* v_scale,
                             void* split_scratch, pda_stream_t stream) {
  if (!plan) return PDA_ERR_NULL;
  if (plan->magic != PDA_PLAN_MAGIC) return PDA_ERR_PLAN;
  // MLA records: one latent (k_new into k_pages, scales into k_scale); the
  // v arguments are not used
  const bool rec = plan->scale_mode == PDA_SCALE_MLA_BLOCK;
  if (!k_new || (!v_new && !rec) || !page_table || !kv_indptr || !kv_len || !qo_indptr ||
      !k_pages || (!v_pages && !rec))
    return PDA_ERR_NULL;
  if (!split_scratch) return PDA_ERR_SCRATCH;
  if (reinterpret_cast<uintptr_t>(split_scratch) % 256) return PDA_ERR_SCRATCH;
  if (max_q_len < 1 || max_q_len > plan->max_q_len) return PDA_ERR_INVALID;
  const bool fp8 = plan->kv_dtype != PDA_BF16;  // one-byte codes (E4M3 or int8) with scales
  if (fp8 && (!k_scale || (!v_scale && !rec))) return PDA_ERR_NULL;
  if (fp8 && plan->scale_mode == PDA_SCALE_NONE) return PDA_ERR_UNSUPPORTED;
  auto a16 = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
  if (rec) {
    if (!a16(k_new) || !a16(k_pages) || !a16(k_scale)) return PDA_ERR_ALIGNMENT;
  } else {
    if (!a16(k_new) || !a16(v_new) || !a16(k_pages) || !a16(v_pages)) return PDA_ERR_ALIGNMENT;
    if (fp8 && (reinterpret_cast<uintptr_t>(k_scale) % 4 || reinterpret_cast<uintptr_t>(v_scale) % 4))
      return PDA_ERR_ALIGNMENT;
  }
  const int D = plan->head_dim;
  if (D != 64 && D != 128 && D != 256 && D != 512 && !(D == 576 && rec)) return PDA_ERR_UNSUPPORTED;
  if (rec && D != 576) return PDA_ERR_UNSUPPORTED;
  if (plan->batch == 0) return PDA_OK;

  pda::AppendArgs a;
  std::memset(&a, 0, sizeof a);
  a.k_new = static_cast<const __nv_bfloat16*>(k_new);
  a.v_new = static_cast<const __nv_bfloat16*>(v_new);
  a.page_table = page_table;
  a.kv_indptr = kv_indptr;
  a.kv_len = kv_len;
  a.qo_indptr = qo_indptr;
  a.k_pages = static_cast<uint8_t*>(k_pages);
  a.v_pages = static_cast<uint8_t*>(v_pages);
  a.k_scale = fp8 ? k_scale : nullptr;
  a.v_scale = fp8 ? v_scale : nullptr;
  a.status = static_cast<uint32_t*>(split_scratch);
  a.sp = plan->kv_stride_page;
  a.st = plan->kv_stride_token;
  a.sh = plan->kv_stride_head;
  a.batch = plan->batch;
  a.hkv = plan->num_kv_heads;
  a.page_size = plan->page_size;
  a.num_pages = plan->num_pages;
  a.max_q_len = max_q_len;
  const int mode = rec ? 5
                 : !fp8 ? 0
                        : (plan->kv_dtype == PDA_INT8 ? 2 : 0) +
                              (plan->scale_mode == PDA_SCALE_TENSOR ? 1 : 2);
  pda::AppendFn fn = D == 64 ? pda::pick_mode<64>(mode)
                     : D == 128 ? pda::pick_mode<128>(mode)
                     : D == 256 ? pda::pick_mode<256>(mode)
                     : D == 512 ? pda::pick_mode<512>(mode)
                                : pda::pick_mode<576>(mode);
  const int64_t warps = (int64_t)plan->batch * max_q_len * plan->num_kv_heads;
  const int64_t blocks = (warps + 7) / 8;
  if (blocks > 0x7fffffffLL) return PDA_ERR_INVALID;
  fn<<<static_cast<unsigned>(blocks), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
  if (cudaGetLastError() != cudaSuccess) return PDA_ERR_CUDA;
  return PDA_OK;
}
