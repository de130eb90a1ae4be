// pda_internal.h -- shared between the planner (host C++) and the CUDA
// translation units. Not part of the public ABI.
#pragma once

#include <stdint.h>

#include <cuda_runtime.h>

#include "pda.h"

#ifdef __CUDACC__
#define PDA_HD __host__ __device__ __forceinline__
#else
#define PDA_HD inline
#endif

namespace pda {

constexpr int kStatusHeaderBytes = 256;  // status word + padding at the start of split_scratch
constexpr int kMaxQLen = 8;              // rows per request ("up to 8 query rows")
constexpr int kMmaRowsPerCta = 64;       // mma.sync path: 4 warps x m16 tiles
constexpr int kTcRowsPerCta = 64;        // tcgen05 path: N of the swapped QK^T MMA

// Arguments of both stage-1 variants and of stage 2 (passed by value).
struct DecodeArgs {
  const void* q;
  const void* k;
  const void* v;
  const int32_t* page_table;
  const int32_t* kv_indptr;
  const int32_t* kv_len;
  const int32_t* qo_indptr;
  const int32_t* window;
  const float* k_scale;
  const float* v_scale;
  void* out;
  float* lse;
  float* part_o;      // [max_splits][rows_cap][Hq][D] fp32, normalised partial output
  float* part_lse;    // [max_splits][rows_cap][Hq] fp32, log2-domain partial LSE
  uint32_t* status;   // sticky device status bits
  float sm_scale;
  int64_t sp, st, sh; // cache strides (elements)
  int batch, hq, hkv, group, head_dim, page_size, num_pages;
  int head_dim_v;  // value channels (MLA: 512 of a 576-channel latent)
  int max_q_len, max_kv_len, max_splits, head_blocks, chunk_pages;
  int tail_from, tail_chunk_pages, head_splits, tail_splits;  // see pda_plan_t
  int64_t merge_item0;  // first (request, row, q head) item the merge grid covers
  int64_t rows_cap;
  int hpc[kMaxQLen + 1];  // q heads per CTA for R rows
  int tma_slot_dim;       // tcgen05 path: tensor-map coordinate holding the slot (1 or 2)
  uint64_t wait_limit_ns; // tcgen05 path: bound of every pipeline wait
  uint32_t inject;        // PDA_INJECT_* test hooks set by the host (0 in normal use)
};

// The KV range one (request, split) covers. Every kernel derives it from the
// device-resident kv_len / qo_indptr / window, so one plan (and one captured
// graph) serves any lengths up to the plan's maxima.
struct SplitRange {
  int32_t lo;          // first visible key of any row of the request
  int32_t lo_page;     // page holding lo
  int32_t num_pages;   // ceil(L / P)
  int32_t num_splits;  // splits with at least one page of [lo_page, num_pages)
};

PDA_HD SplitRange split_range(int32_t L, int32_t R, int32_t W, int32_t P, int32_t chunk_pages) {
  SplitRange s;
  int32_t p0 = L - R;  // position of the first query row
  s.lo = (W > 0) ? (p0 - W + 1 > 0 ? p0 - W + 1 : 0) : 0;
  s.lo_page = s.lo / P;
  s.num_pages = (L + P - 1) / P;
  int32_t span = s.num_pages - s.lo_page;
  s.num_splits = span > 0 ? (span + chunk_pages - 1) / chunk_pages : 0;
  return s;
}

// KV chunk (pages per split) of request b.
PDA_HD int32_t chunk_for(const DecodeArgs& a, int b) {
  return b >= a.tail_from ? a.tail_chunk_pages : a.chunk_pages;
}

// Stage-1 work item of a CTA: requests [0, tail_from) with head_splits
// splits each come first, then the tail requests with tail_splits; inside
// each part the order is (request, kv head, split, head block), head block
// fastest. False past the last request.
struct WorkItem {
  int b, hkv, split, hb;
};
PDA_HD bool work_item(const DecodeArgs& a, int64_t bid, WorkItem& w) {
  const int64_t head_ctas = (int64_t)a.tail_from * a.hkv * a.head_splits * a.head_blocks;
  int splits = a.head_splits, b0 = 0;
  if (bid >= head_ctas) {
    bid -= head_ctas;
    splits = a.tail_splits;
    b0 = a.tail_from;
  }
  w.hb = static_cast<int>(bid % a.head_blocks);
  bid /= a.head_blocks;
  w.split = static_cast<int>(bid % splits);
  bid /= splits;
  w.hkv = static_cast<int>(bid % a.hkv);
  w.b = b0 + static_cast<int>(bid / a.hkv);
  return w.b < a.batch;
}

// Launchers and resource queries of the two stage-1 variants and stage 2.
int mma_smem_bytes(const pda_plan_t* plan);
int mma_ctas_per_sm(const pda_plan_t* plan);
int launch_stage1_mma(const pda_plan_t* plan, const DecodeArgs& args, cudaStream_t s);
bool tc_supported(const pda_plan_t* plan);
int tc_rows_limit(const pda_plan_t* plan);
int tc_variant_rows(const pda_plan_t* plan);
int tc_smem_bytes(const pda_plan_t* plan);
int tc_ctas_per_sm(const pda_plan_t* plan);
int launch_stage1_tc(const pda_plan_t* plan, const DecodeArgs& args, cudaStream_t s);
int launch_stage2(const pda_plan_t* plan, const DecodeArgs& args, cudaStream_t s);

// Host-side checks of pda_decode's arguments (plan, pointers, alignment,
// max_q_len); PDA_OK or the PDA_ERR_* code pda_decode returns for them.
int check_decode_args(const pda_plan_t* plan, const void* q, const void* k_pages,
                      const void* v_pages, const int32_t* page_table, const int32_t* kv_indptr,
                      const int32_t* kv_len, const int32_t* qo_indptr, int32_t max_q_len,
                      const float* k_scale, const float* v_scale, const void* out,
                      const float* lse);

// Device address of the library's built-in split scratch (the array behind
// pda_decode_static) on the current device, which must be `device`; looked
// up afresh unless `s` is capturing a graph (then the last lookup is used).
int static_scratch(int device, cudaStream_t s, void** out);

}  // namespace pda
