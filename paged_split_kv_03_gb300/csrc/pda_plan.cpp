// pda_plan.cpp -- host side of the C ABI: the split planner, argument
// validation, status access and error strings.
//
// The planner keeps the KV split of "perf(attention): run up to 8 query rows
// per request in the triton decode kernel" (FreeToken PR #900, "Changes") and
// sizes it for this GPU: it picks how many KV pages one CTA streams
// (chunk_pages) from the batch, the context and the SM count, and it picks
// how many query heads one CTA packs next to the request's rows so that the
// heads always divide the GQA group (the same section's fix for groups such
// as 48 query / 2 kv heads).
#include <cuda_runtime.h>

#include <algorithm>
#include <cstring>
#include <queue>
#include <vector>

#include "pda_internal.h"

namespace {

bool is_pow2(int v) { return v > 0 && (v & (v - 1)) == 0; }

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

int elem_bytes(int dtype) { return dtype == PDA_BF16 ? 2 : 1; }

}  // namespace

extern "C" int pda_version(void) { return 100; }

extern "C" int pda_struct_sizes(size_t* params_bytes, size_t* plan_bytes) {
  if (params_bytes) *params_bytes = sizeof(pda_params);
  if (plan_bytes) *plan_bytes = sizeof(pda_plan_t);
  return PDA_OK;
}

extern "C" const char* pda_strerror(int code) {
  switch (code) {
    case PDA_OK: return "ok";
    case PDA_ERR_NULL: return "a required pointer is NULL";
    case PDA_ERR_INVALID: return "a size or count is out of range";
    case PDA_ERR_UNSUPPORTED: return "head_dim / page_size / dtype combination not supported";
    case PDA_ERR_ALIGNMENT: return "a base address or stride is not 16-byte aligned";
    case PDA_ERR_SCRATCH: return "split_scratch is NULL or not 256-byte aligned";
    case PDA_ERR_CUDA: return "a CUDA runtime call failed";
    case PDA_ERR_PLAN: return "plan was not produced by pda_plan of this library version";
    case PDA_ERR_TOO_LARGE:
      return "plan needs more split scratch than pda_decode_static's built-in array holds";
    default: return "unknown pda error code";
  }
}

extern "C" int pda_plan(const pda_params* p, pda_plan_t* out, size_t* split_scratch_bytes) {
  if (!p || !out) return PDA_ERR_NULL;
  pda_plan_t pl;
  std::memset(&pl, 0, sizeof pl);
  // ---- shape checks
  if (p->num_qo_heads <= 0 || p->num_kv_heads <= 0 || p->num_qo_heads % p->num_kv_heads)
    return PDA_ERR_INVALID;
  // MLA: a 576-channel latent (512 + 64 rope) whose first 512 channels are V
  const int dv = p->head_dim_v ? p->head_dim_v : p->head_dim;
  const bool mla = p->head_dim == 576 && dv == 512;
  if (p->head_dim_v < 0 || (dv != p->head_dim && !mla)) return PDA_ERR_UNSUPPORTED;
  if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256 && p->head_dim != 512 && !mla)
    return PDA_ERR_UNSUPPORTED;
  // the latent's E4M3 path takes an E4M3 query (FlashMLA's per-tensor Q/K/V);
  // the mixed-precision records take a bf16 query, and only they take block scales
  const bool mla_block = p->scale_mode == PDA_SCALE_MLA_BLOCK;
  if (mla_block && (!mla || p->kv_dtype != PDA_E4M3 || p->q_dtype != PDA_BF16))
    return PDA_ERR_UNSUPPORTED;
  if (mla && !mla_block &&
      (p->kv_dtype == PDA_INT8 || (p->kv_dtype == PDA_E4M3 && p->q_dtype != PDA_E4M3)))
    return PDA_ERR_UNSUPPORTED;
  if (!is_pow2(p->page_size) || p->page_size > 256) return PDA_ERR_UNSUPPORTED;
  if (p->kv_dtype != PDA_BF16 && p->kv_dtype != PDA_E4M3 && p->kv_dtype != PDA_INT8)
    return PDA_ERR_UNSUPPORTED;
  if (p->q_dtype != PDA_BF16 && p->q_dtype != PDA_E4M3) return PDA_ERR_UNSUPPORTED;
  if (p->q_dtype == PDA_E4M3 && p->kv_dtype != PDA_E4M3) return PDA_ERR_UNSUPPORTED;
  if (p->kv_dtype == PDA_BF16 && p->scale_mode != PDA_SCALE_NONE) return PDA_ERR_UNSUPPORTED;
  if (p->kv_dtype != PDA_BF16 && p->scale_mode != PDA_SCALE_TENSOR &&
      p->scale_mode != PDA_SCALE_TOKEN_HEAD && p->scale_mode != PDA_SCALE_MLA_BLOCK)
    return PDA_ERR_UNSUPPORTED;
  if (p->max_batch <= 0 || p->max_q_len < 1 || p->max_q_len > pda::kMaxQLen) return PDA_ERR_INVALID;
  if (p->max_kv_len < 1 || p->num_pages < 1) return PDA_ERR_INVALID;
  if (p->batch < 0 || p->batch > p->max_batch) return PDA_ERR_INVALID;
  if (p->kv_stride_page <= 0 || p->kv_stride_token <= 0 || p->kv_stride_head <= 0)
    return PDA_ERR_INVALID;
  if (p->chunk_pages < 0) return PDA_ERR_INVALID;
  if (p->kernel < PDA_KERNEL_AUTO || p->kernel > PDA_KERNEL_TC) return PDA_ERR_INVALID;
  if (p->wait_limit_us < 0 || (p->inject & ~PDA_INJECT_WITHHOLD_KV)) return PDA_ERR_INVALID;
  // 16-byte alignment of every stride ("require 16-byte aligned cache bases
  // and strides", follow-up commit on the FreeToken page)
  const int eb = elem_bytes(p->kv_dtype);
  if ((p->kv_stride_page * eb) % 16 || (p->kv_stride_token * eb) % 16 ||
      (p->kv_stride_head * eb) % 16)
    return PDA_ERR_ALIGNMENT;

  int num_sms = p->num_sms;
  if (num_sms <= 0) {
    if (cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, p->device) !=
        cudaSuccess) {
      cudaGetLastError();
      return PDA_ERR_CUDA;
    }
  }

  pl.magic = PDA_PLAN_MAGIC;
  pl.num_qo_heads = p->num_qo_heads;
  pl.num_kv_heads = p->num_kv_heads;
  pl.head_dim = p->head_dim;
  pl.head_dim_v = dv;
  pl.page_size = p->page_size;
  pl.q_dtype = p->q_dtype;
  pl.kv_dtype = p->kv_dtype;
  pl.scale_mode = p->scale_mode;
  pl.max_batch = p->max_batch;
  pl.max_q_len = p->max_q_len;
  pl.max_kv_len = p->max_kv_len;
  pl.num_pages = p->num_pages;
  pl.batch = p->batch ? p->batch : p->max_batch;
  pl.kv_stride_page = p->kv_stride_page;
  pl.kv_stride_token = p->kv_stride_token;
  pl.kv_stride_head = p->kv_stride_head;
  pl.group = p->num_qo_heads / p->num_kv_heads;
  pl.num_sms = num_sms;
  pl.device = p->device;
  pl.wait_limit_us = p->wait_limit_us > 0 ? p->wait_limit_us : 2000000;
  pl.inject = p->inject;
  if (p->kernel == PDA_KERNEL_TC && !pda::tc_supported(&pl)) return PDA_ERR_UNSUPPORTED;
  // AUTO takes the tcgen05 path wherever it is built (head_dim 128/256/512/576,
  // pages >= 8); head_dims above 256 have no mma.sync build (their O tile
  // would not fit the registers)
  if (p->kernel == PDA_KERNEL_AUTO)
    pl.kernel = pda::tc_supported(&pl) ? PDA_KERNEL_TC : PDA_KERNEL_MMA;
  else
    pl.kernel = p->kernel;
  if (pl.kernel == PDA_KERNEL_MMA && p->head_dim > 256) return PDA_ERR_UNSUPPORTED;
  pl.rows_per_cta = pl.kernel == PDA_KERNEL_TC ? pda::tc_rows_limit(&pl) : pda::kMmaRowsPerCta;

  // Query heads per CTA for a request with R rows: the largest divisor of the
  // GQA group whose R x heads tile fits the CTA's rows.
  for (int R = 1; R <= pda::kMaxQLen; ++R) {
    int best = 1;
    for (int d = 1; d <= pl.group; ++d)
      if (pl.group % d == 0 && R * d <= pl.rows_per_cta) best = d;
    pl.heads_per_cta[R] = best;
  }
  pl.heads_per_cta[0] = pl.heads_per_cta[1];
  pl.head_blocks = pl.group / pl.heads_per_cta[pl.max_q_len];

  if (pl.kernel == PDA_KERNEL_TC) pl.rows_per_cta = pda::tc_variant_rows(&pl);

  // Context to plan for: the maximum, or the exact host lengths when given.
  int64_t max_len = p->max_kv_len;
  if (p->host_kv_len) {
    int64_t m = 1;
    for (int b = 0; b < pl.batch; ++b) m = std::max<int64_t>(m, p->host_kv_len[b]);
    max_len = std::min<int64_t>(m, p->max_kv_len);
    pl.max_kv_len = (int32_t)max_len;
  }
  const int64_t pages_max = ceil_div(max_len, p->page_size);

  // Split planning: pick the KV chunk (pages per CTA) that minimises a small
  // cost model of stage 1 + stage 2 on this GPU. A CTA costs a fixed
  // overhead (prologue, pipeline fill, epilogue) plus its K/V bytes at its
  // slot's streaming rate; CTAs run in waves of `slots`; more than one
  // split adds the merge (stage 2 launch plus partials written and read).
  // With host lengths, per-request work replaces the uniform worst case.
  const bool tc = pl.kernel == PDA_KERNEL_TC;
  pl.stage1_smem_bytes = tc ? pda::tc_smem_bytes(&pl) : pda::mma_smem_bytes(&pl);
  const int per_sm = std::max(1, tc ? pda::tc_ctas_per_sm(&pl) : pda::mma_ctas_per_sm(&pl));
  const int64_t slots = (int64_t)num_sms * per_sm;
  const int64_t hb_units = (int64_t)pl.num_kv_heads * pl.head_blocks;  // CTAs per (request, split)
  const int64_t units = (int64_t)pl.batch * hb_units;
  const double page_kv_bytes = 2.0 * p->page_size * p->head_dim * eb;  // K+V of one head, one page
  // A CTA works in tiles of 128 tokens: the bytes it costs are those of its
  // pages rounded up to whole tiles (a chunk of 560 tokens costs five tiles,
  // one of 512 four: measured 4 % apart at bs 1)
  auto chunk_cost_bytes = [&](int64_t pages) {
    const int64_t tiles = ceil_div(pages * p->page_size, 128);
    return static_cast<double>(tiles) * 128.0 * (page_kv_bytes / p->page_size);
  };
  const double hbm_bytes_per_us = 44000.0 * num_sms;  // ~6.7 TB/s over 152 SMs
  const double sm_bytes_per_us = 44000.0 / per_sm;     // a slot's share
  // What the CTA of a one-per-SM build can consume when HBM is not the
  // limit (bytes/us, measured on GB300 with fewer CTAs than SMs): head_dim
  // 256 bf16 ~56 KB/us at 16-64 columns; E4M3 ~46 KB/us at 32 columns and
  // ~40 at 64 (two-term S and P); int8 ~24 (the widening pass). Elsewhere
  // (two CTAs per SM, whose siblings share an SM's loads unevenly when
  // fewer than all slots are busy; head_dim 512; MLA) a slot is taken to
  // stream at its share of HBM whatever the number of busy slots.
  double slot_cap = sm_bytes_per_us;
  bool capped = false;
  if (tc && per_sm == 1 && pl.head_dim <= 256 && pl.scale_mode != PDA_SCALE_MLA_BLOCK) {
    const int ncols = ((pl.max_q_len * pl.heads_per_cta[pl.max_q_len] + 15) / 16) * 16;
    capped = true;
    if (pl.kv_dtype == PDA_INT8) slot_cap = 24000.0;
    else if (pl.kv_dtype == PDA_E4M3) slot_cap = 40000.0 + 200.0 * (64 - std::min(ncols, 64));
    else slot_cap = 56000.0;
  }
  // a slot's rate while `active` slots stream at once
  auto slot_rate = [&](int64_t active) {
    if (!capped) return sm_bytes_per_us;
    const int64_t a = std::max<int64_t>(1, std::min(active, slots));
    return std::min(slot_cap, hbm_bytes_per_us / a);
  };
  // The second CTA of an SM streams through its sibling's prologue and
  // epilogue; with one CTA per SM nothing does, and each CTA's start-up
  // (launch, request scalars, page ids, the first tile's round trip) and
  // drain (the last tiles' MMAs, softmax and output) leave its SM idle.
  const double cta_overhead_us = per_sm >= 2 ? 4.0 : 8.0;
  const double merge_us = 3.0;
  const double rows_heads = (double)pl.batch * pl.max_q_len * pl.num_qo_heads;
  // Exact eager planning (host copies of the lengths, rows and windows):
  // each request's visible pages and its own head blocks, the grid's CTAs
  // in launch order (request, kv head, split, head block) taken greedily by
  // `slots` SM slots (a CTA with no work costs a launch), and the merge of
  // the requests that split.
  struct HostReq {
    int64_t pages;
    int nhb, rows;
  };
  std::vector<HostReq> hreq;
  if (p->host_kv_len) {
    hreq.resize(pl.batch);
    for (int b = 0; b < pl.batch; ++b) {
      const int64_t L = std::max<int64_t>(0, std::min<int64_t>(p->host_kv_len[b], max_len));
      int R = p->host_qo_indptr ? p->host_qo_indptr[b + 1] - p->host_qo_indptr[b] : pl.max_q_len;
      R = std::max(0, std::min(R, pl.max_q_len));
      const int W = p->host_window ? p->host_window[b] : 0;
      const int64_t lo = W > 0 ? std::max<int64_t>(0, L - R - W + 1) : 0;
      hreq[b].pages = R > 0 && L > 0 ? ceil_div(L, p->page_size) - lo / p->page_size : 0;
      hreq[b].nhb = R > 0 ? pl.group / pl.heads_per_cta[R] : 0;
      hreq[b].rows = R;
    }
  }
  const int64_t exact_ctas = (int64_t)pl.batch * hb_units;  // times the split count
  auto exact_cost = [&](int64_t chunk) -> double {
    const int64_t nsplit = ceil_div(pages_max, chunk);
    std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
    for (int64_t i = 0; i < slots; ++i) free_at.push(0.0);
    double end = 0.0, merge_bytes = 0.0;
    for (int b = 0; b < pl.batch; ++b) {
      const HostReq& h = hreq[b];
      const int64_t ns = h.pages > 0 ? ceil_div(h.pages, chunk) : 0;
      if (ns > 1) merge_bytes += 2.0 * ns * h.rows * pl.num_qo_heads * (p->head_dim + 1) * 4;
      for (int kvh = 0; kvh < pl.num_kv_heads; ++kvh)
        for (int64_t sp = 0; sp < nsplit; ++sp)
          for (int hb = 0; hb < pl.head_blocks; ++hb) {
            double w = 0.5;  // a CTA without work: launch and exit
            if (sp < ns && hb < h.nhb)
              w = cta_overhead_us +
                  chunk_cost_bytes(std::min<int64_t>(chunk, h.pages - sp * chunk)) / slot_rate(slots);
            const double s0 = free_at.top();
            free_at.pop();
            free_at.push(s0 + w);
            end = std::max(end, s0 + w);
          }
    }
    if (nsplit > 1) end += merge_us + merge_bytes / 6.0e6;
    return end;
  };
  auto cost = [&](int64_t chunk) -> double {
    const int64_t nsplit = ceil_div(pages_max, chunk);
    if (!hreq.empty() && exact_ctas * nsplit <= 400000) return exact_cost(chunk);
    double t;
    if (p->host_kv_len) {
      double total = 0.0, longest = 0.0;
      for (int b = 0; b < pl.batch; ++b) {
        const int64_t pages = std::max<int64_t>(1, ceil_div(p->host_kv_len[b], p->page_size));
        for (int64_t s0 = 0; s0 < pages; s0 += chunk) {
          const double w =
              cta_overhead_us + chunk_cost_bytes(std::min<int64_t>(chunk, pages - s0)) / slot_rate(slots);
          total += w * hb_units;
          longest = std::max(longest, w);
        }
      }
      t = std::max(total / slots, longest);
    } else {
      // full waves at the all-slots rate, then a partial one at its own
      const int64_t n = units * nsplit;
      const double bytes = chunk_cost_bytes(chunk);
      t = (double)(n / slots) * (cta_overhead_us + bytes / slot_rate(slots));
      if (n % slots) t += cta_overhead_us + bytes / slot_rate(n % slots);
    }
    if (nsplit > 1) t += merge_us + 2.0 * nsplit * rows_heads * (p->head_dim + 1) * 4 / 6.0e6;
    return t;
  };
  int64_t chunk;
  if (p->chunk_pages > 0) {
    chunk = p->chunk_pages;
  } else {
    chunk = std::max<int64_t>(pages_max, 1);
    double best = cost(chunk);
    const int64_t max_split = std::min<int64_t>(pages_max, 8 * slots);
    for (int64_t n = 2; n <= max_split; ++n) {
      const int64_t c = ceil_div(pages_max, n);
      if (ceil_div(pages_max, c) != n) continue;  // same chunk as a smaller n
      // the exact model simulates the grid: try split counts 2..16, then
      // about 12 % apart
      if (!hreq.empty() && n > 16 && n % std::max<int64_t>(1, n / 8) != 0) continue;
      const double t = cost(c);
      if (t < best * 0.999) {
        best = t;
        chunk = c;
      }
    }
  }
  chunk = std::min<int64_t>(std::max<int64_t>(chunk, 1), std::max<int64_t>(pages_max, 1));
  pl.chunk_pages = (int32_t)chunk;
  pl.head_splits = (int32_t)ceil_div(pages_max, chunk);
  pl.tail_from = pl.batch;
  pl.tail_chunk_pages = pl.chunk_pages;
  pl.tail_splits = pl.head_splits;

  // Tail split: CTAs of equal length run in waves of `slots`, so a last,
  // partial wave leaves SMs idle. When the planner chose the chunk, the
  // requests whose CTAs would form that wave get chunks k times shorter
  // (k ~ slots / their CTAs) and run last, if a greedy schedule of the CTAs
  // (each SM slot takes the next CTA when free) finishes sooner, merge
  // included.
  if (p->chunk_pages == 0 && pl.batch > 0 && hreq.empty()) {
    const int64_t per_req = hb_units * pl.head_splits;  // CTAs of one request
    const int64_t total = (int64_t)pl.batch * per_req;
    const int64_t rem = total % slots;
    auto cta_us = [&](int64_t c) {
      return cta_overhead_us + chunk_cost_bytes(std::min<int64_t>(c, pages_max)) / slot_rate(slots);
    };
    // makespan of n1 CTAs of t1 then n2 of t2 when each of `slots` slots
    // takes the next CTA as soon as it is free
    auto makespan = [&](int64_t n1, double t1, int64_t n2, double t2) {
      std::priority_queue<double, std::vector<double>, std::greater<double>> free_at;
      for (int64_t i = 0; i < slots; ++i) free_at.push(0.0);
      double end = 0.0;
      auto run = [&](int64_t n, double t) {
        for (int64_t i = 0; i < n; ++i) {
          const double s0 = free_at.top();
          free_at.pop();
          free_at.push(s0 + t);
          end = std::max(end, s0 + t);
        }
      };
      run(n1, t1);
      run(n2, t2);
      return end;
    };
    if (total > slots && rem > 0 && total <= 64 * slots) {
      const int64_t nt = std::min<int64_t>(ceil_div(rem, per_req), pl.batch);
      const int64_t k = slots / (nt * per_req);
      if (k >= 2) {
        const int64_t tchunk = std::max<int64_t>(1, ceil_div(chunk, k));
        const int64_t tsplits = ceil_div(pages_max, tchunk);
        const int64_t head = (int64_t)(pl.batch - nt) * per_req;
        const int64_t tail = nt * hb_units * tsplits;
        const double merge_rows = (double)nt * pl.max_q_len * pl.num_qo_heads;
        double t_with = makespan(head, cta_us(chunk), tail, cta_us(tchunk)) +
                        2.0 * tsplits * merge_rows * (p->head_dim + 1) * 4 / 6.0e6;
        if (pl.head_splits == 1) t_with += merge_us;  // stage 2 was not needed before
        const double t_without = makespan(total, cta_us(chunk), 0, 0.0);
        if (t_with < 0.97 * t_without) {
          pl.tail_from = (int32_t)(pl.batch - nt);
          pl.tail_chunk_pages = (int32_t)tchunk;
          pl.tail_splits = (int32_t)tsplits;
        }
      }
    }
  }
  pl.max_splits = std::max(pl.head_splits, pl.tail_splits);
  pl.grid_ctas = (int64_t)pl.tail_from * hb_units * pl.head_splits +
                 (int64_t)(pl.batch - pl.tail_from) * hb_units * pl.tail_splits;
  if (pl.grid_ctas > 0x7fffffffLL) return PDA_ERR_INVALID;

  pl.rows_cap = (int64_t)pl.max_batch * pl.max_q_len;
  int64_t off = pda::kStatusHeaderBytes;
  pl.scratch_lse_offset = off;
  if (pl.max_splits > 1) {
    off += ceil_div((int64_t)pl.max_splits * pl.rows_cap * pl.num_qo_heads * 4, 256) * 256;
    pl.scratch_o_offset = off;
    off += (int64_t)pl.max_splits * pl.rows_cap * pl.num_qo_heads * pl.head_dim_v * 4;
  } else {
    pl.scratch_o_offset = off;
  }
  pl.scratch_bytes = off;
  *out = pl;
  if (split_scratch_bytes) *split_scratch_bytes = (size_t)pl.scratch_bytes;
  return PDA_OK;
}

namespace pda {

int check_decode_args(const pda_plan_t* plan, const void* q, const void* k_pages,
                      const void* v_pages, const int32_t* page_table, const int32_t* kv_indptr,
                      const int32_t* kv_len, const int32_t* qo_indptr, int32_t max_q_len,
                      const float* k_scale, const float* v_scale, const void* out,
                      const float* lse) {
  if (!plan) return PDA_ERR_NULL;
  if (plan->magic != PDA_PLAN_MAGIC) return PDA_ERR_PLAN;
  if (!q || !k_pages || !v_pages || !page_table || !kv_indptr || !kv_len || !qo_indptr || !out)
    return PDA_ERR_NULL;
  if (max_q_len < 1 || max_q_len > plan->max_q_len) return PDA_ERR_INVALID;
  if (plan->scale_mode != PDA_SCALE_NONE && (!k_scale || !v_scale)) return PDA_ERR_NULL;
  auto a16 = [](const void* p) { return reinterpret_cast<uintptr_t>(p) % 16 == 0; };
  if (!a16(q) || !a16(k_pages) || !a16(v_pages) || !a16(out)) return PDA_ERR_ALIGNMENT;
  if (lse && reinterpret_cast<uintptr_t>(lse) % 4) return PDA_ERR_ALIGNMENT;
  if (plan->scale_mode != PDA_SCALE_NONE &&
      (reinterpret_cast<uintptr_t>(k_scale) % 4 || reinterpret_cast<uintptr_t>(v_scale) % 4))
    return PDA_ERR_ALIGNMENT;
  // MLA records: a token's four block scales are read as one 16-byte vector
  if (plan->scale_mode == PDA_SCALE_MLA_BLOCK && reinterpret_cast<uintptr_t>(k_scale) % 16)
    return PDA_ERR_ALIGNMENT;
  return PDA_OK;
}

}  // namespace pda

extern "C" int pda_decode_stages(const pda_plan_t* plan, const void* q, const void* k_pages,
                                 const void* v_pages, const int32_t* page_table,
                                 const int32_t* kv_indptr, const int32_t* kv_len,
                                 const int32_t* qo_indptr, int32_t max_q_len,
                                 const int32_t* window, float sm_scale, const float* k_scale,
                                 const float* v_scale, void* out, float* lse,
                                 void* split_scratch, uint32_t stages, pda_stream_t stream) {
  if (!plan) return PDA_ERR_NULL;
  if (stages == 0 || (stages & ~(PDA_STAGE_PARTIAL | PDA_STAGE_MERGE))) return PDA_ERR_INVALID;
  if (plan->magic != PDA_PLAN_MAGIC) return PDA_ERR_PLAN;
  if (!q || !k_pages || !v_pages || !page_table || !kv_indptr || !kv_len || !qo_indptr || !out)
    return PDA_ERR_NULL;
  if (!split_scratch) return PDA_ERR_SCRATCH;
  if (reinterpret_cast<uintptr_t>(split_scratch) % 256) return PDA_ERR_SCRATCH;
  const int rc0 = pda::check_decode_args(plan, q, k_pages, v_pages, page_table, kv_indptr, kv_len,
                                         qo_indptr, max_q_len, k_scale, v_scale, out, lse);
  if (rc0 != PDA_OK) return rc0;
  if (plan->batch == 0) return PDA_OK;

  pda::DecodeArgs a;
  std::memset(&a, 0, sizeof a);
  a.q = q;
  a.k = k_pages;
  a.v = v_pages;
  a.page_table = page_table;
  a.kv_indptr = kv_indptr;
  a.kv_len = kv_len;
  a.qo_indptr = qo_indptr;
  a.window = window;
  a.k_scale = plan->scale_mode != PDA_SCALE_NONE ? k_scale : nullptr;
  a.v_scale = plan->scale_mode != PDA_SCALE_NONE ? v_scale : nullptr;
  a.out = out;
  a.lse = lse;
  char* base = static_cast<char*>(split_scratch);
  a.status = reinterpret_cast<uint32_t*>(base);
  a.part_lse = reinterpret_cast<float*>(base + plan->scratch_lse_offset);
  a.part_o = reinterpret_cast<float*>(base + plan->scratch_o_offset);
  a.sm_scale = sm_scale;
  a.sp = plan->kv_stride_page;
  a.st = plan->kv_stride_token;
  a.sh = plan->kv_stride_head;
  a.batch = plan->batch;
  a.hq = plan->num_qo_heads;
  a.hkv = plan->num_kv_heads;
  a.group = plan->group;
  a.head_dim = plan->head_dim;
  a.head_dim_v = plan->head_dim_v;
  a.page_size = plan->page_size;
  a.num_pages = plan->num_pages;
  a.max_q_len = max_q_len;
  a.max_kv_len = plan->max_kv_len;
  a.max_splits = plan->max_splits;
  a.head_blocks = plan->head_blocks;
  a.chunk_pages = plan->chunk_pages;
  a.tail_from = plan->tail_from;
  a.tail_chunk_pages = plan->tail_chunk_pages;
  a.head_splits = plan->head_splits;
  a.tail_splits = plan->tail_splits;
  a.rows_cap = plan->rows_cap;
  a.wait_limit_ns = static_cast<uint64_t>(plan->wait_limit_us > 0 ? plan->wait_limit_us : 2000000) *
                    1000ull;
  a.inject = plan->inject;
  for (int r = 0; r <= pda::kMaxQLen; ++r) a.hpc[r] = plan->heads_per_cta[r];
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int rc = PDA_OK;
  if (stages & PDA_STAGE_PARTIAL)
    rc = plan->kernel == PDA_KERNEL_TC ? pda::launch_stage1_tc(plan, a, s)
                                       : pda::launch_stage1_mma(plan, a, s);
  if (rc == PDA_OK && (stages & PDA_STAGE_MERGE) && plan->max_splits > 1)
    rc = pda::launch_stage2(plan, a, s);
  return rc;
}

extern "C" int pda_decode(const pda_plan_t* plan, const void* q, const void* k_pages,
                          const void* v_pages, const int32_t* page_table,
                          const int32_t* kv_indptr, const int32_t* kv_len,
                          const int32_t* qo_indptr, int32_t max_q_len, const int32_t* window,
                          float sm_scale, const float* k_scale, const float* v_scale, void* out,
                          float* lse, void* split_scratch, pda_stream_t stream) {
  return pda_decode_stages(plan, q, k_pages, v_pages, page_table, kv_indptr, kv_len, qo_indptr,
                           max_q_len, window, sm_scale, k_scale, v_scale, out, lse,
                           split_scratch, PDA_STAGE_PARTIAL | PDA_STAGE_MERGE, stream);
}

extern "C" int pda_get_status(const pda_plan_t* plan, const void* split_scratch,
                              uint32_t* host_bits, pda_stream_t stream) {
  if (!plan || !host_bits) return PDA_ERR_NULL;
  if (plan->magic != PDA_PLAN_MAGIC) return PDA_ERR_PLAN;
  void* fixed = nullptr;
  if (!split_scratch) {  // the built-in array of pda_decode_static
    const int rc =
        pda::static_scratch(plan->device, reinterpret_cast<cudaStream_t>(stream), &fixed);
    if (rc != PDA_OK) return rc;
    split_scratch = fixed;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_bits, split_scratch, sizeof(uint32_t), cudaMemcpyDeviceToHost, s) !=
          cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess) {
    cudaGetLastError();
    return PDA_ERR_CUDA;
  }
  return PDA_OK;
}

extern "C" int pda_reset_status(const pda_plan_t* plan, void* split_scratch, pda_stream_t stream) {
  if (!plan) return PDA_ERR_NULL;
  if (plan->magic != PDA_PLAN_MAGIC) return PDA_ERR_PLAN;
  if (!split_scratch) {  // the built-in array of pda_decode_static
    const int rc = pda::static_scratch(plan->device, reinterpret_cast<cudaStream_t>(stream),
                                       &split_scratch);
    if (rc != PDA_OK) return rc;
  }
  if (cudaMemsetAsync(split_scratch, 0, sizeof(uint32_t),
                      reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return PDA_ERR_CUDA;
  }
  return PDA_OK;
}
