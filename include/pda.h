/*
 * pda.h -- paged split-KV decode attention for GB300 (sm_103a): the C ABI.
 *
 * The operation (per request b with R_b query rows and L_b cached tokens,
 * query row i, query head h, kv head g = h / (Hq / Hkv)):
 *
 *   p_i  = L_b - R_b + i                              row position
 *   V_i  = { j : j <= p_i, and j >= p_i - W_b + 1 if W_b > 0 }
 *   s_j  = sm_scale * (q_i,h . k_j,g)                 j in V_i
 *   out  = sum_j softmax(s)_j * v_j,g                 (bf16)
 *   lse  = ln sum_j exp(s_j)                          (fp32, natural log)
 *
 * with k, v the dequantised cache values (bf16 as stored; E4M3 codes times
 * the per-tensor or per-(token, kv head) scale). Sources, by page and
 * section:
 *  - "perf(attention): run up to 8 query rows per request in the triton
 *    decode kernel" (FreeToken PR #900), "Changes": up to 8 causal query
 *    rows per request (qo_indptr, max_q_len); stage 1 packs query rows x GQA
 *    heads on the M axis and keeps the KV split, each row limited to its own
 *    position and window; stage 2 merges per row; per-row split scratch for
 *    CUDA graphs; a CTA's query heads divide the GQA group.
 *  - same page, "End-to-end A/B": the fp8_per_token_head KV dtype.
 *  - "fp8 support" (FlashMLA PR #54), "Functionality": symmetric per-tensor
 *    FP8 scales.
 *  - "Naive Support for Hopper FP8 Prefill Kernel with Per-Head
 *    Quantization" (FlashInfer PR #869), item 3: QK dequantisation folded
 *    into sm_scale, PV dequantisation folded into the finalize step.
 *  - "[Feature Request] Support q_len > 1 for FP8 decode" (hpc-ops issue
 *    #4): the FP8 decode workload and its byte accounting.
 * Readings taken where the pages are silent: p_i as above (the R new tokens
 * are already in the cache); W counts keys including the row's own, W <= 0
 * means no window; an E4M3 query's scale is folded into sm_scale by the
 * caller; FP8 is OCP E4M3 (e4m3fn).
 *
 * Ownership: every pointer is borrowed. pda_decode allocates nothing, never
 * synchronises, and enqueues work only on `stream`, so it can be captured in
 * a CUDA graph; the same plan and scratch then serve any kv_len, page_table,
 * qo_indptr and window contents within the plan's maxima.
 * Errors: host-side checks return a negative PDA_ERR_* code and launch
 * nothing; the library never aborts and never throws across this ABI.
 * Inputs that only the device can see (a request with kv_len < rows, rows
 * above max_q_len, kv_len above max_kv_len, a page id outside
 * [0, num_pages)) set bits in a status word kept in the scratch header; the
 * affected request's outputs are left unwritten. Kernels never trap.
 */
#ifndef PDA_H_
#define PDA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* pda_stream_t; /* a cudaStream_t; NULL = legacy default stream */

/* Element types. PDA_INT8 (KV cache only): two's-complement codes whose value
 * is the code times the per-tensor or per-(token, kv head) scale; an int8
 * cache is named beside bf16 and fp8 in "perf(attention): run up to 8 query
 * rows per request in the triton decode kernel", Tested on. */
enum { PDA_BF16 = 0, PDA_E4M3 = 1, PDA_INT8 = 2 };
/* PDA_SCALE_MLA_BLOCK: the mixed-precision MLA latent the FlashMLA page's
 * reviewers accept ("fp8 support", FlashMLA PR #54: nope in 8 bits per token
 * and 128 channels, rope in 16 bits). Each (token, kv head) row of the cache
 * is a 640-byte record: 512 E4M3 nope codes, then the 64 bf16 rope channels;
 * strides are in bytes; k_scale = v_scale = fp32 [num_pages, P, Hkv, 4], the
 * scale of each 128-channel nope block. head_dim 576, head_dim_v 512,
 * kv_dtype PDA_E4M3, q_dtype PDA_BF16. */
enum { PDA_SCALE_NONE = 0, PDA_SCALE_TENSOR = 1, PDA_SCALE_TOKEN_HEAD = 2, PDA_SCALE_MLA_BLOCK = 3 };
enum { PDA_KERNEL_AUTO = 0, PDA_KERNEL_MMA = 1, PDA_KERNEL_TC = 2 };

#define PDA_OK 0
#define PDA_ERR_NULL (-1)        /* a required pointer is NULL */
#define PDA_ERR_INVALID (-2)     /* a size or count is out of range */
#define PDA_ERR_UNSUPPORTED (-3) /* head_dim / page_size / dtype combination not built */
#define PDA_ERR_ALIGNMENT (-4)   /* a base address or stride is not 16-byte aligned */
#define PDA_ERR_SCRATCH (-5)     /* split_scratch NULL or not 256-byte aligned */
#define PDA_ERR_CUDA (-6)        /* a CUDA runtime call failed (launch, device query) */
#define PDA_ERR_PLAN (-7)        /* plan not produced by pda_plan, or from another version */
#define PDA_ERR_TOO_LARGE (-8)   /* plan needs more scratch than pda_decode_static's array */

/* Size of the library's own split-scratch array used by pda_decode_static. */
#define PDA_STATIC_SCRATCH_BYTES (32u << 20)

/* Device status bits (sticky in the scratch header until pda_reset_status). */
#define PDA_STATUS_KV_LEN_LT_ROWS 0x1u  /* kv_len[b] < rows of request b */
#define PDA_STATUS_ROWS_GT_MAX 0x2u     /* rows of request b > max_q_len, or negative */
#define PDA_STATUS_KV_LEN_GT_MAX 0x4u   /* kv_len[b] > plan max_kv_len */
#define PDA_STATUS_PAGE_OOB 0x8u        /* a page id read from page_table outside [0, num_pages) */
#define PDA_STATUS_ROWS_GT_CAP 0x10u    /* qo_indptr[batch] > max_batch * max_q_len */
#define PDA_STATUS_WAIT_TIMEOUT 0x20u   /* a pipeline wait ran past its bound; the CTA gave up */
#define PDA_STATUS_SMEM_MISALIGNED 0x40u /* a stage-1 CTA's shared-memory window was not 1024-byte
                                            aligned; that CTA wrote nothing */

/* Everything the planner needs; plain values, no device pointers. */
typedef struct {
  int32_t num_qo_heads;    /* Hq, a multiple of num_kv_heads */
  int32_t num_kv_heads;    /* Hkv >= 1 */
  int32_t head_dim;        /* D: 64, 128, 256 or 512 (512: tcgen05 path, pages >= 8); 576 MLA */
  int32_t page_size;       /* P: power of two in [1, 256] */
  int32_t q_dtype;         /* PDA_BF16, or PDA_E4M3 (then kv_dtype must be PDA_E4M3) */
  int32_t kv_dtype;        /* PDA_BF16, PDA_E4M3 or PDA_INT8 (int8: head_dim <= 256) */
  int32_t scale_mode;      /* PDA_SCALE_NONE for bf16 KV; TENSOR or TOKEN_HEAD for E4M3 / int8;
                              MLA_BLOCK for MLA latent records (E4M3 KV, bf16 Q, 576 / 512) */
  int32_t max_batch;       /* upper bound of `batch` over the plan's lifetime */
  int32_t max_q_len;       /* 1..8: rows per request */
  int32_t max_kv_len;      /* upper bound of kv_len[b] */
  int32_t num_pages;       /* physical pages in k_pages / v_pages */
  int64_t kv_stride_page;  /* cache strides in elements: element (page, slot, kv head, c) */
  int64_t kv_stride_token; /*   lives at page*stride_page + slot*stride_token          */
  int64_t kv_stride_head;  /*   + head*stride_head + c; c is contiguous               */
  int32_t device;          /* CUDA device the plan is for */
  int32_t num_sms;         /* 0: query `device`; > 0: use this SM count (host-only planning) */
  const int32_t* host_kv_len; /* optional host copy of kv_len[batch] for eager planning */
  int32_t batch;           /* requests per call, <= max_batch; 0 = max_batch */
  int32_t chunk_pages;     /* 0: planner chooses the KV chunk per CTA; > 0: forced */
  int32_t kernel;          /* PDA_KERNEL_AUTO, _MMA (mma.sync path) or _TC (tcgen05 path) */
  int32_t head_dim_v;      /* value channels: 0 = head_dim. MLA decode ("fp8 support", FlashMLA
                              PR #54): head_dim 576 (512 latent + 64 rope), head_dim_v 512,
                              one latent cache passed as both k_pages and v_pages, V being its
                              first 512 channels; bf16, or E4M3 with an E4M3 query */
  int32_t wait_limit_us;   /* bound of every stage-1 pipeline wait (tcgen05 path), in
                              microseconds; 0 = 2 s. A wait that runs out sets
                              PDA_STATUS_WAIT_TIMEOUT and its CTA gives up, writing nothing */
  uint32_t inject;         /* test hooks, 0 in normal use: PDA_INJECT_WITHHOLD_KV */
  /* optional host copies for exact eager planning, used with host_kv_len:
   * qo_indptr[batch + 1] (rows of each request) and window[batch]; NULL = every
   * request has max_q_len rows / no window. The plan stays valid for any
   * device contents within its maxima; these only tune its KV chunk. */
  const int32_t* host_qo_indptr;
  const int32_t* host_window;
} pda_params;

/* Test hook (pda_params.inject): the tcgen05 stage-1 CTAs issue no K/V
 * loads at all, so their consumers' waits run out after wait_limit_us and
 * every CTA returns with PDA_STATUS_WAIT_TIMEOUT set and nothing written.
 * It exercises the timeout path without a device fault. */
#define PDA_INJECT_WITHHOLD_KV 0x1u

/* The plan: plain data, owned by the caller, copied freely. Fields are
 * documented for inspection; pda_decode reads only what pda_plan wrote. */
typedef struct {
  uint32_t magic;          /* PDA_PLAN_MAGIC once planned */
  int32_t num_qo_heads, num_kv_heads, head_dim, page_size;
  int32_t q_dtype, kv_dtype, scale_mode;
  int32_t max_batch, max_q_len, max_kv_len, num_pages, batch;
  int64_t kv_stride_page, kv_stride_token, kv_stride_head;
  int32_t group;           /* Hq / Hkv */
  int32_t kernel;          /* resolved PDA_KERNEL_MMA or PDA_KERNEL_TC */
  int32_t rows_per_cta;    /* cap on query rows x heads packed in one CTA */
  int32_t heads_per_cta[9];/* [R]: q heads per CTA for a request with R rows (divides group) */
  int32_t head_blocks;     /* grid extent over head blocks = group / heads_per_cta[max_q_len] */
  int32_t chunk_pages;     /* KV pages per split (CTA) */
  int32_t max_splits;      /* splits per (request, kv head, head block) */
  int32_t num_sms;
  int64_t grid_ctas;       /* stage-1 CTAs per call */
  int64_t rows_cap;        /* max_batch * max_q_len: rows the scratch holds */
  int64_t scratch_bytes;   /* bytes of split_scratch the caller provides */
  int64_t scratch_lse_offset; /* byte offsets inside split_scratch */
  int64_t scratch_o_offset;
  int32_t stage1_smem_bytes;
  /* Requests [tail_from, batch) use chunks of tail_chunk_pages (and up to
   * tail_splits splits) instead of chunk_pages (head_splits): the planner
   * cuts the requests that would run in a last, partial wave of CTAs into
   * shorter chunks, laid out last in the grid. tail_from = batch: none. */
  int32_t tail_from;
  int32_t tail_chunk_pages;
  int32_t head_splits;
  int32_t tail_splits;
  int32_t head_dim_v;      /* value channels (= head_dim but for MLA) */
  int32_t device;          /* pda_params.device */
  int32_t wait_limit_us;   /* pda_params.wait_limit_us, 0 resolved to 2 s */
  uint32_t inject;         /* pda_params.inject */
  int32_t reserved[7];
} pda_plan_t;

#define PDA_PLAN_MAGIC 0x50444131u /* "PDA1" */

/* Plan one decode shape. Host-only (queries the SM count of params->device
 * unless params->num_sms > 0). Writes *out_plan and, when non-NULL,
 * *split_scratch_bytes (>= 256; the caller allocates that many device bytes,
 * 256-byte aligned, zeroes them once, and passes them to every pda_decode of
 * this plan). Returns PDA_OK or a negative PDA_ERR_* code. */
int pda_plan(const pda_params* params, pda_plan_t* out_plan, size_t* split_scratch_bytes);

/* Paged split-KV decode attention (stage 1: per-chunk partial attention of
 * every (request, kv head, head block, KV chunk); stage 2: per-row
 * log-sum-exp merge of the chunks of every (query row, q head)).
 *   q          [qo_indptr[batch], Hq, D] bf16, or E4M3 codes (q_dtype), rows
 *              of request b at [qo_indptr[b], qo_indptr[b+1]); 16-B aligned
 *   k_pages,   paged cache, bf16, E4M3 codes or int8 codes, strides from the plan;
 *   v_pages    16-B aligned; V is the first head_dim_v channels of each v row (MLA:
 *              pass the latent cache as both)
 *   page_table int32 CSR: pages of request b at [kv_indptr[b], kv_indptr[b+1]),
 *              at least ceil(kv_len[b] / P) of them; only those are read
 *   kv_indptr  int32 [batch + 1];  kv_len int32 [batch]
 *   qo_indptr  int32 [batch + 1], non-decreasing, rows per request <= max_q_len
 *   max_q_len  rows-per-request bound of this call, 1..plan max_q_len
 *   window     int32 [batch] sliding window per request (<= 0: none), or NULL
 *   sm_scale   logit scale (times the query's E4M3 scale when q is E4M3)
 *   k_scale,   NULL (bf16), fp32 [1] (per tensor) or fp32 [num_pages, P, Hkv]
 *              (E4M3 / int8)
 *   v_scale    (per token and kv head), device memory
 *   out        [qo_indptr[batch], Hq, head_dim_v] bf16
 *   lse        [qo_indptr[batch], Hq] fp32 natural-log LSE, or NULL
 *   split_scratch  plan->scratch_bytes of device memory (see pda_plan)
 * All device pointers; nothing is allocated or synchronised. */
int pda_decode(const pda_plan_t* plan, const void* q, const void* k_pages, const void* v_pages,
               const int32_t* page_table, const int32_t* kv_indptr, const int32_t* kv_len,
               const int32_t* qo_indptr, int32_t max_q_len, const int32_t* window,
               float sm_scale, const float* k_scale, const float* v_scale, void* out,
               float* lse, void* split_scratch, pda_stream_t stream);

/* pda_decode in two halves, for callers that schedule or time them apart.
 * `stages` is a mask: PDA_STAGE_PARTIAL enqueues stage 1 (the partial
 * attention of every KV chunk; requests whose rows have one chunk get their
 * final out / lse here, the others write partials to split_scratch);
 * PDA_STAGE_MERGE enqueues stage 2 (the per-row merge of those partials; no
 * launch when plan->max_splits is 1). Both bits = pda_decode. The merge
 * must follow stage 1 of the same call on the same stream, with the same
 * arguments. Other bits, or none, return PDA_ERR_INVALID. */
#define PDA_STAGE_PARTIAL 1u
#define PDA_STAGE_MERGE 2u
int pda_decode_stages(const pda_plan_t* plan, const void* q, const void* k_pages,
                      const void* v_pages, const int32_t* page_table, const int32_t* kv_indptr,
                      const int32_t* kv_len, const int32_t* qo_indptr, int32_t max_q_len,
                      const int32_t* window, float sm_scale, const float* k_scale,
                      const float* v_scale, void* out, float* lse, void* split_scratch,
                      uint32_t stages, pda_stream_t stream);

/* Quantise-on-append: write the R_b new tokens of every request into the
 * paged cache, the step before decode reads them ("perf(attention): run up
 * to 8 query rows per request in the triton decode kernel", End-to-end A/B:
 * the fp8_per_token_head cache; "fp8 support", Functionality: symmetric
 * per-tensor FP8). Row i < R_b of request b is token L_b - R_b + i; it lands
 * in page page_table[kv_indptr[b] + t / P], slot t % P, kv head h, with the
 * plan's strides. Per kv dtype and scale mode of the plan:
 *   bf16 cache             the bf16 values, copied;
 *   E4M3, per tensor       codes = RNE(sat(x / s)) with s = k_scale[0] (v_scale[0]), read;
 *   E4M3, per token-head   s = amax / 448 over the D values of (token, kv head)
 *                          (1 if amax = 0), written to k_scale / v_scale
 *                          [num_pages, P, Hkv], and codes = RNE(sat(x / s)).
 *   int8, per tensor       codes = RNE(clamp(x / s, +-127)), s read as for E4M3;
 *   int8, per token-head   s = amax / 127 (1 if amax = 0), written as for E4M3;
 *   MLA records            (PDA_SCALE_MLA_BLOCK, head_dim 576) k_new holds the latents:
 *                          per 128-channel block of the first 512, s = amax / 448 to
 *                          k_scale [num_pages, P, Hkv, 4] and codes = RNE(sat(x / s))
 *                          (a zero block: s = 0 and zero codes, so that it adds nothing
 *                          to any sum of the decode) at record bytes [0, 512); the 64
 *                          rope values copied as bf16 to
 *                          bytes [512, 640); v_new, v_pages and v_scale are not used and
 *                          may be NULL; k_new, k_pages and k_scale 16-byte aligned.
 * x / s is one fp32 division; sat clamps to +-448 (E4M3, OCP e4m3fn); RNE
 * ties go to the even code (int8: the even integer).
 *   k_new, v_new  bf16 [qo_indptr[batch], Hkv, D], rows in qo_indptr order
 *   k_pages, v_pages  the cache (written), layout and strides as planned
 *   page_table, kv_indptr, kv_len, qo_indptr  as for pda_decode (kv_len
 *                 counts the new tokens)
 *   k_scale, v_scale  NULL for bf16; fp32 [1] read (per tensor) or fp32
 *                 [num_pages, P, Hkv] written (per token-head)
 *   split_scratch only its status word is used: page ids outside
 *                 [0, num_pages), kv_len < rows and rows > max_q_len set the
 *                 pda_decode status bits and skip that request
 * Returns PDA_OK or a negative code from the host checks (nothing launched).
 * All device pointers; nothing is allocated or synchronised. */
int pda_append_kv(const pda_plan_t* plan, const void* k_new, const void* v_new,
                  const int32_t* page_table, const int32_t* kv_indptr, const int32_t* kv_len,
                  const int32_t* qo_indptr, int32_t max_q_len, void* k_pages, void* v_pages,
                  float* k_scale, float* v_scale, void* split_scratch, pda_stream_t stream);

/* pda_decode without a caller-provided split_scratch (the pages have no
 * counterpart: this serves callers that cannot allocate device memory, such
 * as a plugin whose host framework owns every allocation and hands it only
 * input and output pointers, or code that must not call cudaMalloc under its
 * host's memory budget). The split scratch lives in a fixed
 * PDA_STATIC_SCRATCH_BYTES array of the library's own device memory, which
 * every GPU that loads the library holds until the process exits. Arguments
 * are those of pda_decode minus split_scratch; the host-side checks are
 * pda_decode's and run before anything is enqueued. Returns
 * PDA_ERR_TOO_LARGE when plan->scratch_bytes exceeds the array, and
 * PDA_ERR_INVALID when the current device is not the plan's device (the
 * array is per device). Allocates nothing. All calls share the array and it
 * keeps the last call's contents; each call first clears the status word (an
 * async memset on `stream`). Calls whose GPU work overlaps race on the
 * array: serialise them (one stream). The array's device address is looked
 * up on every call made outside a stream capture; a call made while `stream`
 * is capturing reuses the last lookup on that device, so make the first call
 * on a device before any stream capture. Read or clear the array's status
 * bits with pda_get_status / pda_reset_status and split_scratch = NULL. */
int pda_decode_static(const pda_plan_t* plan, const void* q, const void* k_pages,
                      const void* v_pages, const int32_t* page_table, const int32_t* kv_indptr,
                      const int32_t* kv_len, const int32_t* qo_indptr, int32_t max_q_len,
                      const int32_t* window, float sm_scale, const float* k_scale,
                      const float* v_scale, void* out, float* lse, pda_stream_t stream);

/* Copy the device status word of `split_scratch` to *host_bits. Synchronises
 * `stream`. split_scratch = NULL reads the status of pda_decode_static's
 * built-in array on the plan's device (which must be current). */
int pda_get_status(const pda_plan_t* plan, const void* split_scratch, uint32_t* host_bits,
                   pda_stream_t stream);

/* Clear the device status word (an async memset on `stream`); NULL clears
 * that of pda_decode_static's built-in array, as for pda_get_status. */
int pda_reset_status(const pda_plan_t* plan, void* split_scratch, pda_stream_t stream);

/* Static text for a PDA_ERR_* code. */
const char* pda_strerror(int code);

/* Library version (major * 10000 + minor * 100 + patch). */
int pda_version(void);

/* sizeof(pda_params) and sizeof(pda_plan_t) as compiled into the library, so
 * that a binding can check its own struct layout. Returns PDA_OK. */
int pda_struct_sizes(size_t* params_bytes, size_t* plan_bytes);

#ifdef __cplusplus
}
#endif

#endif /* PDA_H_ */
