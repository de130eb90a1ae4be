/*
 * pdo_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, fp64 CPU statement of what paged split-KV decode attention
 * computes. Only the test suite, the smoke check and the benchmark's CPU
 * baseline load this file's library; the CUDA library never links it, and it
 * includes nothing from the CUDA library (its own types, its own decoders).
 *
 * What it follows:
 *  - "perf(attention): run up to 8 query rows per request in the triton
 *    decode kernel" (FreeToken PR #900), section "Changes": each request has
 *    up to 8 causal query rows (qo_indptr, max_q_len); every row sees keys up
 *    to its own position and inside its window; the KV split is merged per
 *    row. Query head h reads kv head h / (Hq/Hkv) (contiguous GQA groups).
 *  - "fp8 support" (FlashMLA PR #54), section "Functionality": symmetric
 *    per-tensor FP8 scales.
 *  - FreeToken PR #900, section "End-to-end A/B": the fp8_per_token_head KV
 *    dtype, i.e. one fp32 scale per (token, kv head).
 *  - "Naive Support for Hopper FP8 Prefill Kernel with Per-Head Quantization"
 *    (FlashInfer PR #869), item 3 "Fused Dequantization": the dequant scales
 *    are plain multipliers on the QK logits and on the PV output, so the
 *    oracle applies them to the decoded K and V values directly.
 *
 * Readings of the pages taken here (the pages leave these open):
 *  - Row i of a request with R rows and L cached tokens sits at position
 *    p_i = L - R + i (the R new tokens are already in the cache).
 *  - A window W > 0 counts keys including the row's own: p_i-W+1 <= j <= p_i.
 *    W <= 0, or no window array, means no lower bound.
 *  - lse is the natural log of sum_j exp(s_j) over the scaled logits.
 *  - FP8 is OCP E4M3 ("e4m3fn": bias 7, no infinities, S.1111.111 is NaN).
 *  - MLA decode ("fp8 support", FlashMLA PR #54): the keys are the latent
 *    vectors of d channels (512 nope + 64 rope, the page's kv_rope) and the
 *    values are their first dv = 512 channels; a caller passes the latent
 *    cache as both k and v, and the oracle reads V channels c < dv.
 *  - The mixed-precision latent the FlashMLA page's reviewers accept (the
 *    nope channels in 8 bits with a scale per token and 128 channels, the
 *    64 rope channels in 16 bits): scale_mode 3. Reading: one record per
 *    (token, kv head) of 512 E4M3 codes then 64 bf16 values (640 bytes),
 *    strides in bytes, scales fp32 [num_pages, page_size, hkv, 4]; channel
 *    c < 512 is code(c) * scale[c / 128], channel 512 + r the bf16 r.
 *  - An int8 cache (named beside bf16 and fp8 in the register-spill check of
 *    FreeToken PR #900, "Tested on") holds two's-complement bytes; the value
 *    is the byte times the same per-tensor or per-(token, kv head) scale.
 *
 * Split mode (split_tokens > 0) cuts the key axis into chunks
 * [c*T, (c+1)*T), computes (o_c, lse_c) per chunk with the same two-pass
 * softmax and merges them: M = max lse_c, w_c = exp(lse_c - M),
 * o = sum w_c o_c / sum w_c, lse = M + ln sum w_c; a chunk with no visible
 * key has lse_c = -inf and weight 0 (the per-row merge of "Changes").
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Mutation hooks. The normal build defines PDO_MUTATION as 0, so every MUT(k)
 * below is the constant 0 and changes nothing. The test suite compiles extra
 * copies with one PDO_MUTATION = k each: every such copy carries one
 * plausible mistake, and the suite checks that the oracle's pins reject it. */
#ifndef PDO_MUTATION
#define PDO_MUTATION 0
#endif
#define MUT(k) (PDO_MUTATION == (k))

#define PDO_OK 0
#define PDO_ERR_ARG (-1)
#define PDO_ERR_KVLEN (-2) /* a request has kv_len < rows: its outputs are NaN */
#define PDO_ERR_PAGE (-3)  /* append: a page id outside [0, num_pages) */

/* bf16 is the upper half of an IEEE binary32 word. */
static double pdo_bf16_to_double(uint16_t bits) {
  uint32_t w = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

/* OCP 8-bit floating point, E4M3: sign bit 7, exponent bits 6..3 with bias 7,
 * mantissa bits 2..0. Exponent field 0 is subnormal (2^-6 * m/8). The pattern
 * with exponent 15 and mantissa 7 is NaN; there is no infinity. */
double pdo_e4m3_to_double(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 0xF;
  int m = code & 0x7;
  double mag;
  if (e == 0xF && m == 0x7) return NAN;
  if (e == 0)
    mag = ldexp((double)m / 8.0, -6 - MUT(7));
  else
    mag = ldexp(1.0 + (double)m / 8.0, e - 7 - MUT(6));
  return sign ? -mag : mag;
}

/* Two's-complement signed byte (int8 cache element). */
static double pdo_int8_to_double(uint8_t byte) {
  int v = MUT(20) ? (int)byte : (byte >= 128 ? (int)byte - 256 : (int)byte);
  return (double)v;
}

#define PDO_KV_BF16 0
#define PDO_KV_E4M3 1
#define PDO_KV_INT8 2

typedef struct {
  int batch, hq, hkv, d, page_size;
  int dv;                           /* value channels (<= d): o has dv entries */
  int q_e4m3, kv_dtype, scale_mode; /* kv_dtype: PDO_KV_*; scale_mode: 0 none, 1 per tensor,
                                       2 per (token, kv head) */
  int64_t sp, st, sh;              /* cache strides in elements: page, token-in-page, kv head */
  int64_t num_pages;
  const void *q, *k, *v;
  const int32_t *page_table, *kv_indptr, *kv_len, *qo_indptr, *window;
  double sm_scale;
  const float *k_scale, *v_scale;
} pdo_problem;

static double pdo_q_elem(const pdo_problem* p, int64_t row, int h, int d) {
  int64_t idx = ((row - MUT(14) * (row > 0)) * p->hq + h) * (int64_t)p->d + d;
  if (p->q_e4m3) return pdo_e4m3_to_double(((const uint8_t*)p->q)[idx]);
  return pdo_bf16_to_double(((const uint16_t*)p->q)[idx]);
}

/* Dequantised K or V element of kv head g at token j of request b. */
static double pdo_kv_elem(const pdo_problem* p, const void* cache, const float* scale, int b,
                          int64_t j, int g, int d) {
  int64_t page = p->page_table[p->kv_indptr[b] + j / p->page_size + MUT(13)];
  int64_t slot = j % p->page_size;
  int64_t idx = MUT(10) ? page * p->sp + slot * p->sh + (int64_t)g * p->st + d
                        : page * p->sp + slot * p->st + (int64_t)g * p->sh + d;
  double x;
  if (p->scale_mode == 3) { /* MLA record: E4M3 nope with 128-channel scales, bf16 rope */
    const uint8_t* rec = (const uint8_t*)cache + (page * p->sp + slot * p->st + (int64_t)g * p->sh);
    if (d < 512) {
      int blk = MUT(25) ? d / 64 % 4 : d / 128;
      return pdo_e4m3_to_double(rec[d]) *
             (double)scale[((page * p->page_size + slot) * p->hkv + g) * 4 + blk];
    }
    uint16_t bits;
    memcpy(&bits, rec + 512 + 2 * (d - 512) - MUT(26) * (d - 512), 2);
    return pdo_bf16_to_double(bits);
  }
  if (p->kv_dtype == PDO_KV_E4M3)
    x = pdo_e4m3_to_double(((const uint8_t*)cache)[idx]);
  else if (p->kv_dtype == PDO_KV_INT8)
    x = pdo_int8_to_double(((const uint8_t*)cache)[idx]);
  else
    x = pdo_bf16_to_double(((const uint16_t*)cache)[idx]);
  if (p->scale_mode == 1) x *= (double)scale[0];
  if (p->scale_mode == 2) x *= (double)scale[(page * p->page_size + slot) * p->hkv + (MUT(4) ? 0 : g)];
  return x;
}

/* Two-pass softmax attention of one query row over keys [lo, hi] (inclusive)
 * of request b, kv head g. Writes o[0..d) and returns lse; an empty range
 * gives o = 0 and lse = -inf. */
static double pdo_attend_range(const pdo_problem* p, int b, int64_t row, int h, int g,
                               int64_t lo, int64_t hi, double* s, double* o) {
  int64_t n = hi - lo + 1;
  for (int d = 0; d < p->dv; ++d) o[d] = 0.0;
  if (n <= 0) return -INFINITY;
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    double acc = 0.0;
    for (int d = 0; d < p->d; ++d) acc += pdo_q_elem(p, row, h, d) * pdo_kv_elem(p, p->k, p->k_scale, b, lo + j, g, d);
    s[j] = MUT(12) ? acc : p->sm_scale * acc;
    if (s[j] > m) m = s[j];
  }
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    double w = exp(s[j] - m);
    l += w;
    for (int d = 0; d < p->dv; ++d)
      o[d] += w * pdo_kv_elem(p, p->v, MUT(9) ? p->k_scale : p->v_scale, b, lo + j, g,
                              d + MUT(24) * (p->d - p->dv));
  }
  if (!MUT(15))
    for (int d = 0; d < p->dv; ++d) o[d] /= l;
  return MUT(5) ? log(l) : m + log(l);
}

/* One (query row, q head) item; returns PDO_OK or PDO_ERR_KVLEN. */
static int pdo_item(const pdo_problem* p, int64_t row, int h, int64_t split_tokens, double* s,
                    double* oc, double* out, double* lse_out) {
  int b = 0;
  while (b < p->batch && p->qo_indptr[b + 1] <= row) ++b; /* request owning this row */
  int64_t rows_b = p->qo_indptr[b + 1] - p->qo_indptr[b];
  int64_t i = row - p->qo_indptr[b];
  int64_t L = p->kv_len[b];
  if (L < rows_b) {
    for (int d = 0; d < p->dv; ++d) out[d] = NAN;
    *lse_out = NAN;
    return PDO_ERR_KVLEN;
  }
  int64_t pos = L - rows_b + i - MUT(11);
  int64_t w = p->window ? p->window[b] : 0;
  int64_t lo = (w > 0) ? pos - w + 1 - MUT(1) : 0;
  if (lo < 0) lo = 0;
  if (MUT(2)) pos = L - 1;
  int g = MUT(3) ? h % p->hkv : h / (p->hq / p->hkv);
  if (split_tokens <= 0) {
    *lse_out = pdo_attend_range(p, b, row, h, g, lo, pos, s, out);
    return PDO_OK;
  }
  /* Split mode: per-chunk partials, then the log-sum-exp merge. */
  int64_t nchunks = pos / split_tokens + 1;
  double* lse_c = (double*)malloc(sizeof(double) * (size_t)nchunks);
  double* o_c = (double*)malloc(sizeof(double) * (size_t)nchunks * (size_t)p->dv);
  double big = -INFINITY;
  for (int64_t c = 0; c < nchunks; ++c) {
    int64_t a = c * split_tokens, e = a + split_tokens - 1;
    if (a < lo) a = lo;
    if (e > pos) e = pos;
    lse_c[c] = pdo_attend_range(p, b, row, h, g, a, e, s, oc);
    memcpy(o_c + c * p->dv, oc, sizeof(double) * (size_t)p->dv);
    if (lse_c[c] > big) big = lse_c[c];
  }
  double wsum = 0.0;
  for (int d = 0; d < p->dv; ++d) out[d] = 0.0;
  for (int64_t c = 0; c < nchunks; ++c) {
    if (lse_c[c] == -INFINITY) continue; /* weight 0 */
    double wc = exp(lse_c[c] - big);
    wsum += wc;
    for (int d = 0; d < p->dv; ++d) out[d] += wc * o_c[c * p->dv + d];
  }
  if (!MUT(8))
    for (int d = 0; d < p->dv; ++d) out[d] /= wsum;
  *lse_out = big + log(wsum);
  free(lse_c);
  free(o_c);
  return PDO_OK;
}

/*
 * Attention output for the requested (query row, q head) items.
 *   q        [total_rows, hq, d]   bf16 bits (uint16) or e4m3 codes (uint8)
 *   k, v     paged cache, element (page, slot, kv head, c) at
 *            page*sp + slot*st + head*sh + c; bf16 bits, e4m3 codes or int8
 *            bytes (kv_dtype 0 / 1 / 2)
 *   k_scale, v_scale: NULL (scale_mode 0), [1] (1) or
 *            [num_pages, page_size, hkv] (2)
 *   dv       value channels, 1..d: V is channels [0, dv) of each v row
 *   items    NULL: all total_rows*hq items in order; else flat indices
 *            row*hq + h, n_items of them
 *   out      [n_items, dv] fp64; lse [n_items] fp64 (natural log)
 * Returns PDO_OK, PDO_ERR_ARG, or PDO_ERR_KVLEN (some rows set to NaN).
 */
int pdo_attention(int batch, int hq, int hkv, int d, int dv, int page_size, int q_e4m3, int kv_dtype,
                  int scale_mode, int64_t sp, int64_t st, int64_t sh, int64_t num_pages,
                  const void* q, const void* k, const void* v, const int32_t* page_table,
                  const int32_t* kv_indptr, const int32_t* kv_len, const int32_t* qo_indptr,
                  const int32_t* window, double sm_scale, const float* k_scale,
                  const float* v_scale, int64_t split_tokens, const int64_t* items,
                  int64_t n_items, double* out, double* lse, int num_threads) {
  if (batch < 0 || hq <= 0 || hkv <= 0 || hq % hkv || d <= 0 || page_size <= 0) return PDO_ERR_ARG;
  if (dv <= 0 || dv > d) return PDO_ERR_ARG;
  if (kv_dtype < PDO_KV_BF16 || kv_dtype > PDO_KV_INT8) return PDO_ERR_ARG;
  if (scale_mode < 0 || scale_mode > 3 || ((scale_mode != 0) != (kv_dtype != PDO_KV_BF16)))
    return PDO_ERR_ARG;
  if (scale_mode == 3 && (kv_dtype != PDO_KV_E4M3 || d != 576 || dv != 512 || q_e4m3))
    return PDO_ERR_ARG;
  if (q_e4m3 && kv_dtype != PDO_KV_E4M3) return PDO_ERR_ARG;
  pdo_problem p = {batch, hq, hkv, d, page_size, dv, q_e4m3, kv_dtype, scale_mode, sp, st, sh, num_pages,
                   q, k, v, page_table, kv_indptr, kv_len, qo_indptr, window, sm_scale,
                   k_scale, v_scale};
  int64_t total_rows = batch > 0 ? qo_indptr[batch] : 0;
  int64_t n = items ? n_items : total_rows * hq;
  int64_t max_len = 0;
  for (int b = 0; b < batch; ++b)
    if (kv_len[b] > max_len) max_len = kv_len[b];
  int status = PDO_OK;
#ifdef _OPENMP
  if (num_threads > 0) omp_set_num_threads(num_threads);
#else
  (void)num_threads;
#endif
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * (size_t)(max_len + 1));
    double* oc = (double*)malloc(sizeof(double) * (size_t)dv);
#pragma omp for schedule(dynamic, 1)
    for (int64_t t = 0; t < n; ++t) {
      int64_t flat = items ? items[t] : t;
      int rc = pdo_item(&p, flat / hq, (int)(flat % hq), split_tokens, s, oc, out + t * dv, lse + t);
      if (rc != PDO_OK) {
#pragma omp atomic write
        status = rc;
      }
    }
    free(s);
    free(oc);
  }
  return status;
}

/* ------------------------------------------------------------------------
 * Quantise-on-append (the step before decode reads the cache): FreeToken PR
 * #900, "End-to-end A/B" (the fp8_per_token_head cache: one fp32 scale per
 * token and kv head) and FlashMLA PR #54, "Functionality" (symmetric
 * per-tensor FP8). The code decision is taken in fp32, the precision the
 * kernel takes it in (the pages fix none): s = fp32(amax / 448) (1 if amax
 * is 0), y = fp32(x / s), code = the E4M3 value nearest to y, ties to the
 * even code, |y| above 448 saturating to 448.
 * ------------------------------------------------------------------------ */

/* Nearest E4M3 code to y (OCP e4m3fn), ties to the even code, saturating to
 * +-448; NaN -> 0x7F. By exhaustive comparison with every finite code. */
uint8_t pdo_e4m3_encode(float y) {
  if (isnan(y)) return 0x7F;
  uint8_t sign = (signbit(y) && !MUT(19)) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a > 448.0) return (uint8_t)(sign | 0x7E);
  uint8_t best = 0;
  double best_d = INFINITY;
  for (int c = 0; c <= 0x7E; ++c) {
    double dist = fabs(pdo_e4m3_to_double((uint8_t)c) - a);
    /* strictly nearer wins; on a tie the even code wins */
    if (dist < best_d || (dist == best_d && (c & 1) == MUT(17))) {
      best = (uint8_t)c;
      best_d = dist;
    }
  }
  return (uint8_t)(sign | best);
}

/* Nearest integer to y, ties to the even integer, clamped to [-127, 127]
 * (symmetric int8; -128 is never produced); NaN -> 0. By comparing the two
 * integers that bracket y. */
uint8_t pdo_int8_encode(float y) {
  if (isnan(y)) return 0;
  double a = (double)y;
  double lo = floor(a), hi = ceil(a);
  double r;
  if (a - lo < hi - a)
    r = lo;
  else if (hi - a < a - lo)
    r = hi;
  else /* a tie (or y already an integer: lo == hi) */
    r = MUT(22) ? (a < 0 ? lo : hi) : (fmod(lo, 2.0) == 0.0 ? lo : hi);
  if (!MUT(23)) {
    if (r > 127.0) r = 127.0;
    if (r < -127.0) r = -127.0;
  }
  int v = (int)r;
  return (uint8_t)(v & 0xFF);
}

/*
 * pdo_append: writes row i < R_b of every request b (token t = L_b - R_b + i)
 * into page page_table[kv_indptr[b] + t / P], slot t % P, kv head h.
 *   mode 0: bf16 cache, the bf16 bits copied
 *   mode 1: E4M3 cache, s = k_scale[0] / v_scale[0] (read)
 *   mode 2: E4M3 cache, s per (token, kv head) from the row's amax, written
 *           to k_scale / v_scale [num_pages, page_size, hkv]
 *   mode 3: int8 cache, s = k_scale[0] / v_scale[0] (read)
 *   mode 4: int8 cache, s = fp32(amax / 127) per (token, kv head) (1 if amax
 *           is 0), written like mode 2; code = pdo_int8_encode(fp32(x / s))
 *   mode 5: MLA records (d = 576): per 128-channel block of the first 512
 *           channels s = fp32(amax / 448) (1 if 0), written to k_scale
 *           [num_pages, page_size, hkv, 4], codes as mode 2 at record bytes
 *           [0, 512); the 64 rope channels copied as bf16 to bytes [512, 640);
 *           v_new and v are not used (the latent is both K and V)
 *   k_new, v_new  bf16 bits [total_rows, hkv, d]
 *   k, v          caches (bytes; bf16 cache: 2 bytes per element), strides in elements
 * Returns PDO_OK, PDO_ERR_ARG, PDO_ERR_KVLEN (a request with L < R, skipped)
 * or PDO_ERR_PAGE (a page id outside [0, num_pages), that row skipped).
 */
int pdo_append(int batch, int hkv, int d, int page_size, int mode, int64_t sp, int64_t st,
               int64_t sh, int64_t num_pages, const uint16_t* k_new, const uint16_t* v_new,
               const int32_t* page_table, const int32_t* kv_indptr, const int32_t* kv_len,
               const int32_t* qo_indptr, uint8_t* k, uint8_t* v, float* k_scale,
               float* v_scale) {
  if (batch < 0 || hkv <= 0 || d <= 0 || page_size <= 0 || mode < 0 || mode > 5) return PDO_ERR_ARG;
  if (mode == 5 && d != 576) return PDO_ERR_ARG;
  if (mode != 0 && (!k_scale || (mode != 5 && !v_scale))) return PDO_ERR_ARG;
  int status = PDO_OK;
  for (int b = 0; b < batch; ++b) {
    int R = qo_indptr[b + 1] - qo_indptr[b];
    int L = kv_len[b];
    if (R <= 0) continue;
    if (L < R) {
      status = PDO_ERR_KVLEN;
      continue;
    }
    for (int i = 0; i < R; ++i) {
      int64_t t = (int64_t)L - R + i - MUT(18);
      int32_t page = page_table[kv_indptr[b] + t / page_size];
      int64_t slot = t % page_size;
      if (page < 0 || page >= num_pages) {
        status = PDO_ERR_PAGE;
        continue;
      }
      for (int h = 0; h < hkv; ++h) {
        int64_t row = ((int64_t)(qo_indptr[b] + i) * hkv + h) * d;
        int64_t base = (int64_t)page * sp + slot * st + (int64_t)h * sh;
        int64_t sidx = ((int64_t)page * page_size + slot) * hkv + h;
        if (mode == 5) {
          const uint16_t* src = k_new + row;
          for (int blk = 0; blk < 4; ++blk) {
            float amax = 0.0f;
            for (int c = 128 * blk; c < 128 * blk + (MUT(27) ? 64 : 128); ++c) {
              float x = (float)pdo_bf16_to_double(src[c]);
              if (fabsf(x) > amax) amax = fabsf(x);
            }
            /* a zero block: scale 0 and zero codes (its decoded values are
               zero, and a scale of 0 gives it no weight in any sum) */
            float sc = amax > 0.0f ? amax / 448.0f : (MUT(28) ? 1.0f : 0.0f);
            k_scale[sidx * 4 + blk] = sc;
            for (int c = 128 * blk; c < 128 * (blk + 1); ++c) {
              float y = (float)pdo_bf16_to_double(src[c]) / (amax > 0.0f ? sc : 1.0f);
              k[base + c] = pdo_e4m3_encode(y);
            }
          }
          for (int c = 0; c < 64; ++c) memcpy(k + base + 512 + 2 * c, src + 512 + c, 2);
          continue;
        }
        for (int kv = 0; kv < 2; ++kv) {
          const uint16_t* src = (kv ? v_new : k_new) + row;
          uint8_t* cache = kv ? v : k;
          float* scale = kv ? v_scale : k_scale;
          if (mode == 0) {
            for (int c = 0; c < d; ++c) memcpy(cache + (base + c) * 2, src + c, 2);
            continue;
          }
          float amax = 0.0f;
          for (int c = 0; c < d; ++c) {
            float x = (float)pdo_bf16_to_double(src[c]);
            if (fabsf(x) > amax) amax = fabsf(x);
          }
          const int int8 = mode >= 3;
          float s;
          if (mode == 1 || mode == 3) {
            s = scale[0];
          } else if (!int8) {
            s = amax > 0.0f ? amax / (MUT(16) ? 256.0f : 448.0f) : 1.0f;
            scale[sidx] = s;
          } else {
            s = amax > 0.0f ? amax / (MUT(21) ? 128.0f : 127.0f) : 1.0f;
            scale[sidx] = s;
          }
          for (int c = 0; c < d; ++c) {
            float y = (float)pdo_bf16_to_double(src[c]) / s;
            cache[base + c] = int8 ? pdo_int8_encode(y) : pdo_e4m3_encode(y);
          }
        }
      }
    }
  }
  return status;
}

/* Threads the OpenMP runtime would use for a parallel region. */
int pdo_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
