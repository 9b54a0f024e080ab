/*
 * oracle.c -- plain, slow, fp64 CPU oracle for PagedAttention decode and for the
 * per-token KV-cache write (bf16 copy and INT8 symmetric quantisation).
 *
 * TEST INFRASTRUCTURE, NOT PRODUCT CODE.  Only the tests, the smoke check and the
 * benchmark's CPU-baseline / reference legs load this file's library.  It shares no
 * source, header, table or helper with the CUDA library; the two meet only through
 * the seeded inputs that both are handed.
 *
 * What is computed, and where it is defined:
 *  - Attention for one query token over T cached tokens,
 *        out = softmax(q K^T * scale) V,   q in R^{1 x d}, K, V in R^{T x d},
 *    "Lesson 4: Model deployment and inference acceleration" (docs.lazyllm.ai),
 *    section 4.2 "PagedAttention: virtual-memory-style KV management", the
 *    attention-invariance equation.  That section states that PagedAttention leaves
 *    this formula unchanged and only changes where K and V live, so the oracle is the
 *    plain formula: it walks the sequence in logical token order and fetches each
 *    token's K/V row through the page table.
 *  - The page table: each request keeps a table from logical block to physical
 *    block; blocks hold a fixed 16 tokens; all blocks come from one pre-allocated
 *    pool (same section 4.2; "Efficient AI Lecture 13: LLM Deployment Techniques",
 *    section "PagedAttention / How it works", step 4).
 *  - GQA: query heads are split into groups and each group shares one K/V head
 *    ("LLM/MLLM inference optimisation", section 2.3 table, MQA/GQA rows; section 2.2
 *    defines 1 <= n_kv < n_head for GQA).  Groups are contiguous: q head h reads
 *    kv head h / (Hq / Hkv).
 *  - INT8 symmetric KV quantisation, K_q = round(K / s_K), s_K = max|K| / 127
 *    ("Lesson 4", section 5.3 "KV Cache Quantization").  One scale per
 *    (token, kv head) row of d values; fp32 arithmetic with IEEE round-to-nearest
 *    division, round-half-to-even to the integer code, codes clamped to [-127, 127].
 *  - Multi-query decode for speculative verification: the target model checks k draft
 *    tokens in one pass ("Lesson 4", 5.2 "Speculative Decoding", algorithm step 2; "LLM/MLLM
 *    inference optimisation", 6.1).  The drafts are the last k tokens in the cache; query i
 *    (position T - k + i) attends causally, to tokens 0 .. T - k + i.
 *  - Sliding window ("LLM/MLLM inference optimisation", 2.3, KV-cache table: keep only the
 *    most recent window of the cache, for a fixed memory footprint): with a window of W
 *    tokens a query at position p attends to tokens p - W + 1 .. p (those that exist).
 *  - FP8 KV cache (same section names FP8 with its larger dynamic range, and that vLLM
 *    supports an FP8 KV cache; it gives no scaling rule).  Read here as the INT8 scheme
 *    with the E4M3 format in place of int8: s = max|x| / 448 per (token, kv head) row,
 *    code = E4M3(x / s) rounded to nearest, ties to even, saturating at +-448.  E4M3 is
 *    1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits, no infinities; the largest
 *    finite value is 448 and S.1111.111 is NaN.
 *
 * All floating point in the attention path is fp64.  bf16 values are widened exactly
 * (a bf16 is the top 16 bits of an fp32).  INT8 values are dequantised exactly in
 * fp64 as (double)scale * (double)code.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_BLOCK_SIZE 16

enum {
  ORACLE_OK = 0,
  ORACLE_ERR_ARG = -1,        /* a size or pointer argument is invalid            */
  ORACLE_ERR_CONTEXT = -2,    /* a context length is < 1 or exceeds the table     */
  ORACLE_ERR_BLOCK_ID = -3,   /* a block-table entry that is read is out of range */
  ORACLE_ERR_SLOT = -4,       /* a slot_mapping entry is >= num_blocks * 16       */
  ORACLE_ERR_NOMEM = -5
};

enum { ORACLE_KV_BF16 = 0, ORACLE_KV_INT8 = 1, ORACLE_KV_FP8 = 2 };

/* ---------------------------------------------------------------- threads */

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/* ------------------------------------------------------------ conversions */

/* A bf16 value is the upper half of an IEEE-754 binary32; widening is exact. */
float oracle_bf16_to_float(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* ------------------------------------------------------ cache write: bf16 */

/*
 * Write each new token's key and value rows into the slot that slot_mapping names:
 * block = slot / 16, offset = slot % 16, cache[block][head][offset][:] = row.
 * A negative slot means "no write" (a padding token).  Only the new token's K/V are
 * appended ("Lesson 4", section 4.2; "LLM Engineer's Handbook -- inference
 * optimisation", section "KV cache").
 * key, value: [num_tokens, kv_heads, head_dim]; caches: [num_blocks, kv_heads, 16, head_dim].
 */
int oracle_reshape_and_cache_bf16(const uint16_t* key, const uint16_t* value,
                                  const int32_t* slot_mapping, int64_t num_tokens,
                                  int kv_heads, int head_dim, int64_t num_blocks,
                                  uint16_t* k_cache, uint16_t* v_cache) {
  if (num_tokens < 0 || kv_heads < 1 || head_dim < 1 || num_blocks < 1) return ORACLE_ERR_ARG;
  int64_t t;
  for (t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    if (slot >= num_blocks * ORACLE_BLOCK_SIZE) return ORACLE_ERR_SLOT;
  }
  for (t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t block = slot / ORACLE_BLOCK_SIZE;
    int64_t offset = slot % ORACLE_BLOCK_SIZE;
    for (int h = 0; h < kv_heads; ++h) {
      int64_t src = (t * kv_heads + h) * (int64_t)head_dim;
      int64_t dst = ((block * kv_heads + h) * ORACLE_BLOCK_SIZE + offset) * (int64_t)head_dim;
      for (int c = 0; c < head_dim; ++c) {
        k_cache[dst + c] = key[src + c];
        v_cache[dst + c] = value[src + c];
      }
    }
  }
  return ORACLE_OK;
}

/* ------------------------------------------------- INT8 symmetric quantiser */

/*
 * Quantise one row of n fp32 values, following "Lesson 4", section 5.3:
 *   s = max|x| / 127            (fp32 division, IEEE round to nearest even)
 *   code = round(x / s)          (fp32 division, then round half to even)
 * The code is clamped to [-127, 127] so that the range stays symmetric.  A row of
 * zeros has s = 0; no division is done and every code is 0, which dequantises to 0.
 */
void oracle_quantize_row_f32(const float* x, int n, int8_t* codes, float* scale_out) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float s = amax / 127.0f;
  *scale_out = s;
  for (int i = 0; i < n; ++i) {
    if (amax == 0.0f) {
      codes[i] = 0;
      continue;
    }
    float y = x[i] / s;
    float r = rintf(y);
    if (r > 127.0f) r = 127.0f;
    if (r < -127.0f) r = -127.0f;
    codes[i] = (int8_t)r;
  }
}

/* Quantise many rows of bf16 values (each row widened exactly to fp32 first). */
int oracle_quantize_rows_bf16(const uint16_t* x, int64_t rows, int n, int8_t* codes,
                              float* scales) {
  if (rows < 0 || n < 1) return ORACLE_ERR_ARG;
  float* tmp = (float*)malloc(sizeof(float) * (size_t)n);
  if (!tmp) return ORACLE_ERR_NOMEM;
  for (int64_t r = 0; r < rows; ++r) {
    for (int i = 0; i < n; ++i) tmp[i] = oracle_bf16_to_float(x[r * n + i]);
    oracle_quantize_row_f32(tmp, n, codes + r * n, scales + r);
  }
  free(tmp);
  return ORACLE_OK;
}

/*
 * INT8 cache write: the same slot addressing as the bf16 write, but each
 * (token, kv head) row of K and of V is quantised with its own scale, and the scale
 * is stored at [block][head][offset] of the matching scale array.
 */
int oracle_reshape_and_cache_int8(const uint16_t* key, const uint16_t* value,
                                  const int32_t* slot_mapping, int64_t num_tokens,
                                  int kv_heads, int head_dim, int64_t num_blocks,
                                  int8_t* k_cache, int8_t* v_cache, float* k_scale,
                                  float* v_scale) {
  if (num_tokens < 0 || kv_heads < 1 || head_dim < 1 || num_blocks < 1) return ORACLE_ERR_ARG;
  int64_t t;
  for (t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot >= num_blocks * ORACLE_BLOCK_SIZE) return ORACLE_ERR_SLOT;
  }
  float* row = (float*)malloc(sizeof(float) * (size_t)head_dim);
  if (!row) return ORACLE_ERR_NOMEM;
  for (t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t block = slot / ORACLE_BLOCK_SIZE;
    int64_t offset = slot % ORACLE_BLOCK_SIZE;
    for (int h = 0; h < kv_heads; ++h) {
      int64_t src = (t * kv_heads + h) * (int64_t)head_dim;
      int64_t srow = (block * kv_heads + h) * ORACLE_BLOCK_SIZE + offset;
      int64_t dst = srow * (int64_t)head_dim;
      for (int c = 0; c < head_dim; ++c) row[c] = oracle_bf16_to_float(key[src + c]);
      oracle_quantize_row_f32(row, head_dim, k_cache + dst, k_scale + srow);
      for (int c = 0; c < head_dim; ++c) row[c] = oracle_bf16_to_float(value[src + c]);
      oracle_quantize_row_f32(row, head_dim, v_cache + dst, v_scale + srow);
    }
  }
  free(row);
  return ORACLE_OK;
}

/* ---------------------------------------------------------- FP8 (E4M3) */

/* Value of an E4M3 byte: exponent field e (bits 6..3), mantissa m (bits 2..0).
 * e == 0: subnormal m * 2^-9; e == 15 and m == 7: NaN; otherwise (1 + m/8) * 2^(e - 7). */
double oracle_e4m3_to_double(uint8_t b) {
  const int sign = (b >> 7) & 1;
  const int e = (b >> 3) & 15;
  const int m = b & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

/* Nearest E4M3 to a finite y, ties to the even mantissa, saturating at +-448.
 * With |y| = f * 2^k, 1 <= f < 2: the grid spacing is 2^(k-3) for normal numbers
 * (k >= -6) and 2^-9 below; q = round(|y| / spacing) is then an exact scaling by a power
 * of two followed by one rounding, and code = (biased exponent) * 8 + q - 8 also covers a
 * mantissa that rounds up into the next binade. */
uint8_t oracle_float_to_e4m3(float y) {
  const uint8_t sign = (y < 0.0f || (y == 0.0f && signbit(y))) ? 0x80 : 0x00;
  double a = fabs((double)y);
  if (a >= 448.0) return sign | 0x7E;
  if (a == 0.0) return sign;
  int k;
  frexp(a, &k); /* a = f * 2^k with f in [0.5, 1): floor(log2 a) = k - 1 */
  k -= 1;
  int code;
  if (k < -6) {
    const double q = rint(ldexp(a, 9)); /* units of 2^-9 */
    code = (int)q;                       /* q == 8 is the smallest normal, 0x08 */
  } else {
    const double q = rint(ldexp(a, 3 - k)); /* in [8, 16] */
    code = (k + 7) * 8 + (int)q - 8;
  }
  if (code > 0x7E) code = 0x7E;
  return sign | (uint8_t)code;
}

/* Quantise one row to E4M3 with its own fp32 scale s = max|x| / 448 (IEEE division);
 * a zero row gets s = 0 and zero codes. */
void oracle_quantize_row_fp8_f32(const float* x, int n, uint8_t* codes, float* scale_out) {
  float amax = 0.0f;
  for (int i = 0; i < n; ++i) {
    float a = fabsf(x[i]);
    if (a > amax) amax = a;
  }
  float s = amax / 448.0f;
  *scale_out = s;
  for (int i = 0; i < n; ++i) codes[i] = amax == 0.0f ? 0 : oracle_float_to_e4m3(x[i] / s);
}

int oracle_quantize_rows_fp8_bf16(const uint16_t* x, int64_t rows, int n, uint8_t* codes,
                                  float* scales) {
  if (rows < 0 || n < 1) return ORACLE_ERR_ARG;
  float* tmp = (float*)malloc(sizeof(float) * (size_t)n);
  if (!tmp) return ORACLE_ERR_NOMEM;
  for (int64_t r = 0; r < rows; ++r) {
    for (int i = 0; i < n; ++i) tmp[i] = oracle_bf16_to_float(x[r * n + i]);
    oracle_quantize_row_fp8_f32(tmp, n, codes + r * n, scales + r);
  }
  free(tmp);
  return ORACLE_OK;
}

/* FP8 cache write: the INT8 write's addressing with the E4M3 quantiser. */
int oracle_reshape_and_cache_fp8(const uint16_t* key, const uint16_t* value,
                                 const int32_t* slot_mapping, int64_t num_tokens, int kv_heads,
                                 int head_dim, int64_t num_blocks, uint8_t* k_cache,
                                 uint8_t* v_cache, float* k_scale, float* v_scale) {
  if (num_tokens < 0 || kv_heads < 1 || head_dim < 1 || num_blocks < 1) return ORACLE_ERR_ARG;
  int64_t t;
  for (t = 0; t < num_tokens; ++t)
    if ((int64_t)slot_mapping[t] >= num_blocks * ORACLE_BLOCK_SIZE) return ORACLE_ERR_SLOT;
  float* row = (float*)malloc(sizeof(float) * (size_t)head_dim);
  if (!row) return ORACLE_ERR_NOMEM;
  for (t = 0; t < num_tokens; ++t) {
    int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    int64_t block = slot / ORACLE_BLOCK_SIZE;
    int64_t offset = slot % ORACLE_BLOCK_SIZE;
    for (int h = 0; h < kv_heads; ++h) {
      int64_t src = (t * kv_heads + h) * (int64_t)head_dim;
      int64_t srow = (block * kv_heads + h) * ORACLE_BLOCK_SIZE + offset;
      int64_t dst = srow * (int64_t)head_dim;
      for (int c = 0; c < head_dim; ++c) row[c] = oracle_bf16_to_float(key[src + c]);
      oracle_quantize_row_fp8_f32(row, head_dim, k_cache + dst, k_scale + srow);
      for (int c = 0; c < head_dim; ++c) row[c] = oracle_bf16_to_float(value[src + c]);
      oracle_quantize_row_fp8_f32(row, head_dim, v_cache + dst, v_scale + srow);
    }
  }
  free(row);
  return ORACLE_OK;
}

/* ------------------------------------------------------------ decode */

/* Value of element c of the cached row (block, head, offset) as fp64. */
static double cache_value(const void* cache, const float* scales, int kv_dtype,
                          int64_t row, int head_dim, int c) {
  if (kv_dtype == ORACLE_KV_BF16) {
    const uint16_t* p = (const uint16_t*)cache;
    return (double)oracle_bf16_to_float(p[row * head_dim + c]);
  }
  if (kv_dtype == ORACLE_KV_FP8) {
    const uint8_t* p = (const uint8_t*)cache;
    return (double)scales[row] * oracle_e4m3_to_double(p[row * head_dim + c]);
  }
  const int8_t* p = (const int8_t*)cache;
  return (double)scales[row] * (double)p[row * head_dim + c];
}

/*
 * out[b][h][:] = sum_t softmax_t(scale * q[b][h] . k_t) v_t  over the T_b tokens of
 * sequence b, in logical order t = 0 .. T_b - 1.  Token t lives in logical block
 * j = t / 16 at offset i = t % 16; its physical block is block_tables[b][j]; its key
 * row is k_cache[phys][kvh][i][:] with kvh = h / (Hq / Hkv).  INT8 and FP8 rows are
 * dequantised as (double)scale * value(code).
 * The softmax is evaluated in two passes (find the largest logit, then exponentiate
 * the differences); this is the same value as exp(l_t) / sum exp(l_u).
 *
 * q: bf16 bits [B, Hq, d]; block_tables: [B, max_blocks_per_seq]; context_lens: [B];
 * out: fp64 [B, Hq, d].  Entries of block_tables past the last used block are never read.
 */
int oracle_paged_decode_window(const uint16_t* q, const void* k_cache, const void* v_cache,
                               const float* k_scale, const float* v_scale, int kv_dtype,
                               int64_t num_blocks, int kv_heads, int head_dim,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int num_seqs, int num_queries,
                               int window, int num_q_heads, double scale, double* out) {
  if (num_seqs < 0 || kv_heads < 1 || head_dim < 1 || num_blocks < 1 || max_blocks_per_seq < 1 ||
      num_queries < 1 || window < 0)
    return ORACLE_ERR_ARG;
  if (num_q_heads < kv_heads || num_q_heads % kv_heads != 0) return ORACLE_ERR_ARG;
  if (kv_dtype != ORACLE_KV_BF16 && kv_dtype != ORACLE_KV_INT8 && kv_dtype != ORACLE_KV_FP8)
    return ORACLE_ERR_ARG;
  if (kv_dtype != ORACLE_KV_BF16 && (!k_scale || !v_scale)) return ORACLE_ERR_ARG;

  /* Validate everything that will be read before any arithmetic: the table entries of the
   * blocks that hold a token some query sees (with a window, earlier entries are never
   * read and may hold anything). */
  for (int b = 0; b < num_seqs; ++b) {
    int T = context_lens[b];
    if (T < num_queries || (int64_t)T > (int64_t)max_blocks_per_seq * ORACLE_BLOCK_SIZE)
      return ORACLE_ERR_CONTEXT;
    int first = 0;  /* the first query's first visible token */
    if (window > 0 && T - (num_queries - 1) - window > 0) first = T - (num_queries - 1) - window;
    int nblk = (T + ORACLE_BLOCK_SIZE - 1) / ORACLE_BLOCK_SIZE;
    for (int j = first / ORACLE_BLOCK_SIZE; j < nblk; ++j) {
      int32_t phys = block_tables[(int64_t)b * max_blocks_per_seq + j];
      if (phys < 0 || (int64_t)phys >= num_blocks) return ORACLE_ERR_BLOCK_ID;
    }
  }

  const int group = num_q_heads / kv_heads;
  const int64_t pairs = (int64_t)num_seqs * num_queries * num_q_heads;  /* (b, query, head) */
  int err = ORACLE_OK;

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t bh = 0; bh < pairs; ++bh) {
    const int b = (int)(bh / ((int64_t)num_queries * num_q_heads));
    const int qi = (int)((bh / num_q_heads) % num_queries);
    const int h = (int)(bh % num_q_heads);
    const int kvh = h / group;
    /* query qi sits at position T - num_queries + qi and sees tokens up to and including it,
     * and with a window only the last `window` of those */
    const int T = context_lens[b] - (num_queries - 1 - qi);
    const int lo = (window > 0 && T > window) ? T - window : 0;
    const uint16_t* qrow = q + bh * head_dim;
    double* orow = out + bh * head_dim;

    double* logits = (double*)malloc(sizeof(double) * (size_t)(T - lo));
    double* qd = (double*)malloc(sizeof(double) * (size_t)head_dim);
    if (!logits || !qd) {
      free(logits);
      free(qd);
#pragma omp atomic write
      err = ORACLE_ERR_NOMEM;
      continue;
    }
    for (int c = 0; c < head_dim; ++c) qd[c] = (double)oracle_bf16_to_float(qrow[c]);

    /* Pass 1: the logits, walking the page table in logical order. */
    double lmax = -INFINITY;
    for (int t = lo; t < T; ++t) {
      int j = t / ORACLE_BLOCK_SIZE;
      int i = t % ORACLE_BLOCK_SIZE;
      int64_t phys = block_tables[(int64_t)b * max_blocks_per_seq + j];
      int64_t row = (phys * kv_heads + kvh) * ORACLE_BLOCK_SIZE + i;
      double dot = 0.0;
      for (int c = 0; c < head_dim; ++c)
        dot += qd[c] * cache_value(k_cache, k_scale, kv_dtype, row, head_dim, c);
      logits[t - lo] = scale * dot;
      if (logits[t - lo] > lmax) lmax = logits[t - lo];
    }

    /* Pass 2: softmax weights and the weighted sum of the value rows. */
    double denom = 0.0;
    for (int t = lo; t < T; ++t) {
      logits[t - lo] = exp(logits[t - lo] - lmax);
      denom += logits[t - lo];
    }
    for (int c = 0; c < head_dim; ++c) orow[c] = 0.0;
    for (int t = lo; t < T; ++t) {
      int j = t / ORACLE_BLOCK_SIZE;
      int i = t % ORACLE_BLOCK_SIZE;
      int64_t phys = block_tables[(int64_t)b * max_blocks_per_seq + j];
      int64_t row = (phys * kv_heads + kvh) * ORACLE_BLOCK_SIZE + i;
      double w = logits[t - lo] / denom;
      for (int c = 0; c < head_dim; ++c)
        orow[c] += w * cache_value(v_cache, v_scale, kv_dtype, row, head_dim, c);
    }
    free(logits);
    free(qd);
  }
  return err;
}

/* Every query over its whole causal prefix: the windowed decode with no window. */
int oracle_paged_decode_multi(const uint16_t* q, const void* k_cache, const void* v_cache,
                              const float* k_scale, const float* v_scale, int kv_dtype,
                              int64_t num_blocks, int kv_heads, int head_dim,
                              const int32_t* block_tables, int max_blocks_per_seq,
                              const int32_t* context_lens, int num_seqs, int num_queries,
                              int num_q_heads, double scale, double* out) {
  return oracle_paged_decode_window(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, num_blocks,
                                    kv_heads, head_dim, block_tables, max_blocks_per_seq,
                                    context_lens, num_seqs, num_queries, 0, num_q_heads, scale, out);
}

/* One query token per sequence (the newest): the multi-query decode with k = 1. */
int oracle_paged_decode(const uint16_t* q, const void* k_cache, const void* v_cache,
                        const float* k_scale, const float* v_scale, int kv_dtype,
                        int64_t num_blocks, int kv_heads, int head_dim,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* context_lens, int num_seqs, int num_q_heads,
                        double scale, double* out) {
  return oracle_paged_decode_multi(q, k_cache, v_cache, k_scale, v_scale, kv_dtype, num_blocks,
                                   kv_heads, head_dim, block_tables, max_blocks_per_seq,
                                   context_lens, num_seqs, 1, num_q_heads, scale, out);
}
