/*
 * pkv_oracle.c -- plain, slow, fp64 CPU restatement of what the paged KV-cache decode path
 * computes.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the bench's CPU
 * baseline load it; the library's own path never does.  It shares no code, header, table
 * or constant with the CUDA library: every operation is written here straight from its
 * definition, in the order the definition states it, with no blocking, fusion or
 * reordering.  bf16 values are widened exactly to double; sums and exponentials are fp64.
 * The one exception is INT8 quantization, whose integer codes are decided in fp32 (see
 * quantize_row); dequantized values are exact in fp64.
 *
 * Page names used in the citations below:
 *   [primer]  KV-cache primer article, cf-1.com/news/5988169 (sections numbered as on the page)
 *   [novita]  "How KV Sparsity Achieves 1.5x Acceleration for vLLM", blogs.novita.ai
 *   [naive]   naive KV cache post, koas-w.github.io/posts/20260325-kvcache
 *   [tfcache] "Transformer模型中的KV Cache优化推理策略", yutianautomatic.com
 *
 * Return codes: 0 = ok, negative = the input breaks the stated contract (the oracle
 * refuses to guess).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_BLOCK 16 /* tokens per block: [primer] section 4.1 and section 5.2 (--block-size 16) */

#define ORC_OK 0
#define ORC_ERR_ARG (-1)
#define ORC_ERR_SLOT (-2)
#define ORC_ERR_BLOCK (-3)
#define ORC_ERR_INDEX (-4)
#define ORC_ERR_LEN (-5)
#define ORC_ERR_NAN (-6)
#define ORC_ERR_MEM (-7)
#define ORC_ERR_VALUE (-8)

/* bfloat16 is the upper half of an IEEE binary32: widening is exact. */
static double bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static float bf16_to_float(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/*
 * A K or V pool as the decode reads it: bf16 elements, or INT8 codes (bytes code + 128) with one
 * fp32 scale per (block, kv head, token) row, whose values are code * scale (exact in fp64).
 * Row r = (physical block * Hkv + kv head) * 16 + offset; element e of row r is at r * d + e.
 */
typedef struct {
  const uint16_t* bf16;
  const uint8_t* codes;
  const float* scales;
} pool_t;

static double pool_value(const pool_t* p, int64_t row, int head_dim, int e) {
  if (p->bf16) return bf16_to_double(p->bf16[row * head_dim + e]);
  return (double)((int)p->codes[row * head_dim + e] - 128) * (double)p->scales[row];
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads of the parallel loops from now on (n >= 1); a no-op without OpenMP. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

/*
 * KV-cache size in bytes: 2 (K and V) x batch x layers x heads x head_dim x seq_len x
 * bytes per element.  [primer] section 3.1 (size formula).
 */
int64_t oracle_kv_cache_bytes(int64_t batch, int64_t layers, int64_t heads, int64_t head_dim,
                              int64_t seq_len, int64_t dtype_bytes) {
  return 2 * batch * layers * heads * head_dim * seq_len * dtype_bytes;
}

/*
 * Append: each new token's K and V rows are stored at its slot, for every kv head.
 * A slot is physical block * 16 + offset inside the block ([primer] section 4.1: blocks of
 * 16 tokens mapped through a block table); the decode step stores only the new token's K,V
 * ([primer] section 2.2).  Slot < 0 skips the token.
 * Pools are [NB][Hkv][16][d] uint16 (bf16 bits); k, v are [T][Hkv][d].
 */
int oracle_kv_append(uint16_t* k_cache, uint16_t* v_cache, const uint16_t* k, const uint16_t* v,
                     const int64_t* slot_mapping, int64_t num_tokens, int num_kv_heads,
                     int head_dim, int64_t num_blocks) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0) return ORC_ERR_ARG;
  for (int64_t i = 0; i < num_tokens; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    if (slot >= num_blocks * ORC_BLOCK) return ORC_ERR_SLOT;
    int64_t block = slot / ORC_BLOCK;
    int64_t offset = slot % ORC_BLOCK;
    for (int g = 0; g < num_kv_heads; ++g) {
      int64_t dst = ((block * num_kv_heads + g) * ORC_BLOCK + offset) * head_dim;
      int64_t src = (i * num_kv_heads + g) * head_dim;
      for (int e = 0; e < head_dim; ++e) {
        k_cache[dst + e] = k[src + e];
        v_cache[dst + e] = v[src + e];
      }
    }
  }
  return ORC_OK;
}

/*
 * Attention of one query row over an explicit list of logical token positions:
 *   s_t = scale * sum_e q[e] * K_t[e]           (dot product with each cached key)
 *   out = sum_t exp(s_t - max s) V_t / sum_t exp(s_t - max s)     (softmax, then weighted V)
 * [tfcache] section on why plain recomputation fails (the Attention formula);
 * [primer] section 2.2 (the new token's Q against all cached K, weights applied to V).
 * Logical token t of the sequence lives in physical block block_row[t / 16], offset t % 16
 * ([primer] section 4.1).  Subtracting the max is the textbook stable softmax; it does not
 * change the value.  An empty list gives a zero row.
 */
static int attend_one_row(double* out, const uint16_t* q_row, const pool_t* k_pool,
                          const pool_t* v_pool, const int32_t* block_row,
                          int max_blocks_per_seq, int64_t num_blocks, int num_kv_heads,
                          int head_dim, int kv_head, double scale, const int64_t* tokens,
                          int64_t n_tokens) {
  for (int e = 0; e < head_dim; ++e) out[e] = 0.0;
  if (n_tokens == 0) return ORC_OK;
  double* logits = (double*)malloc((size_t)n_tokens * sizeof(double));
  if (!logits) return ORC_ERR_MEM;
  int64_t* rows = (int64_t*)malloc((size_t)n_tokens * sizeof(int64_t));
  if (!rows) {
    free(logits);
    return ORC_ERR_MEM;
  }
  for (int64_t j = 0; j < n_tokens; ++j) {
    int64_t t = tokens[j];
    int64_t logical_block = t / ORC_BLOCK;
    int64_t offset = t % ORC_BLOCK;
    if (t < 0 || logical_block >= max_blocks_per_seq) {
      free(logits);
      free(rows);
      return ORC_ERR_INDEX;
    }
    int64_t physical = block_row[logical_block];
    if (physical < 0 || physical >= num_blocks) {
      free(logits);
      free(rows);
      return ORC_ERR_BLOCK;
    }
    rows[j] = (physical * num_kv_heads + kv_head) * ORC_BLOCK + offset;
    double dot = 0.0;
    for (int e = 0; e < head_dim; ++e)
      dot += bf16_to_double(q_row[e]) * pool_value(k_pool, rows[j], head_dim, e);
    logits[j] = scale * dot;
  }
  double m = logits[0];
  for (int64_t j = 1; j < n_tokens; ++j)
    if (logits[j] > m) m = logits[j];
  double denom = 0.0;
  for (int64_t j = 0; j < n_tokens; ++j) {
    logits[j] = exp(logits[j] - m); /* now the unnormalised weight */
    denom += logits[j];
  }
  for (int64_t j = 0; j < n_tokens; ++j)
    for (int e = 0; e < head_dim; ++e)
      out[e] += logits[j] * pool_value(v_pool, rows[j], head_dim, e);
  for (int e = 0; e < head_dim; ++e) out[e] /= denom;
  free(logits);
  free(rows);
  return ORC_OK;
}

/*
 * Paged decode attention for the rows listed in `row_ids` (each = b * Hq + h), or for all
 * B*Hq rows when row_ids is NULL; out has one d-vector per computed row, in list order.
 * Query head h reads kv head h / (Hq / Hkv) (grouped-query attention, as [novita] section
 * "Key technique 1" requires the sparse path to stay compatible with).  The attended tokens
 * are [start, L_b), start = max(0, L_b - window) when window > 0, else 0: the sliding window
 * keeps only the most recent `window` tokens ([primer] section 4.3).  L_b counts the token
 * appended this step.
 */
static int paged_decode_pools(double* out, const uint16_t* q, const pool_t* k_pool,
                              const pool_t* v_pool, const int32_t* block_tables,
                              const int32_t* context_lens, int batch, int num_q_heads,
                              int num_kv_heads, int head_dim, int64_t num_blocks,
                              int max_blocks_per_seq, double scale, int window,
                              const int64_t* row_ids, int64_t n_rows) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return ORC_ERR_ARG;
  if (num_q_heads % num_kv_heads != 0) return ORC_ERR_ARG;
  int group = num_q_heads / num_kv_heads;
  int64_t total = row_ids ? n_rows : (int64_t)batch * num_q_heads;
  int status = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < total; ++r) {
    int64_t row = row_ids ? row_ids[r] : r;
    int b = (int)(row / num_q_heads);
    int h = (int)(row % num_q_heads);
    int st = ORC_OK;
    if (b < 0 || b >= batch) {
      st = ORC_ERR_ARG;
    } else {
      int64_t len = context_lens[b];
      if (len < 0 || len > (int64_t)max_blocks_per_seq * ORC_BLOCK) {
        st = ORC_ERR_LEN;
      } else {
        int64_t start = 0;
        if (window > 0 && len > window) start = len - window;
        int64_t n = len - start;
        int64_t* tokens = (int64_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
        if (!tokens) {
          st = ORC_ERR_MEM;
        } else {
          for (int64_t j = 0; j < n; ++j) tokens[j] = start + j;
          st = attend_one_row(out + r * head_dim, q + row * head_dim, k_pool, v_pool,
                              block_tables + (int64_t)b * max_blocks_per_seq,
                              max_blocks_per_seq, num_blocks, num_kv_heads, head_dim,
                              h / group, scale, tokens, n);
          free(tokens);
        }
      }
    }
    if (st != ORC_OK) {
#pragma omp critical
      status = st;
    }
  }
  return status;
}

int oracle_paged_decode(double* out, const uint16_t* q, const uint16_t* k_cache,
                        const uint16_t* v_cache, const int32_t* block_tables,
                        const int32_t* context_lens, int batch, int num_q_heads,
                        int num_kv_heads, int head_dim, int64_t num_blocks,
                        int max_blocks_per_seq, double scale, int window,
                        const int64_t* row_ids, int64_t n_rows) {
  pool_t k_pool = {k_cache, NULL, NULL}, v_pool = {v_cache, NULL, NULL};
  return paged_decode_pools(out, q, &k_pool, &v_pool, block_tables, context_lens, batch,
                            num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks_per_seq,
                            scale, window, row_ids, n_rows);
}

/*
 * INT8 KV cache.  [primer] section 4.2 stores K and V as 8-bit integers to halve the cache,
 * and section 5.2 turns it on with vLLM's --kv-cache-dtype int8; neither gives the scheme.
 * Read as symmetric absmax quantization of each (token, kv head) row of d values:
 *   s = max_e |x_e| / 127            (one fp32 scale per row)
 *   c_e = round_half_even(x_e / s), clamped to [-127, 127]
 * and the row's values are c_e * s.  The division and the rounding are single-precision
 * IEEE operations: they decide an integer, so they are taken in the precision the kernel
 * takes them in.  A row of zeros gets s = 0 and codes 0; a non-finite element is refused.
 * A code c is stored as the byte c + 128 (the library's pool format); a byte b reads as the
 * code b - 128.
 */
static int quantize_row(uint8_t* codes, float* scale, const uint16_t* x, int head_dim) {
  float amax = 0.0f;
  for (int e = 0; e < head_dim; ++e) {
    float v = bf16_to_float(x[e]);
    if (!isfinite(v)) return ORC_ERR_VALUE;
    if (fabsf(v) > amax) amax = fabsf(v);
  }
  float s = amax / 127.0f;
  *scale = s;
  for (int e = 0; e < head_dim; ++e) {
    if (s == 0.0f) {
      codes[e] = 128;  /* code 0 */
      continue;
    }
    float c = rintf(bf16_to_float(x[e]) / s);
    if (c > 127.0f) c = 127.0f;
    if (c < -127.0f) c = -127.0f;
    codes[e] = (uint8_t)((int)c + 128);
  }
  return ORC_OK;
}

/* Quantize n_rows rows of d bf16 values: codes [n_rows][d], scales [n_rows]. */
int oracle_quantize_rows(uint8_t* codes, float* scales, const uint16_t* x, int64_t n_rows,
                         int head_dim) {
  if (n_rows < 0 || head_dim <= 0) return ORC_ERR_ARG;
  for (int64_t r = 0; r < n_rows; ++r) {
    int st = quantize_row(codes + r * head_dim, scales + r, x + r * head_dim, head_dim);
    if (st != ORC_OK) return st;
  }
  return ORC_OK;
}

/*
 * Append into INT8 pools: as oracle_kv_append, with each (token, kv head) row of K and of V
 * quantized on the way in.  Code pools are [NB][Hkv][16][d] bytes (code + 128), scale pools
 * [NB][Hkv][16].
 */
int oracle_kv_append_q8(uint8_t* k_codes, uint8_t* v_codes, float* k_scales, float* v_scales,
                        const uint16_t* k, const uint16_t* v, const int64_t* slot_mapping,
                        int64_t num_tokens, int num_kv_heads, int head_dim, int64_t num_blocks) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0) return ORC_ERR_ARG;
  for (int64_t i = 0; i < num_tokens; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    if (slot >= num_blocks * ORC_BLOCK) return ORC_ERR_SLOT;
    int64_t block = slot / ORC_BLOCK;
    int64_t offset = slot % ORC_BLOCK;
    for (int g = 0; g < num_kv_heads; ++g) {
      int64_t row = (block * num_kv_heads + g) * ORC_BLOCK + offset;
      int64_t src = (i * num_kv_heads + g) * head_dim;
      int st = quantize_row(k_codes + row * head_dim, k_scales + row, k + src, head_dim);
      if (st == ORC_OK) st = quantize_row(v_codes + row * head_dim, v_scales + row, v + src, head_dim);
      if (st != ORC_OK) return st;
    }
  }
  return ORC_OK;
}

/*
 * Paged decode attention over INT8 pools: oracle_paged_decode with every K and V element
 * dequantized (code * scale, exact in fp64) where it is used.
 */
int oracle_paged_decode_q8(double* out, const uint16_t* q, const uint8_t* k_codes,
                           const float* k_scales, const uint8_t* v_codes, const float* v_scales,
                           const int32_t* block_tables, const int32_t* context_lens, int batch,
                           int num_q_heads, int num_kv_heads, int head_dim, int64_t num_blocks,
                           int max_blocks_per_seq, double scale, int window,
                           const int64_t* row_ids, int64_t n_rows) {
  pool_t k_pool = {NULL, k_codes, k_scales}, v_pool = {NULL, v_codes, v_scales};
  return paged_decode_pools(out, q, &k_pool, &v_pool, block_tables, context_lens, batch,
                            num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks_per_seq,
                            scale, window, row_ids, n_rows);
}

/*
 * Sparse decode attention: the attended set of (b, kv head g) is the kept list
 * kept[b][g][0 : kept_lens[b]] ([novita] section "System model": the layer attends only the
 * KV pairs it retained).  The list must be strictly ascending and inside [0, L_b).
 */
static int sparse_decode_pools(double* out, const uint16_t* q, const pool_t* k_pool,
                               const pool_t* v_pool, const int32_t* block_tables,
                               const int32_t* context_lens, const int32_t* kept,
                               const int32_t* kept_lens, int max_kept, int batch, int num_q_heads,
                               int num_kv_heads, int head_dim, int64_t num_blocks,
                               int max_blocks_per_seq, double scale, const int64_t* row_ids,
                               int64_t n_rows) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || max_kept < 0)
    return ORC_ERR_ARG;
  if (num_q_heads % num_kv_heads != 0) return ORC_ERR_ARG;
  int group = num_q_heads / num_kv_heads;
  int64_t total = row_ids ? n_rows : (int64_t)batch * num_q_heads;
  int status = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < total; ++r) {
    int64_t row = row_ids ? row_ids[r] : r;
    int b = (int)(row / num_q_heads);
    int h = (int)(row % num_q_heads);
    int g = h / group;
    int st = ORC_OK;
    int64_t n = (b >= 0 && b < batch) ? kept_lens[b] : -1;
    if (n < 0 || n > max_kept) {
      st = ORC_ERR_LEN;
    } else {
      const int32_t* list = kept + ((int64_t)b * num_kv_heads + g) * max_kept;
      int64_t* tokens = (int64_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
      if (!tokens) {
        st = ORC_ERR_MEM;
      } else {
        for (int64_t j = 0; j < n && st == ORC_OK; ++j) {
          tokens[j] = list[j];
          if (list[j] < 0 || list[j] >= context_lens[b]) st = ORC_ERR_INDEX;
          if (j > 0 && list[j] <= list[j - 1]) st = ORC_ERR_INDEX;
        }
        if (st == ORC_OK)
          st = attend_one_row(out + r * head_dim, q + row * head_dim, k_pool, v_pool,
                              block_tables + (int64_t)b * max_blocks_per_seq,
                              max_blocks_per_seq, num_blocks, num_kv_heads, head_dim, g,
                              scale, tokens, n);
        free(tokens);
      }
    }
    if (st != ORC_OK) {
#pragma omp critical
      status = st;
    }
  }
  return status;
}

int oracle_sparse_decode(double* out, const uint16_t* q, const uint16_t* k_cache,
                         const uint16_t* v_cache, const int32_t* block_tables,
                         const int32_t* context_lens, const int32_t* kept, const int32_t* kept_lens,
                         int max_kept, int batch, int num_q_heads, int num_kv_heads,
                         int head_dim, int64_t num_blocks, int max_blocks_per_seq, double scale,
                         const int64_t* row_ids, int64_t n_rows) {
  pool_t k_pool = {k_cache, NULL, NULL}, v_pool = {v_cache, NULL, NULL};
  return sparse_decode_pools(out, q, &k_pool, &v_pool, block_tables, context_lens, kept,
                             kept_lens, max_kept, batch, num_q_heads, num_kv_heads, head_dim,
                             num_blocks, max_blocks_per_seq, scale, row_ids, n_rows);
}

/* Sparse decode attention over INT8 pools: every K and V element read as code * row scale. */
int oracle_sparse_decode_q8(double* out, const uint16_t* q, const uint8_t* k_codes,
                            const float* k_scales, const uint8_t* v_codes, const float* v_scales,
                            const int32_t* block_tables, const int32_t* context_lens,
                            const int32_t* kept, const int32_t* kept_lens, int max_kept,
                            int batch, int num_q_heads, int num_kv_heads, int head_dim,
                            int64_t num_blocks, int max_blocks_per_seq, double scale,
                            const int64_t* row_ids, int64_t n_rows) {
  pool_t k_pool = {NULL, k_codes, k_scales}, v_pool = {NULL, v_codes, v_scales};
  return sparse_decode_pools(out, q, &k_pool, &v_pool, block_tables, context_lens, kept,
                             kept_lens, max_kept, batch, num_q_heads, num_kv_heads, head_dim,
                             num_blocks, max_blocks_per_seq, scale, row_ids, n_rows);
}

/*
 * Logits of one query row over an explicit list of logical positions:
 * logits[j] = scale * sum_e q[e] * K_{tokens[j]}[e]  (as in attend_one_row; K read through its
 * pool, so INT8 rows are code * scale).
 */
static int row_logits(double* logits, const uint16_t* q_row, const pool_t* k_pool,
                      const int32_t* block_row, int max_blocks_per_seq, int64_t num_blocks,
                      int num_kv_heads, int head_dim, int kv_head, double scale,
                      const int64_t* tokens, int64_t n_tokens) {
  for (int64_t j = 0; j < n_tokens; ++j) {
    int64_t t = tokens[j];
    int64_t logical_block = t / ORC_BLOCK;
    if (t < 0 || logical_block >= max_blocks_per_seq) return ORC_ERR_INDEX;
    int64_t physical = block_row[logical_block];
    if (physical < 0 || physical >= num_blocks) return ORC_ERR_BLOCK;
    int64_t row = (physical * num_kv_heads + kv_head) * ORC_BLOCK + t % ORC_BLOCK;
    double dot = 0.0;
    for (int e = 0; e < head_dim; ++e)
      dot += bf16_to_double(q_row[e]) * pool_value(k_pool, row, head_dim, e);
    logits[j] = scale * dot;
  }
  return ORC_OK;
}

/*
 * Sparsification score of one decode step ([novita] section "2. Attention modification",
 * the scoring step built on FlashAttention): the attention pass yields each query row's
 * maximum logit m (rowmax) and normaliser l = sum_t exp(s_t - m); a second step turns every
 * attended key's logit into its softmax probability p_t = exp(s_t - m) / l and sums those
 * probabilities into the key's score.  One KV row serves the G query heads of its kv head,
 * so the score of (b, kv head g, position t) adds the probabilities of those G heads.
 * For each listed segment seg = b * Hkv + g (all B*Hkv when seg_ids is NULL):
 *   score_add[seg][t] = sum over the group's heads h of p_{h,t}   (t attended; 0 elsewhere),
 *   lse[seg][i]      = m + log(l) of head h = g*G + i              (the row's log-sum-exp).
 * The attended set is that of oracle_paged_decode (window as there); stride >= every L_b.
 * An empty set gives a zero score row and lse = -infinity.
 */
static int decode_scores_pools(double* score_add, double* lse, const uint16_t* q,
                               const pool_t* k_pool, const int32_t* block_tables,
                               const int32_t* context_lens, int batch, int num_q_heads,
                               int num_kv_heads, int head_dim, int64_t num_blocks,
                               int max_blocks_per_seq, double scale, int window, int64_t stride,
                               const int64_t* seg_ids, int64_t n_segs) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0) return ORC_ERR_ARG;
  if (num_q_heads % num_kv_heads != 0 || stride < 0) return ORC_ERR_ARG;
  int group = num_q_heads / num_kv_heads;
  int64_t total = seg_ids ? n_segs : (int64_t)batch * num_kv_heads;
  int status = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < total; ++r) {
    int64_t seg = seg_ids ? seg_ids[r] : r;
    int b = (int)(seg / num_kv_heads);
    int g = (int)(seg % num_kv_heads);
    double* score = score_add + r * stride;
    for (int64_t t = 0; t < stride; ++t) score[t] = 0.0;
    int st = ORC_OK;
    if (b < 0 || b >= batch) {
      st = ORC_ERR_ARG;
    } else {
      int64_t len = context_lens[b];
      int64_t start = 0;
      if (len < 0 || len > (int64_t)max_blocks_per_seq * ORC_BLOCK || len > stride) {
        st = ORC_ERR_LEN;
      } else {
        if (window > 0 && len > window) start = len - window;
        int64_t n = len - start;
        int64_t* tokens = (int64_t*)malloc((size_t)(n > 0 ? n : 1) * sizeof(int64_t));
        double* logits = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
        if (!tokens || !logits) {
          st = ORC_ERR_MEM;
        } else {
          for (int64_t j = 0; j < n; ++j) tokens[j] = start + j;
          for (int i = 0; i < group && st == ORC_OK; ++i) {
            int h = g * group + i;
            double* lse_out = lse + r * group + i;
            if (n == 0) {
              *lse_out = -INFINITY;
              continue;
            }
            st = row_logits(logits, q + ((int64_t)b * num_q_heads + h) * head_dim, k_pool,
                            block_tables + (int64_t)b * max_blocks_per_seq, max_blocks_per_seq,
                            num_blocks, num_kv_heads, head_dim, g, scale, tokens, n);
            if (st != ORC_OK) break;
            /* first pass: rowmax and l */
            double m = logits[0];
            for (int64_t j = 1; j < n; ++j)
              if (logits[j] > m) m = logits[j];
            double l = 0.0;
            for (int64_t j = 0; j < n; ++j) l += exp(logits[j] - m);
            /* second pass: probabilities, summed into the keys' scores */
            for (int64_t j = 0; j < n; ++j) score[tokens[j]] += exp(logits[j] - m) / l;
            *lse_out = m + log(l);
          }
        }
        free(tokens);
        free(logits);
      }
    }
    if (st != ORC_OK) {
#pragma omp critical
      status = st;
    }
  }
  return status;
}

/* The decode score over a bf16 K pool (the attended set of oracle_paged_decode). */
int oracle_decode_scores(double* score_add, double* lse, const uint16_t* q,
                         const uint16_t* k_cache, const int32_t* block_tables,
                         const int32_t* context_lens, int batch, int num_q_heads,
                         int num_kv_heads, int head_dim, int64_t num_blocks,
                         int max_blocks_per_seq, double scale, int window, int64_t stride,
                         const int64_t* seg_ids, int64_t n_segs) {
  pool_t k_pool = {k_cache, NULL, NULL};
  return decode_scores_pools(score_add, lse, q, &k_pool, block_tables, context_lens, batch,
                             num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks_per_seq,
                             scale, window, stride, seg_ids, n_segs);
}

/* The decode score over an INT8 K pool: every K element read as code * scale of its row. */
int oracle_decode_scores_q8(double* score_add, double* lse, const uint16_t* q,
                            const uint8_t* k_codes, const float* k_scales,
                            const int32_t* block_tables, const int32_t* context_lens, int batch,
                            int num_q_heads, int num_kv_heads, int head_dim, int64_t num_blocks,
                            int max_blocks_per_seq, double scale, int window, int64_t stride,
                            const int64_t* seg_ids, int64_t n_segs) {
  pool_t k_pool = {NULL, k_codes, k_scales};
  return decode_scores_pools(score_add, lse, q, &k_pool, block_tables, context_lens, batch,
                             num_q_heads, num_kv_heads, head_dim, num_blocks, max_blocks_per_seq,
                             scale, window, stride, seg_ids, n_segs);
}

/*
 * Prefill-side sparsification score ([novita] section "2. Attention modification": the
 * PyramidKV-style score).  After a prompt of L_b tokens, the score of key i in kv head g is
 * the sum of its softmax probabilities A[j][i] over the instruction window, the last alpha
 * query positions j in [L_b - alpha, L_b), and over the G query heads sharing kv head g.
 * Attention is causal: row j attends keys [0, j].  The page computes it from the forward
 * pass's rowmax and l (their log-sum-exp lse_j): A[j][i] = exp(s_ji - lse_j).  With
 * lse_given == 0 the oracle first computes lse_j itself (max + log of the sum of
 * exponentials, the textbook stable form) and writes it out; otherwise it takes lse as given.
 *   q_win [B][alpha][Hq][d]: the query of position L_b - alpha + r is row r (rows whose
 *                           position is negative, L_b < alpha, are not used)
 *   lse   [B][Hq][alpha]:   in (lse_given) or out; unused rows get -infinity
 *   score_add [segments][stride]: each key's score (this call's addition), stride >= L_b.
 */
int oracle_prefill_scores(double* score_add, double* lse, int lse_given, const uint16_t* q_win,
                          const uint16_t* k_cache, const int32_t* block_tables,
                          const int32_t* context_lens, int batch, int num_q_heads, int num_kv_heads,
                          int head_dim, int64_t num_blocks, int max_blocks_per_seq, int alpha,
                          double scale, int64_t stride, const int64_t* seg_ids, int64_t n_segs) {
  if (batch < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || alpha <= 0) return ORC_ERR_ARG;
  if (num_q_heads % num_kv_heads != 0 || stride < 0) return ORC_ERR_ARG;
  pool_t k_pool = {k_cache, NULL, NULL};
  int group = num_q_heads / num_kv_heads;
  int64_t total = seg_ids ? n_segs : (int64_t)batch * num_kv_heads;
  int status = ORC_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < total; ++r) {
    int64_t seg = seg_ids ? seg_ids[r] : r;
    int b = (int)(seg / num_kv_heads);
    int g = (int)(seg % num_kv_heads);
    double* score = score_add + r * stride;
    for (int64_t t = 0; t < stride; ++t) score[t] = 0.0;
    int st = ORC_OK;
    int64_t len = (b >= 0 && b < batch) ? context_lens[b] : -1;
    if (len < 0 || len > (int64_t)max_blocks_per_seq * ORC_BLOCK || len > stride) st = ORC_ERR_LEN;
    int64_t* tokens = (int64_t*)malloc((size_t)(len > 0 ? len : 1) * sizeof(int64_t));
    double* logits = (double*)malloc((size_t)(len > 0 ? len : 1) * sizeof(double));
    if (st == ORC_OK && (!tokens || !logits)) st = ORC_ERR_MEM;
    for (int64_t t = 0; st == ORC_OK && t < len; ++t) tokens[t] = t;
    for (int hi = 0; st == ORC_OK && hi < group; ++hi) {
      int h = g * group + hi;
      for (int rw = 0; rw < alpha && st == ORC_OK; ++rw) {
        int64_t j = len - alpha + rw; /* this window row's position */
        double* lse_jh = lse + ((int64_t)b * num_q_heads + h) * alpha + rw;
        if (j < 0) {
          if (!lse_given) *lse_jh = -INFINITY;
          continue;
        }
        /* causal: row j attends keys [0, j] */
        st = row_logits(logits, q_win + (((int64_t)b * alpha + rw) * num_q_heads + h) * head_dim,
                        &k_pool, block_tables + (int64_t)b * max_blocks_per_seq, max_blocks_per_seq,
                        num_blocks, num_kv_heads, head_dim, g, scale, tokens, j + 1);
        if (st != ORC_OK) break;
        double row_lse;
        if (lse_given) {
          row_lse = *lse_jh;
        } else {
          double m = logits[0];
          for (int64_t i = 1; i <= j; ++i)
            if (logits[i] > m) m = logits[i];
          double l = 0.0;
          for (int64_t i = 0; i <= j; ++i) l += exp(logits[i] - m);
          row_lse = m + log(l);
          *lse_jh = row_lse;
        }
        for (int64_t i = 0; i <= j; ++i) score[i] += exp(logits[i] - row_lse);
      }
    }
    free(tokens);
    free(logits);
    if (st != ORC_OK) {
#pragma omp critical
      status = st;
    }
  }
  return status;
}

/* Candidate ordering for the top-k: higher score first; equal scores, lower position first. */
typedef struct {
  double score;
  int32_t position;
} orc_candidate;

static int candidate_order(const void* a, const void* b) {
  const orc_candidate* x = (const orc_candidate*)a;
  const orc_candidate* y = (const orc_candidate*)b;
  if (x->score > y->score) return -1;
  if (x->score < y->score) return 1;
  return (x->position < y->position) ? -1 : (x->position > y->position);
}

/*
 * Kept-token selection per (sequence b, kv head g) ([novita] section "System model": drop
 * low-score KV, retain high-score and recent KV; section "2. Attention modification": per
 * layer and head, keep the top-k tokens by score; the introduction's attention sinks: the
 * start token is always important):
 *   K = n_sink + k_top + n_recent.  If L <= K keep every position 0..L-1.
 *   Otherwise keep [0, n_sink), the k_top best candidates of [n_sink, L - n_recent) by
 *   (score descending, position ascending), and [L - n_recent, L); output ascending.
 * Scores are compared as the fp32 values given (widening to double is exact; -0 == +0).
 */
int oracle_select_topk(int32_t* kept_out, int32_t* kept_lens_out, const float* scores,
                       int score_stride, const int32_t* context_lens, int batch,
                       int num_kv_heads, int n_sink, int n_recent, int k_top) {
  if (batch < 0 || num_kv_heads <= 0 || n_sink < 0 || n_recent < 0 || k_top < 0)
    return ORC_ERR_ARG;
  int64_t keep_max = (int64_t)n_sink + k_top + n_recent;
  int status = ORC_OK;
  for (int b = 0; b < batch; ++b) {
    int64_t len = context_lens[b];
    if (len < 0 || len > score_stride) return ORC_ERR_LEN;
    kept_lens_out[b] = (int32_t)(len < keep_max ? len : keep_max);
  }
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t pair = 0; pair < (int64_t)batch * num_kv_heads; ++pair) {
    int b = (int)(pair / num_kv_heads);
    int64_t len = context_lens[b];
    const float* row = scores + pair * score_stride;
    int32_t* dst = kept_out + pair * keep_max;
    if (len <= keep_max) {
      for (int64_t t = 0; t < len; ++t) dst[t] = (int32_t)t;
      continue;
    }
    int64_t first = n_sink, last = len - n_recent; /* candidate range [first, last) */
    int64_t n_cand = last - first;
    orc_candidate* cand = (orc_candidate*)malloc((size_t)n_cand * sizeof(orc_candidate));
    unsigned char* chosen = (unsigned char*)calloc((size_t)len, 1);
    int st = (cand && chosen) ? ORC_OK : ORC_ERR_MEM;
    for (int64_t c = 0; c < n_cand && st == ORC_OK; ++c) {
      float s = row[first + c];
      if (isnan(s)) st = ORC_ERR_NAN;
      cand[c].score = (double)s;
      cand[c].position = (int32_t)(first + c);
    }
    if (st == ORC_OK) {
      qsort(cand, (size_t)n_cand, sizeof(orc_candidate), candidate_order);
      for (int64_t t = 0; t < n_sink; ++t) chosen[t] = 1;
      for (int64_t c = 0; c < k_top; ++c) chosen[cand[c].position] = 1;
      for (int64_t t = last; t < len; ++t) chosen[t] = 1;
      int64_t w = 0;
      for (int64_t t = 0; t < len; ++t)
        if (chosen[t]) dst[w++] = (int32_t)t;
      if (w != keep_max) st = ORC_ERR_ARG;
    }
    free(cand);
    free(chosen);
    if (st != ORC_OK) {
#pragma omp critical
      status = st;
    }
  }
  return status;
}

/*
 * Compaction: compact position j of (b, g) -- slot dst_block_tables[b][j / 16]*16 + j % 16
 * of the destination pool -- receives source token kept[b][g][j] (found through the source
 * block table).  This realises the per-layer block-table policy of [novita] section "Key
 * technique 1" (Fig. 5): a sparse layer's retained KV lives in its own 16-token blocks.
 * The copy behind both compactions moves rows of elem_bytes * head_dim bytes (bf16 elements,
 * or INT8 codes whose row scales move with them when the scale arrays are given).
 */
static int compact_pools(unsigned char* dst_k, unsigned char* dst_v, float* dst_ks, float* dst_vs,
                         const int32_t* dst_block_tables, int64_t dst_num_blocks,
                         int dst_max_blocks_per_seq, const unsigned char* src_k,
                         const unsigned char* src_v, const float* src_ks, const float* src_vs,
                         const int32_t* src_block_tables, const int32_t* context_lens,
                         const int32_t* kept, const int32_t* kept_lens, int max_kept, int batch,
                         int num_kv_heads, int head_dim, int64_t src_num_blocks,
                         int src_max_blocks_per_seq, size_t elem_bytes) {
  if (batch < 0 || num_kv_heads <= 0 || head_dim <= 0 || max_kept < 0) return ORC_ERR_ARG;
  size_t row_bytes = elem_bytes * (size_t)head_dim;
  for (int b = 0; b < batch; ++b) {
    int64_t n = kept_lens[b];
    if (n < 0 || n > max_kept || n > (int64_t)dst_max_blocks_per_seq * ORC_BLOCK)
      return ORC_ERR_LEN;
    for (int g = 0; g < num_kv_heads; ++g) {
      const int32_t* list = kept + ((int64_t)b * num_kv_heads + g) * max_kept;
      for (int64_t j = 0; j < n; ++j) {
        int64_t t = list[j];
        if (t < 0 || t >= context_lens[b] || t / ORC_BLOCK >= src_max_blocks_per_seq)
          return ORC_ERR_INDEX;
        int64_t src_block = src_block_tables[(int64_t)b * src_max_blocks_per_seq + t / ORC_BLOCK];
        int64_t dst_block = dst_block_tables[(int64_t)b * dst_max_blocks_per_seq + j / ORC_BLOCK];
        if (src_block < 0 || src_block >= src_num_blocks) return ORC_ERR_BLOCK;
        if (dst_block < 0 || dst_block >= dst_num_blocks) return ORC_ERR_BLOCK;
        int64_t src = (src_block * num_kv_heads + g) * ORC_BLOCK + t % ORC_BLOCK;
        int64_t dst = (dst_block * num_kv_heads + g) * ORC_BLOCK + j % ORC_BLOCK;
        memcpy(dst_k + dst * row_bytes, src_k + src * row_bytes, row_bytes);
        memcpy(dst_v + dst * row_bytes, src_v + src * row_bytes, row_bytes);
        if (dst_ks) {
          dst_ks[dst] = src_ks[src];
          dst_vs[dst] = src_vs[src];
        }
      }
    }
  }
  return ORC_OK;
}

int oracle_compact(uint16_t* dst_k, uint16_t* dst_v, const int32_t* dst_block_tables,
                   int64_t dst_num_blocks, int dst_max_blocks_per_seq, const uint16_t* src_k,
                   const uint16_t* src_v, const int32_t* src_block_tables,
                   const int32_t* context_lens, const int32_t* kept, const int32_t* kept_lens,
                   int max_kept, int batch, int num_kv_heads, int head_dim,
                   int64_t src_num_blocks, int src_max_blocks_per_seq) {
  return compact_pools((unsigned char*)dst_k, (unsigned char*)dst_v, NULL, NULL, dst_block_tables,
                       dst_num_blocks, dst_max_blocks_per_seq, (const unsigned char*)src_k,
                       (const unsigned char*)src_v, NULL, NULL, src_block_tables, context_lens,
                       kept, kept_lens, max_kept, batch, num_kv_heads, head_dim, src_num_blocks,
                       src_max_blocks_per_seq, sizeof(uint16_t));
}

/*
 * Compaction of INT8 pools: the kept rows' codes and their row scales move together, so the
 * compact pool holds the same values (code * scale) at the new positions.
 */
int oracle_compact_q8(uint8_t* dst_k, uint8_t* dst_v, float* dst_ks, float* dst_vs,
                      const int32_t* dst_block_tables, int64_t dst_num_blocks,
                      int dst_max_blocks_per_seq, const uint8_t* src_k, const uint8_t* src_v,
                      const float* src_ks, const float* src_vs, const int32_t* src_block_tables,
                      const int32_t* context_lens, const int32_t* kept, const int32_t* kept_lens,
                      int max_kept, int batch, int num_kv_heads, int head_dim,
                      int64_t src_num_blocks, int src_max_blocks_per_seq) {
  if (!dst_ks || !dst_vs || !src_ks || !src_vs) return ORC_ERR_ARG;
  return compact_pools((unsigned char*)dst_k, (unsigned char*)dst_v, dst_ks, dst_vs,
                       dst_block_tables, dst_num_blocks, dst_max_blocks_per_seq,
                       (const unsigned char*)src_k, (const unsigned char*)src_v, src_ks, src_vs,
                       src_block_tables, context_lens, kept, kept_lens, max_kept, batch,
                       num_kv_heads, head_dim, src_num_blocks, src_max_blocks_per_seq, 1);
}

/*
 * A K/V pool pair being written: bf16 elements, or INT8 codes with one fp32 scale per row.
 * write_row stores one bf16 row of K and of V at row r (rows as in pool_t), quantizing them
 * (quantize_row) for INT8 pools; a non-finite value leaves both rows unwritten.
 */
typedef struct {
  uint16_t* k_bf16;
  uint16_t* v_bf16;
  uint8_t* k_codes;
  uint8_t* v_codes;
  float* k_scales;
  float* v_scales;
} wpool_t;

static int write_row(const wpool_t* p, int64_t r, const uint16_t* k, const uint16_t* v,
                     int head_dim) {
  if (p->k_bf16) {
    memcpy(p->k_bf16 + r * head_dim, k, (size_t)head_dim * sizeof(uint16_t));
    memcpy(p->v_bf16 + r * head_dim, v, (size_t)head_dim * sizeof(uint16_t));
    return ORC_OK;
  }
  uint8_t* kc = (uint8_t*)malloc((size_t)head_dim);
  uint8_t* vc = (uint8_t*)malloc((size_t)head_dim);
  float ks = 0.0f, vs = 0.0f;
  int st = (kc && vc) ? ORC_OK : ORC_ERR_MEM;
  if (st == ORC_OK) st = quantize_row(kc, &ks, k, head_dim);
  if (st == ORC_OK) st = quantize_row(vc, &vs, v, head_dim);
  if (st == ORC_OK) {
    memcpy(p->k_codes + r * head_dim, kc, (size_t)head_dim);
    memcpy(p->v_codes + r * head_dim, vc, (size_t)head_dim);
    p->k_scales[r] = ks;
    p->v_scales[r] = vs;
  }
  free(kc);
  free(vc);
  return st;
}

/*
 * Rolling admission of one decode step's token into a sparse layer of fixed budget ([novita]
 * section "System model": a sparse layer keeps the high-score and the recent KV and drops the
 * rest; the token entering the cache takes the place of the lowest-score KV).  The layer's
 * compact pool holds, per (b, kv head g), `capacity` slots (slot s lives at block
 * block_tables[b][s / 16], offset s % 16); slot_pos[b][g][s] is the logical position a slot
 * holds, slot_score[b][g][s] its accumulated score, kept_lens[b] the slots in use.  The new
 * token has position L_b - 1 (context_lens counts it) and rows k_new[b][g], v_new[b][g].
 *   - Budget not full (kept_lens[b] < capacity): the token takes slot kept_lens[b].
 *   - Full: the token at position p = L_b - 1 - n_recent leaves the recent window.  It
 *     competes with the top-k set -- the slots whose positions lie in [n_sink, p).  If its
 *     score is strictly greater than the lowest score of that set (among equal lowest scores,
 *     the highest position is the weakest), the weakest one is dropped; otherwise the leaving
 *     token is dropped.  The new token takes the dropped token's slot.  Sinks and the recent
 *     window are never dropped.
 * The slot taken gets the new rows, position L_b - 1 and score 0; kept_lens[b] grows by one
 * while below capacity.  NaN scores, a missing leaving token or a bad block are refused.
 */
static int rolling_admit_pools(const wpool_t* pool, const int32_t* block_tables,
                               int64_t num_blocks, int max_blocks_per_seq, int32_t* slot_pos,
                               float* slot_score, int32_t* kept_lens, const int32_t* context_lens,
                               const uint16_t* k_new, const uint16_t* v_new, int batch,
                               int num_kv_heads, int head_dim, int capacity, int n_sink,
                               int n_recent) {
  if (batch < 0 || num_kv_heads <= 0 || head_dim <= 0 || capacity <= 0 || n_sink < 0 ||
      n_recent < 0 || n_sink + n_recent > capacity)
    return ORC_ERR_ARG;
  for (int b = 0; b < batch; ++b) {
    int64_t len = context_lens[b];
    int used = kept_lens[b];
    if (len < 1 || used < 0 || used > capacity) return ORC_ERR_LEN;
    int full = used == capacity;
    for (int g = 0; g < num_kv_heads; ++g) {
      int32_t* pos = slot_pos + ((int64_t)b * num_kv_heads + g) * capacity;
      float* score = slot_score + ((int64_t)b * num_kv_heads + g) * capacity;
      int target = used;
      if (full) {
        int64_t leaving = len - 1 - n_recent;
        int s_out = -1, s_min = -1;
        for (int s = 0; s < capacity; ++s) {
          if (score[s] != score[s]) return ORC_ERR_ARG; /* NaN */
          if (pos[s] == leaving) s_out = s;
          if (pos[s] >= n_sink && pos[s] < leaving) {
            if (s_min < 0 || score[s] < score[s_min] ||
                (score[s] == score[s_min] && pos[s] > pos[s_min]))
              s_min = s;
          }
        }
        if (s_out < 0) return ORC_ERR_INDEX;
        target = (s_min >= 0 && score[s_out] > score[s_min]) ? s_min : s_out;
      }
      int64_t logical_block = target / ORC_BLOCK;
      if (logical_block >= max_blocks_per_seq) return ORC_ERR_INDEX;
      int64_t physical = block_tables[(int64_t)b * max_blocks_per_seq + logical_block];
      if (physical < 0 || physical >= num_blocks) return ORC_ERR_BLOCK;
      int64_t row = (physical * num_kv_heads + g) * ORC_BLOCK + target % ORC_BLOCK;
      int64_t src = ((int64_t)b * num_kv_heads + g) * head_dim;
      int st = write_row(pool, row, k_new + src, v_new + src, head_dim);
      if (st != ORC_OK) return st;
      pos[target] = (int32_t)(len - 1);
      score[target] = 0.0f;
    }
    if (!full) kept_lens[b] = used + 1;
  }
  return ORC_OK;
}

int oracle_rolling_admit(uint16_t* k_cache, uint16_t* v_cache, const int32_t* block_tables,
                         int64_t num_blocks, int max_blocks_per_seq, int32_t* slot_pos,
                         float* slot_score, int32_t* kept_lens, const int32_t* context_lens,
                         const uint16_t* k_new, const uint16_t* v_new, int batch,
                         int num_kv_heads, int head_dim, int capacity, int n_sink, int n_recent) {
  wpool_t pool = {k_cache, v_cache, NULL, NULL, NULL, NULL};
  return rolling_admit_pools(&pool, block_tables, num_blocks, max_blocks_per_seq, slot_pos,
                             slot_score, kept_lens, context_lens, k_new, v_new, batch,
                             num_kv_heads, head_dim, capacity, n_sink, n_recent);
}

/*
 * Rolling admission into INT8 pools: the same choice of slot; the new token's K and V rows
 * are quantized into it (codes and row scale, as oracle_kv_append_q8 does).
 */
int oracle_rolling_admit_q8(uint8_t* k_codes, uint8_t* v_codes, float* k_scales, float* v_scales,
                            const int32_t* block_tables, int64_t num_blocks,
                            int max_blocks_per_seq, int32_t* slot_pos, float* slot_score,
                            int32_t* kept_lens, const int32_t* context_lens,
                            const uint16_t* k_new, const uint16_t* v_new, int batch,
                            int num_kv_heads, int head_dim, int capacity, int n_sink,
                            int n_recent) {
  wpool_t pool = {NULL, NULL, k_codes, v_codes, k_scales, v_scales};
  return rolling_admit_pools(&pool, block_tables, num_blocks, max_blocks_per_seq, slot_pos,
                             slot_score, kept_lens, context_lens, k_new, v_new, batch,
                             num_kv_heads, head_dim, capacity, n_sink, n_recent);
}
