/*
 * MLA decode oracle: the plain definition, in fp64, on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the package smoke check and the CPU
 * baseline leg of the benchmark do.  It shares no code, header, table or
 * helper with the CUDA kernels.
 *
 * Sources (cited by page title and section):
 *   [TL]  "用 TileLang 编写高性能 DeepSeek MLA 内核：从 FlashAttention 到
 *          FlashMLA 级性能的完整实战指南" (lmnt.cn/news/253096)
 *   [FM]  "DeepSeek开源周第一天：FlashMLA 深度分析" (pxiaoer.blog)
 *
 * What is computed (one shared latent KV head; seqlen_q query tokens per
 * sequence, one by default):
 *   [TL §先看核心难点]  q and k rows are 576 wide: 512 latent + 64 RoPE;
 *                       v is 512 wide.
 *   [TL §Split Kernel]  the same cached tile feeds both the score GEMM and the
 *                       value GEMM, so v = the first 512 columns of the cached
 *                       row; the score is q_nope.k_nope + q_pe.k_pe, i.e. one
 *                       dot product over all 576 columns.
 *   [TL §参考实现与正确性验证]  the reference concatenates the two parts,
 *                       takes einsum scores, a softmax, and the weighted sum
 *                       of v.  That is what this file does, in fp64, without
 *                       any tiling, splitting or exp2 rewriting.
 *   [TL §变体内核], [FM §内存访问优化]  the cache is paged: token t of
 *                       sequence b lives in physical page
 *                       block_table[b][t / page_size], row t % page_size;
 *                       tokens at or beyond cache_seqlens[b] do not exist.
 *
 *   [TL §变体内核]  an experimental variant keeps the KV cache in FP8
 *                       (example_mla_decode_kv_fp8.py); no format is given.
 *
 * Readings where the pages are silent:
 *   - lse is the natural-log log-sum-exp of the scaled scores,
 *     lse = m + ln(sum_t exp(s_t - m)), m = max_t s_t  (the FlashAttention
 *     convention; the kernels' base-2 internals convert to it).
 *   - a sequence of length 0 gives out = 0 and lse = -inf.
 *   - inputs are the bf16 / fp16 bit patterns exactly as stored; the oracle
 *     widens them to double and rounds nothing afterwards (the kernels round
 *     P to the input dtype; the parity tolerance absorbs that).
 *   - FP8 cache: q and every cached row are stored as e4m3 (1 sign bit, 4
 *     exponent bits with bias 7, 3 fraction bits, no infinities, S.1111.111 is
 *     NaN), each tensor with one fp32 dequantisation scale: the values the
 *     definition uses are q = q_scale * q8, k = kv_scale * k8 and
 *     v = kv_scale * v8 (v the first 512 columns of the dequantised row).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

#define MLA_D 576  /* q/k head dim: 512 latent + 64 RoPE */
#define MLA_DV 512 /* v head dim: the latent part of the cached row */

/* IEEE binary16 -> double, straight from the format's definition
 * (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits). */
static double half_bits_to_double(uint16_t x) {
  int sign = (x >> 15) & 1;
  int e = (x >> 10) & 0x1f;
  int f = x & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24); /* subnormal: f * 2^-14 * 2^-10 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(f | 0x400), e - 25); /* (1024+f) * 2^(e-15-10) */
  }
  return sign ? -v : v;
}

/* bfloat16 -> double: bf16 is the top half of an IEEE binary32. */
static double bf16_bits_to_double(uint16_t x) {
  uint32_t u = (uint32_t)x << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* e4m3 -> double, from the format's definition: 1 sign bit, 4 exponent bits
 * with bias 7, 3 fraction bits; exponent 0 is subnormal, S.1111.111 is NaN and
 * there are no infinities. */
static double e4m3_bits_to_double(uint8_t x) {
  int sign = (x >> 7) & 1;
  int e = (x >> 3) & 0xf;
  int f = x & 7;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -9); /* subnormal: f * 2^-3 * 2^-6 */
  } else if (e == 15 && f == 7) {
    v = NAN;
  } else {
    v = ldexp((double)(f | 8), e - 10); /* (8+f) * 2^(e-7-3) */
  }
  return sign ? -v : v;
}

/* dtype: 0 = fp16, 1 = bf16, 2 = e4m3 */
static double widen(uint16_t x, int dtype) {
  if (dtype == 2) return e4m3_bits_to_double((uint8_t)x);
  return dtype == 1 ? bf16_bits_to_double(x) : half_bits_to_double(x);
}

/* Element i of a stored array: 16-bit patterns (fp16, bf16) or bytes (e4m3). */
static double elem(const void *base, int64_t i, int dtype) {
  if (dtype == 2) return e4m3_bits_to_double(((const uint8_t *)base)[i]);
  return widen(((const uint16_t *)base)[i], dtype);
}

static int elem_size(int dtype) { return dtype == 2 ? 1 : 2; }

/* Exported for the exhaustive conversion pins. */
double oracle_widen(uint16_t x, int dtype) { return widen(x, dtype); }

/*
 * One (sequence, head) row of the definition.
 *   q_row       : 576 stored values of this head's query
 *   kv          : [num_pages][page_size][576] stored values
 *   table_row   : this sequence's block_table row
 *   out_row     : 512 doubles
 *   abs_row     : 512 doubles or NULL: sum_t p_t |v_t[d]|, the scale of the terms
 *                 that out_row[d] sums (the bound of its rounding error)
 *   scores      : scratch, at least seqlen doubles
 * Returns 0, or -1 if the block table points outside the cache.
 */
static int one_row(const void *q_row, const void *kv, int64_t num_pages,
                   int page_size, const int32_t *table_row, int seqlen,
                   double softmax_scale, int dtype, double q_scale, double kv_scale,
                   double *out_row, double *abs_row, double *lse_out, double *scores) {
  for (int d = 0; d < MLA_DV; ++d) out_row[d] = 0.0;
  if (abs_row)
    for (int d = 0; d < MLA_DV; ++d) abs_row[d] = 0.0;
  if (seqlen <= 0) {
    *lse_out = -INFINITY;
    return 0;
  }
  /* s_t = scale * sum_c q[c] * k_t[c]  over all 576 columns, with the
   * dequantised values q = q_scale * q_stored and k = kv_scale * k_stored */
  double m = -INFINITY;
  for (int t = 0; t < seqlen; ++t) {
    int32_t page = table_row[t / page_size];
    if (page < 0 || page >= num_pages) return -1;
    const int64_t k = ((int64_t)page * page_size + t % page_size) * MLA_D;
    double dot = 0.0;
    for (int c = 0; c < MLA_D; ++c)
      dot += q_scale * elem(q_row, c, dtype) * (kv_scale * elem(kv, k + c, dtype));
    scores[t] = softmax_scale * dot;
    if (scores[t] > m) m = scores[t];
  }
  /* Z = sum_t exp(s_t - m);  out = sum_t exp(s_t - m) / Z * v_t */
  double z = 0.0;
  for (int t = 0; t < seqlen; ++t) z += exp(scores[t] - m);
  for (int t = 0; t < seqlen; ++t) {
    int32_t page = table_row[t / page_size];
    const int64_t v = ((int64_t)page * page_size + t % page_size) * MLA_D;
    double p = exp(scores[t] - m) / z;
    for (int d = 0; d < MLA_DV; ++d) out_row[d] += p * (kv_scale * elem(kv, v + d, dtype));
    if (abs_row)
      for (int d = 0; d < MLA_DV; ++d) abs_row[d] += p * fabs(kv_scale * elem(kv, v + d, dtype));
  }
  *lse_out = m + log(z);
  return 0;
}

/*
 * Selected rows of the MLA decode definition, with seqlen_q query tokens per
 * sequence [FM §内存访问优化: Flash_fwd_mla_params carries seqlen_q, ngroups and
 * is_causal].  With one KV head the seqlen_q * h query rows of a sequence all
 * read the same cache (ngroups = h); they are stored token-major:
 *   q            : [b][seqlen_q * h][576] stored values, row r = qi * h + head
 *   kv           : [num_pages][page_size][576] stored values (one KV head)
 *   block_table  : [b][max_blocks]
 *   cache_seqlens: [b]; the cache already holds the seqlen_q new tokens, so
 *                  query token qi stands at position L - seqlen_q + qi
 *   is_causal    : query token qi sees the cached tokens t < L - (seqlen_q-1-qi)
 *                  (none if that is <= 0); otherwise every t < L
 *   row_b, row_r : n_rows (sequence, query row) pairs to evaluate
 *   out          : [n_rows][512] doubles
 *   lse          : [n_rows] doubles
 *   absw         : [n_rows][512] doubles or NULL: the softmax-weighted mean of
 *                  |v| per column (see one_row)
 *   scratch      : at least max(cache_seqlens) doubles
 * Returns 0 on success, -1 on an out-of-range page or row index.
 */
int oracle_mla_decode_rows_qs(int b, int seqlen_q, int h, int is_causal, const void *q,
                              const void *kv, int64_t num_pages, int page_size,
                              const int32_t *block_table, int max_blocks,
                              const int32_t *cache_seqlens, double softmax_scale, int dtype,
                              double q_scale, double kv_scale, int n_rows,
                              const int32_t *row_b, const int32_t *row_r, double *out,
                              double *lse, double *scratch, double *absw) {
  if (seqlen_q < 1) return -1;
  const int rows_per_seq = seqlen_q * h;
  for (int r = 0; r < n_rows; ++r) {
    int bi = row_b[r], ri = row_r[r];
    if (bi < 0 || bi >= b || ri < 0 || ri >= rows_per_seq) return -1;
    int L = cache_seqlens[bi];
    if (L > max_blocks * page_size) return -1;
    int qi = ri / h; /* query token of this row */
    int visible = is_causal ? L - (seqlen_q - 1 - qi) : L;
    if (visible < 0) visible = 0;
    const char *q_row = (const char *)q + ((int64_t)bi * rows_per_seq + ri) * MLA_D * elem_size(dtype);
    int rc = one_row(q_row, kv, num_pages, page_size, block_table + (int64_t)bi * max_blocks,
                     visible, softmax_scale, dtype, q_scale, kv_scale, out + (int64_t)r * MLA_DV,
                     absw ? absw + (int64_t)r * MLA_DV : 0, lse + r, scratch);
    if (rc) return rc;
  }
  return 0;
}

/* 16-bit inputs (no dequantisation scales). */
int oracle_mla_decode_rows_q(int b, int seqlen_q, int h, int is_causal, const uint16_t *q,
                             const uint16_t *kv, int64_t num_pages, int page_size,
                             const int32_t *block_table, int max_blocks,
                             const int32_t *cache_seqlens, double softmax_scale, int dtype,
                             int n_rows, const int32_t *row_b, const int32_t *row_r,
                             double *out, double *lse, double *scratch, double *absw) {
  return oracle_mla_decode_rows_qs(b, seqlen_q, h, is_causal, q, kv, num_pages, page_size,
                                   block_table, max_blocks, cache_seqlens, softmax_scale, dtype,
                                   1.0, 1.0, n_rows, row_b, row_r, out, lse, scratch, absw);
}

/* One query token per sequence: q is [b][h][576] and the rows are (sequence, head). */
int oracle_mla_decode_rows(int b, int h, const uint16_t *q, const uint16_t *kv,
                           int64_t num_pages, int page_size,
                           const int32_t *block_table, int max_blocks,
                           const int32_t *cache_seqlens, double softmax_scale,
                           int dtype, int n_rows, const int32_t *row_b,
                           const int32_t *row_h, double *out, double *lse,
                           double *scratch, double *absw) {
  return oracle_mla_decode_rows_q(b, 1, h, 0, q, kv, num_pages, page_size, block_table,
                                  max_blocks, cache_seqlens, softmax_scale, dtype, n_rows,
                                  row_b, row_h, out, lse, scratch, absw);
}
