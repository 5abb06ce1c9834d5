/*
 * qsa_oracle.c -- plain, slow, fp64 CPU restatement of one Qwen Sparse
 * Attention (QSA) layer step.  TEST INFRASTRUCTURE ONLY: the test suite, the
 * smoke check and the benchmark's CPU-baseline leg call it; the CUDA library
 * never links, loads or calls it, and it shares no code with that library.
 *
 * Sources, by page:
 *   [QSA]  hipfire, "QSA sparse attention and the VMM KV backend",
 *          section 02 "How QSA chooses what to read" (pooling by 4, the
 *          four-head ReLU score scaled by 1/sqrt(128), the 512-block budget
 *          plus the always-kept incomplete tail, <= 2,048 + 3 rows per query)
 *          and section 03 "How hipfire runs it on RDNA" (24 query heads over
 *          2 KV heads, one KV group of 12 query heads per selected row).
 *   [SEG]  MTPLX pull request #610 (segmented KV cache), "How it works, in
 *          plain terms" (per-segment partials merged by their log-sum-exp
 *          equal single-buffer attention) and "What changes" (rows with no
 *          visible key merge to zeros; partials stay fp32 and are rounded
 *          once).
 *
 * Readings where the pages leave a step open (each is repeated where used):
 *   R1 blocks are aligned at token 0: block b holds tokens 4b .. 4b+3.
 *   R2 completeness and the tail are judged per query row: a row at absolute
 *      position p sees tokens 0..p, has nb(p) = floor((p+1)/4) complete
 *      blocks and a tail of (p+1) mod 4 tokens, 4*nb(p) .. p.
 *   R3 the four index heads are summed without weights.
 *   R4 with nb(p) <= k every complete block is kept; the tail is outside k.
 *   R5 ties in score go to the lower block id.
 *   R6 query head h reads KV head floor(h / (Hq / Hkv)).
 *   R7 the attention logit scale is given by the caller (1/sqrt(D) by
 *      default on the Python side); lse is a natural logarithm.
 *   R8 with KV segments, attention runs over the selected rows that some
 *      segment covers; a row with no such key has output 0 and lse -inf.
 *   R9 the fp8 K/V state (hipfire section 02 table "State formats": E4M3
 *      K/V plus an f16 scale per head and token): a stored element is the
 *      E4M3 code times its row's scale.  E4M3 is sign, 4 exponent bits
 *      (bias 7), 3 mantissa bits, subnormals below 2^-6, largest finite 448,
 *      S.1111.111 NaN, no infinities.  Writing a row (the pages give no
 *      recipe): scale = f16(f32(amax / 448)), code = the E4M3 value nearest
 *      to f32(x / scale), ties to even, magnitudes above 448 saturated to
 *      448; a row whose scale is 0 stores zeros.
 *   R10 the q8 K/V state (the same table: "Q8_0 K/V"): a row is stored in
 *      blocks of 32 consecutive elements, each block as an f16 scale d and
 *      32 int8 codes, value = code * d.  Writing a block: d = f16(f32(amax
 *      / 127)), code = the integer nearest to f32(x / d), halves away from
 *      zero, limited to +-127; a block whose scale is 0 stores zeros.
 *
 * Arithmetic is IEEE fp64 throughout (built without -ffast-math).  Inputs
 * are read in their stored format (fp32, bf16 bit patterns or fp64) and
 * widened exactly to double before any arithmetic.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_F64 = 2 };

static int g_threads = 1;

/* Number of host threads the row loops may use (1 = serial). */
int qsa_oracle_set_threads(int n) {
  if (n < 1) n = 1;
  g_threads = n;
  return g_threads;
}

int qsa_oracle_get_threads(void) { return g_threads; }

/* Exact widening of one stored element to double. */
static double load_elem(const void* base, int dtype, int64_t i) {
  if (dtype == ORC_F32) return (double)((const float*)base)[i];
  if (dtype == ORC_F64) return ((const double*)base)[i];
  /* bf16: the upper 16 bits of an IEEE binary32. */
  uint32_t bits = (uint32_t)((const uint16_t*)base)[i] << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* nb(p): complete 4-token blocks visible to a row at position p (R1, R2). */
int64_t qsa_oracle_visible_blocks(int64_t p) { return (p + 1) / 4; }

/* Tail tokens of a row at position p (R2). */
int64_t qsa_oracle_tail_tokens(int64_t p) { return (p + 1) % 4; }

/*
 * Step 1, pooling [QSA 02]: each pooled block key is the mean of the 4
 * consecutive index keys of its block.
 *   idxk   [n_tokens, dim] stored values, row stride tok_stride elements
 *   pooled [n_blocks, dim] fp64, block first_block + i at row i
 * Returns 0, or -1 if a requested block is not complete in n_tokens.
 */
int qsa_oracle_pool(const void* idxk, int dtype, int64_t n_tokens, int64_t dim, int64_t tok_stride,
                    int64_t first_block, int64_t n_blocks, double* pooled) {
  if (first_block < 0 || n_blocks < 0 || 4 * (first_block + n_blocks) > n_tokens) return -1;
  for (int64_t i = 0; i < n_blocks; ++i) {
    int64_t b = first_block + i;
    for (int64_t d = 0; d < dim; ++d) {
      double s = 0.0;
      for (int64_t j = 0; j < 4; ++j) s += load_elem(idxk, dtype, (4 * b + j) * tok_stride + d);
      pooled[i * dim + d] = s / 4.0;
    }
  }
  return 0;
}

/*
 * Step 2, block scoring [QSA 02]:
 *   score[r][b] = scale * sum_{h < n_heads} max(0, q_idx[r][h] . pooled[b])
 * for every complete block b < nb(p_r) visible to row r (R2, R3); the
 * method's scale is 1/sqrt(128).  Entries b >= nb(p_r) are set to -inf:
 * those blocks are not candidates for that row.
 *   q_idx  [M, n_heads, dim] stored values
 *   pooled [n_pooled, dim] fp64
 *   scores [M, ld] fp64
 */
int qsa_oracle_score(const void* q_idx, int q_dtype, int64_t M, int64_t n_heads, int64_t dim,
                     const double* pooled, int64_t n_pooled, const int64_t* row_pos, double scale,
                     double* scores, int64_t ld) {
  for (int64_t r = 0; r < M; ++r) {
    int64_t nb = qsa_oracle_visible_blocks(row_pos[r]);
    if (nb > n_pooled || nb > ld) return -1;
  }
  for (int64_t r = 0; r < M; ++r) {
    int64_t nb = qsa_oracle_visible_blocks(row_pos[r]);
    double* srow = scores + r * ld;
    int64_t b;
#pragma omp parallel for num_threads(g_threads) schedule(static)
    for (b = 0; b < nb; ++b) {
      double acc = 0.0;
      for (int64_t h = 0; h < n_heads; ++h) {
        double dot = 0.0;
        for (int64_t d = 0; d < dim; ++d)
          dot += load_elem(q_idx, q_dtype, (r * n_heads + h) * dim + d) * pooled[b * dim + d];
        acc += dot > 0.0 ? dot : 0.0;
      }
      srow[b] = scale * acc;
    }
    for (b = nb; b < ld; ++b) srow[b] = -INFINITY;
  }
  return 0;
}

typedef struct {
  double s;
  int32_t id;
} scored_block;

/* Order for selection: higher score first; equal scores, lower id first (R5). */
static int by_score_then_id(const void* pa, const void* pb) {
  const scored_block* a = (const scored_block*)pa;
  const scored_block* b = (const scored_block*)pb;
  if (a->s > b->s) return -1;
  if (a->s < b->s) return 1;
  return (a->id > b->id) - (a->id < b->id);
}

static int ascending_int(const void* pa, const void* pb) {
  int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
  return (a > b) - (a < b);
}

/*
 * Step 3, selection [QSA 02, 03]: per row, the min(top_k, nb(p_r)) best
 * blocks by (score descending, id ascending), found by a full sort of every
 * visible block.  Output ids ascending in sel[r][0 .. cnt[r]), -1 after.
 * tau[r] is the score of the last block kept when the budget binds
 * (nb > top_k), else -inf (every complete block kept, R4).
 * Scores of -0.0 compare equal to +0.0, as IEEE comparison does.
 */
int qsa_oracle_select(const double* scores, int64_t M, int64_t ld, const int64_t* row_pos,
                      int64_t top_k, int32_t* sel, int32_t* cnt, double* tau) {
  if (top_k < 1) return -1;
  for (int64_t r = 0; r < M; ++r) {
    int64_t nb = qsa_oracle_visible_blocks(row_pos[r]);
    if (nb > ld) return -1;
    scored_block* all = (scored_block*)malloc(sizeof(scored_block) * (size_t)(nb > 0 ? nb : 1));
    if (!all) return -2;
    for (int64_t b = 0; b < nb; ++b) {
      all[b].s = scores[r * ld + b];
      all[b].id = (int32_t)b;
    }
    qsort(all, (size_t)nb, sizeof(scored_block), by_score_then_id);
    int64_t k = nb < top_k ? nb : top_k;
    int32_t* out = sel + r * top_k;
    for (int64_t i = 0; i < k; ++i) out[i] = all[i].id;
    qsort(out, (size_t)k, sizeof(int32_t), ascending_int);
    for (int64_t i = k; i < top_k; ++i) out[i] = -1;
    cnt[r] = (int32_t)k;
    tau[r] = nb > top_k ? all[k - 1].s : -INFINITY;
    free(all);
  }
  return 0;
}

/*
 * The token rows R_r a query row attends to [QSA 02]: the 4 tokens of each
 * selected block plus the tail tokens 4*nb(p) .. p, kept only where
 * visible[t] != 0 (R8; visible == NULL keeps all).  Writes at most
 * 4*cnt + 3 token ids in ascending order of the selected list and returns
 * their number.
 */
int64_t qsa_oracle_row_tokens(int64_t p, const int32_t* sel_row, int32_t cnt, const uint8_t* visible,
                              int64_t* tokens) {
  int64_t n = 0;
  for (int32_t i = 0; i < cnt; ++i)
    for (int64_t j = 0; j < 4; ++j) {
      int64_t t = 4 * (int64_t)sel_row[i] + j;
      if (!visible || visible[t]) tokens[n++] = t;
    }
  for (int64_t t = 4 * qsa_oracle_visible_blocks(p); t <= p; ++t)
    if (!visible || visible[t]) tokens[n++] = t;
  return n;
}

/*
 * Step 4, exact softmax attention over R_r [QSA 02, 03], grouped-query:
 * head h reads KV head floor(h / (Hq/Hkv)) (R6).
 *   q   [M, Hq, D] stored values;  k, v [Hkv, L, D] stored values
 *   out [M, Hq, D] fp64;  lse [M, Hq] fp64 (natural log, R7)
 * For each (r, h): z_t = scale * q.k_t for t in R_r, m = max z,
 *   lse = m + log(sum exp(z_t - m)),  out = sum exp(z_t - lse) v_t.
 * An empty R_r gives out = 0, lse = -inf (R8).
 */
int qsa_oracle_attn(const void* q, int q_dtype, int64_t M, int64_t Hq, int64_t Hkv, int64_t D,
                    const void* k, const void* v, int kv_dtype, int64_t L, const uint8_t* visible,
                    const int64_t* row_pos, const int32_t* sel, const int32_t* cnt, int64_t sel_ld,
                    double scale, double* out, double* lse) {
  if (Hkv < 1 || Hq % Hkv != 0) return -1;
  int64_t group = Hq / Hkv;
  for (int64_t r = 0; r < M; ++r) {
    if (row_pos[r] < 0 || row_pos[r] >= L || cnt[r] < 0 || cnt[r] > sel_ld) return -1;
    for (int32_t i = 0; i < cnt[r]; ++i) {
      int64_t b = sel[r * sel_ld + i];
      if (b < 0 || b >= qsa_oracle_visible_blocks(row_pos[r])) return -1;
    }
  }
  int64_t rh;
#pragma omp parallel for num_threads(g_threads) schedule(dynamic, 1)
  for (rh = 0; rh < M * Hq; ++rh) {
    int64_t r = rh / Hq, h = rh % Hq, g = h / group;
    int64_t* tokens = (int64_t*)malloc(sizeof(int64_t) * (size_t)(4 * sel_ld + 4));
    double* z = (double*)malloc(sizeof(double) * (size_t)(4 * sel_ld + 4));
    int64_t n = qsa_oracle_row_tokens(row_pos[r], sel + r * sel_ld, cnt[r], visible, tokens);
    double* o = out + rh * D;
    for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
    if (n == 0) {
      lse[rh] = -INFINITY;
    } else {
      double m = -INFINITY;
      for (int64_t i = 0; i < n; ++i) {
        const int64_t kv_row = (g * L + tokens[i]) * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
          dot += load_elem(q, q_dtype, rh * D + d) * load_elem(k, kv_dtype, kv_row + d);
        z[i] = scale * dot;
        if (z[i] > m) m = z[i];
      }
      double sum = 0.0;
      for (int64_t i = 0; i < n; ++i) sum += exp(z[i] - m);
      double l = m + log(sum);
      for (int64_t i = 0; i < n; ++i) {
        const int64_t kv_row = (g * L + tokens[i]) * D;
        double w = exp(z[i] - l);
        for (int64_t d = 0; d < D; ++d) o[d] += w * load_elem(v, kv_dtype, kv_row + d);
      }
      lse[rh] = l;
    }
    free(tokens);
    free(z);
  }
  return 0;
}

/*
 * Step 5, log-sum-exp merge of partial attention results [SEG]:
 *   m = max_s lse_s,  w_s = exp(lse_s - m),
 *   out = sum_s w_s out_s / sum_s w_s,  lse = m + log(sum_s w_s).
 * When every lse_s is -inf the row saw no key: out = 0, lse = -inf.
 *   o_parts [S, R, D], lse_parts [S, R] (fp64);  out [R, D], lse [R]
 */
int qsa_oracle_lse_merge(const double* o_parts, const double* lse_parts, int64_t S, int64_t R, int64_t D,
                         double* out, double* lse) {
  if (S < 1) return -1;
  for (int64_t i = 0; i < R; ++i) {
    double m = -INFINITY;
    for (int64_t s = 0; s < S; ++s)
      if (lse_parts[s * R + i] > m) m = lse_parts[s * R + i];
    double* o = out + i * D;
    for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
    if (m == -INFINITY) {
      lse[i] = -INFINITY;
      continue;
    }
    double wsum = 0.0;
    for (int64_t s = 0; s < S; ++s) {
      double w = exp(lse_parts[s * R + i] - m);
      wsum += w;
      for (int64_t d = 0; d < D; ++d) o[d] += w * o_parts[(s * R + i) * D + d];
    }
    for (int64_t d = 0; d < D; ++d) o[d] /= wsum;
    lse[i] = m + log(wsum);
  }
  return 0;
}

/* ---------------------------------------------------------------- fp8 state (R9) */

/* Value of an E4M3 code (NaN for S.1111.111). */
double qsa_oracle_e4m3_decode(uint8_t c) {
  const int sign = c >> 7, e = (c >> 3) & 15, m = c & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0)
    v = ldexp((double)m, -9);               /* subnormal: m * 2^-9 */
  else
    v = ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -v : v;
}

/* Nearest E4M3 code to a finite x (ties to even), saturated at +-448. */
uint8_t qsa_oracle_e4m3_encode(double x) {
  const uint8_t sign = x < 0 || (x == 0 && signbit(x)) ? 0x80 : 0;
  double a = fabs(x);
  if (a >= 448.0) return sign | 0x7E;
  if (a < ldexp(1.0, -6)) {                 /* subnormal range: a multiple of 2^-9 */
    const double q = nearbyint(ldexp(a, 9)); /* 0 .. 8; 8 is the smallest normal */
    return sign | (uint8_t)q;
  }
  int e;
  frexp(a, &e);                              /* a = f * 2^e, f in [0.5, 1) */
  e -= 1;                                    /* a = (1 + t) * 2^e, t in [0, 1) */
  double mant = nearbyint((ldexp(a, -e) - 1.0) * 8.0);
  if (mant == 8.0) {
    mant = 0.0;
    e += 1;
  }
  if (e > 8 || (e == 8 && mant > 6.0)) return sign | 0x7E;
  return sign | (uint8_t)(((e + 7) << 3) | (int)mant);
}

/* binary16 bits -> double and double -> binary16 bits (nearest, ties to even). */
double qsa_oracle_f16_decode(uint16_t h) {
  const int sign = h >> 15, e = (h >> 10) & 31, m = h & 1023;
  double v;
  if (e == 31) v = m ? NAN : INFINITY;
  else if (e == 0) v = ldexp((double)m, -24);
  else v = ldexp(1.0 + m / 1024.0, e - 15);
  return sign ? -v : v;
}

uint16_t qsa_oracle_f16_encode(double x) {
  const uint16_t sign = signbit(x) ? 0x8000 : 0;
  double a = fabs(x);
  if (isnan(x)) return 0x7E00;
  if (a < ldexp(1.0, -14)) {                 /* subnormal: multiples of 2^-24 */
    const double q = nearbyint(ldexp(a, 24));
    return sign | (uint16_t)q;               /* q = 1024 is the smallest normal */
  }
  int e;
  frexp(a, &e);
  e -= 1;
  double mant = nearbyint((ldexp(a, -e) - 1.0) * 1024.0);
  if (mant == 1024.0) {
    mant = 0.0;
    e += 1;
  }
  if (e > 15) return sign | 0x7C00;          /* overflow to infinity */
  return sign | (uint16_t)(((e + 15) << 10) | (int)mant);
}

/*
 * Write rows of an fp8 state (R9): x [rows, D] in its stored format ->
 * codes [rows, D] and f16 scale bits [rows].  The scale and the quotient are
 * rounded to binary32 before their final rounding, as a GPU computes them.
 */
int qsa_oracle_fp8_quantize(const void* x, int dtype, int64_t rows, int64_t D, uint8_t* codes, uint16_t* scales) {
  for (int64_t r = 0; r < rows; ++r) {
    double amax = 0.0;
    for (int64_t d = 0; d < D; ++d) {
      const double a = fabs(load_elem(x, dtype, r * D + d));
      if (a > amax) amax = a;
    }
    const float s32 = (float)amax / 448.0f;          /* binary32 division (amax is exact in binary32) */
    const uint16_t sh = qsa_oracle_f16_encode((double)s32);
    scales[r] = sh;
    const float sc = (float)qsa_oracle_f16_decode(sh);
    for (int64_t d = 0; d < D; ++d) {
      if (sc == 0.0f) {
        codes[r * D + d] = 0;
        continue;
      }
      const float q = (float)load_elem(x, dtype, r * D + d) / sc;   /* binary32 quotient */
      codes[r * D + d] = qsa_oracle_e4m3_encode((double)q);
    }
  }
  return 0;
}

/* Stored fp8 rows back to values: out[r, d] = decode(codes[r, d]) * f16(scales[r]), exact in fp64. */
int qsa_oracle_fp8_dequantize(const uint8_t* codes, const uint16_t* scales, int64_t rows, int64_t D, double* out) {
  for (int64_t r = 0; r < rows; ++r) {
    const double sc = qsa_oracle_f16_decode(scales[r]);
    for (int64_t d = 0; d < D; ++d) out[r * D + d] = qsa_oracle_e4m3_decode(codes[r * D + d]) * sc;
  }
  return 0;
}

/* ---------------------------------------------------------------- q8 state (R10) */

int qsa_oracle_q8_quantize(const void* x, int dtype, int64_t rows, int64_t D, int8_t* codes, uint16_t* scales) {
  if (D % 32) return -1;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t b = 0; b < D / 32; ++b) {
      double amax = 0.0;
      for (int64_t d = 0; d < 32; ++d) {
        const double a = fabs(load_elem(x, dtype, r * D + 32 * b + d));
        if (a > amax) amax = a;
      }
      const float s32 = (float)amax / 127.0f;
      const uint16_t sh = qsa_oracle_f16_encode((double)s32);
      scales[r * (D / 32) + b] = sh;
      const float sc = (float)qsa_oracle_f16_decode(sh);
      for (int64_t d = 0; d < 32; ++d) {
        int8_t c = 0;
        if (sc != 0.0f) {
          const float q = (float)load_elem(x, dtype, r * D + 32 * b + d) / sc;
          double n = round((double)q);                     /* halves away from zero */
          if (n > 127.0) n = 127.0;
          if (n < -127.0) n = -127.0;
          c = (int8_t)n;
        }
        codes[r * D + 32 * b + d] = c;
      }
    }
  return 0;
}

int qsa_oracle_q8_dequantize(const int8_t* codes, const uint16_t* scales, int64_t rows, int64_t D, double* out) {
  if (D % 32) return -1;
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t d = 0; d < D; ++d)
      out[r * D + d] = (double)codes[r * D + d] * qsa_oracle_f16_decode(scales[r * (D / 32) + d / 32]);
  return 0;
}
