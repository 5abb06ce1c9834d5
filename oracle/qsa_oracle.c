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
