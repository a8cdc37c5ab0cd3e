/*
 * sl8 oracle: a plain, slow, obviously correct CPU definition of the W8A8 INT8
 * attention path.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the
 * benchmark's CPU-baseline leg call it; the library under w8a8_int8_flashattention_gb300/
 * never does, and shares no code with it.
 *
 * Sources (the "SuperL8" README, github.com/jajmangold/superl8):
 *   - "Supporting kernels" table, quant_rowwise row: symmetric per-row int8 quantisation.
 *   - "Quantization" table, "Per-row int8" row: symmetric, K-smoothing.
 *   - "Attention kernels" table, attn_int8_fwd row: W8A8 FlashAttention-2, causal, GQA/MQA,
 *     head dims 32/64/128/256; attn_varlen_fwd row: ragged prefill; attn_decode row:
 *     split-KV decode over an int8 KV cache with int8 V.
 *   - "Quick start" section: q [B,Hq,N,d], k/v [B,Hkv,N,d], attn_int8_fwd(q, k, v, causal=True),
 *     which quantises internally.
 * The pages name these operations but print no formula.  The readings taken here
 * (each one restated beside the code that takes it):
 *   R1  s = max|x| / 127 as an IEEE fp32 division; code = clamp(RNE(x / s), -127, 127).
 *   R3  a row whose s is 0 gets s = 0 and all-zero codes.
 *   R4  the K channel mean sums fp32 in fixed 64-token chunks, each in ascending token
 *       order, then the chunk sums in ascending order, then divides by the token count.
 *   R5  the mean runs over every token of the sequence; Q is not smoothed.
 *   R8  GQA maps query head hq to kv head hq / (Hq / Hkv).
 *   R9  causal is top-left aligned: key j is allowed for query i iff j <= i.
 *   R12 decode quantises q per (b, hq) row with R1/R3; V rows are s_v[t] * code.
 *   R13 split-KV uses contiguous chunks; an empty split has lse = -inf and weight 0.
 *   R21 attn_w8a8_fwd: Q and K scales shared by groups of consecutive rows, Q outliers
 *       keep their own scale (restated at oracle_quant_groups).
 * Everything after the int32 dot runs in fp64: logits, softmax, P.V and the LSE.
 *
 * Build: gcc -O2 -std=c11 -fopenmp -ffp-contract=off (no -ffast-math): every fp32
 * operation below rounds once, as written.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_MEAN_CHUNK 64

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ---------------------------------------------------------------- quantisation */

/* One row of d values, optionally smoothed by mu (fp32 subtraction), quantised
 * per R1/R3.  Writes d codes and one scale. */
static void quant_row(const float* x, const float* mu, int d, int8_t* codes, float* scale) {
  float a = 0.0f;
  for (int c = 0; c < d; ++c) {
    float r = mu ? x[c] - mu[c] : x[c];
    float m = fabsf(r);
    if (m > a) a = m;
  }
  float s = a / 127.0f;
  *scale = s;
  for (int c = 0; c < d; ++c) {
    if (s == 0.0f) {
      codes[c] = 0;
      continue;
    }
    float r = mu ? x[c] - mu[c] : x[c];
    float t = r / s;
    float n = nearbyintf(t); /* round half to even in the default rounding mode */
    if (n > 127.0f) n = 127.0f;
    if (n < -127.0f) n = -127.0f;
    codes[c] = (int8_t)n;
  }
}

/* rows x d contiguous fp32; mu (nullable) is [groups][d], row r uses group r / rows_per_group. */
void oracle_quant_rows(const float* x, int64_t rows, int d, const float* mu, int64_t rows_per_group,
                       int8_t* codes, float* scales) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < rows; ++r) {
    const float* m = mu ? mu + (r / rows_per_group) * (int64_t)d : NULL;
    quant_row(x + r * (int64_t)d, m, d, codes + r * (int64_t)d, scales + r);
  }
}

/* ---------------------------------------------------------------- grouped quantisation */

static int cmp_float(const void* a, const void* b) {
  float x = *(const float*)a, y = *(const float*)b;
  return (x > y) - (x < y);
}

/*
 * "Attention kernels" table, attn_w8a8_fwd row (a W8A8 forward whose scales are set per
 * warp and which takes outliers into account), and the "Quantization" table's per-row
 * int8 row, which lists outlier detection for Q.  The pages give no formula, so this is
 * reading R21:
 *   - the n rows (one sequence and head, in token order, optionally smoothed by mu)
 *     form groups of `group` consecutive rows starting at row 0 (the last group may be
 *     shorter); a = max|x| of each row (fp32, exact);
 *   - with tau > 0 a row is an outlier when a > tau * med (one fp32 product), med the
 *     lower median of its group's a values (element (cnt - 1) / 2 of the ascending
 *     sort); an outlier keeps its own scale a / 127;
 *   - every other row of the group takes s = (max a over the group's non-outliers) / 127,
 *     an IEEE fp32 division, and its codes clamp(RNE(x / s), -127, 127) (R1, R3).
 * group = 1 is the per-row quantiser.  outlier (nullable) receives one flag per row.
 */
void oracle_quant_groups(const float* x, int64_t n, int d, const float* mu, int64_t group, float tau,
                         int8_t* codes, float* scales, uint8_t* outlier) {
  for (int64_t g0 = 0; g0 < n; g0 += group) {
    int64_t g1 = g0 + group < n ? g0 + group : n, cnt = g1 - g0;
    float* a = (float*)malloc((size_t)cnt * sizeof(float));
    float* sorted = (float*)malloc((size_t)cnt * sizeof(float));
    uint8_t* out = (uint8_t*)calloc((size_t)cnt, 1);
    for (int64_t r = g0; r < g1; ++r) {
      float m = 0.0f;
      for (int c = 0; c < d; ++c) {
        float v = mu ? x[r * (int64_t)d + c] - mu[c] : x[r * (int64_t)d + c];
        if (fabsf(v) > m) m = fabsf(v);
      }
      a[r - g0] = m;
    }
    if (tau > 0.0f) {
      memcpy(sorted, a, (size_t)cnt * sizeof(float));
      qsort(sorted, (size_t)cnt, sizeof(float), cmp_float);
      float thr = tau * sorted[(cnt - 1) / 2];
      for (int64_t i = 0; i < cnt; ++i) out[i] = a[i] > thr;
    }
    float inlier_max = 0.0f;
    for (int64_t i = 0; i < cnt; ++i)
      if (!out[i] && a[i] > inlier_max) inlier_max = a[i];
    for (int64_t r = g0; r < g1; ++r) {
      float s = (out[r - g0] ? a[r - g0] : inlier_max) / 127.0f;
      scales[r] = s;
      if (outlier) outlier[r] = out[r - g0];
      for (int c = 0; c < d; ++c) {
        float v = mu ? x[r * (int64_t)d + c] - mu[c] : x[r * (int64_t)d + c];
        float t = s == 0.0f ? 0.0f : v / s;
        float q = nearbyintf(t);
        if (q > 127.0f) q = 127.0f;
        if (q < -127.0f) q = -127.0f;
        codes[r * (int64_t)d + c] = (int8_t)q;
      }
    }
    free(a);
    free(sorted);
    free(out);
  }
}

/* ---------------------------------------------------------------- K smoothing */

/* Per-channel mean of n token rows (row t starts at k + t * tok_stride), order R4. */
void oracle_k_mean(const float* k, int64_t n, int64_t tok_stride, int d, float* mu) {
  for (int c = 0; c < d; ++c) {
    float total = 0.0f;
    for (int64_t t0 = 0; t0 < n; t0 += ORACLE_MEAN_CHUNK) {
      int64_t t1 = t0 + ORACLE_MEAN_CHUNK < n ? t0 + ORACLE_MEAN_CHUNK : n;
      float part = 0.0f;
      for (int64_t t = t0; t < t1; ++t) part += k[t * tok_stride + c];
      total += part;
    }
    mu[c] = n > 0 ? total / (float)n : 0.0f;
  }
}

/* ---------------------------------------------------------------- attention */

static int64_t dot_i8(const int8_t* a, const int8_t* b, int d) {
  int64_t s = 0;
  for (int c = 0; c < d; ++c) s += (int64_t)a[c] * (int64_t)b[c];
  return s;
}

/* Softmax attention of one quantised query row against keys [0, n), fp64 after the
 * int32 dot.  v rows are v[t*v_stride + c] * (v_scale ? v_scale[t] : 1).  With n == 0
 * the output is 0 and lse = -inf.  logits (nullable) receives the n int32 dots. */
static void attn_row(const int8_t* qc, float qs, const int8_t* kc, const float* ks, const float* v,
                     const float* v_scale, int64_t n, int d, double* o, double* lse,
                     int32_t* logits, int* overflow) {
  double inv_sqrt_d = 1.0 / sqrt((double)d);
  double* x = (double*)malloc((size_t)(n > 0 ? n : 1) * sizeof(double));
  double m = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    int64_t s = dot_i8(qc, kc + j * (int64_t)d, d);
    if (s > INT32_MAX || s < INT32_MIN) *overflow = 1;
    if (logits) logits[j] = (int32_t)s;
    x[j] = (double)s * (double)qs * (double)ks[j] * inv_sqrt_d;
    if (x[j] > m) m = x[j];
  }
  for (int c = 0; c < d; ++c) o[c] = 0.0;
  double l = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    double p = exp(x[j] - m);
    l += p;
    double w = v_scale ? p * (double)v_scale[j] : p;
    const float* vr = v + j * (int64_t)d;
    for (int c = 0; c < d; ++c) o[c] += w * (double)vr[c];
  }
  if (n > 0) {
    for (int c = 0; c < d; ++c) o[c] /= l;
    *lse = m + log(l);
  } else {
    *lse = -INFINITY;
  }
  free(x);
}

/*
 * Prefill attention for one (sequence, query head): nq query rows and nk key rows of
 * one kv head, all already quantised (codes [rows][d] int8, scales [rows]).  v is
 * [nk][d] fp32 (the widened bf16/fp16 input).  Query i (0-based within the query
 * rows) sees keys j < nk, and j <= i + q_off when causal: q_off = 0 is the top-left
 * alignment of a self-attention prefill (R9); q_off = nk - nq aligns the nq queries
 * with the last nq keys (bottom-right, a chunk of a longer sequence, R19).
 * rows (nullable) lists the query rows to compute (nrows of them); NULL means all nq.
 * Outputs are per listed row: o [nrows][d], lse [nrows], logits [nrows][nk] (nullable;
 * entries for keys a row may not see are left untouched).
 * Returns 0, or 1 if some int32 dot overflowed (cannot happen for d <= 256).
 */
int oracle_attn_prefill_head(const int8_t* qc, const float* qs, const int8_t* kc, const float* ks,
                             const float* v, int64_t nq, int64_t nk, int d, int causal, int64_t q_off,
                             const int64_t* rows, int64_t nrows, double* o, double* lse,
                             int32_t* logits) {
  int overflow = 0;
  if (!rows) nrows = nq;
#pragma omp parallel for schedule(dynamic, 4) reduction(| : overflow)
  for (int64_t r = 0; r < nrows; ++r) {
    int64_t i = rows ? rows[r] : r;
    int64_t n = nk;
    if (causal && i + 1 + q_off < n) n = i + 1 + q_off;
    int ov = 0;
    attn_row(qc + i * (int64_t)d, qs[i], kc, ks, v, NULL, n, d, o + r * (int64_t)d, lse + r,
             logits ? logits + r * nk : NULL, &ov);
    overflow |= ov;
  }
  return overflow;
}

/*
 * Decode for one (b, hq): a quantised query row against the first L rows of one kv
 * head's int8 cache (k codes/scales, v codes/scales), restricted to the key range
 * [t0, t1) ∩ [0, L).  With t0 = 0, t1 >= L this is the whole decode (R12); a proper
 * sub-range gives one split-KV partial (R13), whose normalised O and lse feed
 * oracle_decode_combine.  An empty range gives O = 0, lse = -inf.
 */
int oracle_decode_row(const int8_t* qc, float qs, const int8_t* kc, const float* ks,
                      const int8_t* vc, const float* vs, int64_t L, int64_t t0, int64_t t1, int d,
                      double* o, double* lse, int32_t* logits) {
  if (t1 > L) t1 = L;
  if (t0 < 0) t0 = 0;
  int64_t n = t1 > t0 ? t1 - t0 : 0;
  float* vf = (float*)malloc((size_t)(n > 0 ? n : 1) * (size_t)d * sizeof(float));
  for (int64_t j = 0; j < n; ++j)
    for (int c = 0; c < d; ++c) vf[j * (int64_t)d + c] = (float)vc[(t0 + j) * (int64_t)d + c];
  int overflow = 0;
  attn_row(qc, qs, kc + t0 * (int64_t)d, ks + t0, vf, vs + t0, n, d, o, lse, logits, &overflow);
  free(vf);
  return overflow;
}

/*
 * Decode for one (b, hq) over a cache whose V is kept in fp16: the attn_decode "fp16 V"
 * variant.  As oracle_decode_row, but the V rows v [L][d] are the fp16 values widened to
 * fp32 (exact) and carry no per-token scale: O = sum_t p_t * v[t].
 */
int oracle_decode_row_fv(const int8_t* qc, float qs, const int8_t* kc, const float* ks, const float* v,
                         int64_t L, int64_t t0, int64_t t1, int d, double* o, double* lse, int32_t* logits) {
  if (t1 > L) t1 = L;
  if (t0 < 0) t0 = 0;
  int64_t n = t1 > t0 ? t1 - t0 : 0;
  int overflow = 0;
  attn_row(qc, qs, kc + t0 * (int64_t)d, ks + t0, v + t0 * (int64_t)d, NULL, n, d, o, lse, logits, &overflow);
  return overflow;
}

/* Merge nsplit partials (o [nsplit][d] normalised, lse [nsplit]) into one row, R13. */
void oracle_decode_combine(const double* o, const double* lse, int nsplit, int d, double* out,
                           double* lse_out) {
  double m = -INFINITY;
  for (int s = 0; s < nsplit; ++s)
    if (lse[s] > m) m = lse[s];
  for (int c = 0; c < d; ++c) out[c] = 0.0;
  if (m == -INFINITY) {
    *lse_out = -INFINITY;
    return;
  }
  double wsum = 0.0;
  for (int s = 0; s < nsplit; ++s) {
    double w = lse[s] == -INFINITY ? 0.0 : exp(lse[s] - m);
    wsum += w;
    for (int c = 0; c < d; ++c) out[c] += w * o[(int64_t)s * d + c];
  }
  for (int c = 0; c < d; ++c) out[c] /= wsum;
  *lse_out = m + log(wsum);
}
