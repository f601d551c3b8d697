/*
 * Reference (oracle) for paged FP8 MLA decode: plain, slow, fp64 CPU code.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code,
 * header, table or constant generator with the CUDA path.
 *
 * What it computes (the plain definition; the split-KV method reaches the same
 * result up to rounding because it is an exact refactoring of softmax):
 *
 *   Geometry, from "CuTe DSL FP8 MLA decode regression" (TensorRT-LLM issue
 *   #20510, section "Setup"): each KV row is 576 E4M3 values, 512 latent + 64
 *   rope; K is the whole row and V is its first 512 values (same issue,
 *   "Analysis": the V operand is the latent part of the rows K already read).
 *   Page size 32: token j of request b sits in slot j % 32 of page
 *   page_table[b][j / 32].
 *
 *   For query row (b, qi, h):
 *     q   = q_scale  * dec(Q[b][qi][h][0:576])
 *     k_j = kv_scale * dec(KV row of token j),   v_j = k_j[0:512]
 *     n   = L_b - q_len + qi + 1 if causal (MTP verify: query token i sees keys
 *           [0, L - q_len + i], inclusive), else L_b
 *     s_j = softmax_scale * (q . k_j),           j < n
 *     M = max_j s_j,  Z = sum_j exp(s_j - M)
 *     O = sum_j exp(s_j - M) v_j / Z,  LSE = M + ln Z   (natural log)
 *
 *   dec() is the exact E4M3 ("FN", no infinities) decode: sign s, 4-bit
 *   exponent e with bias 7, 3-bit mantissa m; e == 0 is subnormal m/8 * 2^-6;
 *   e == 15 && m == 7 is NaN; otherwise (1 + m/8) * 2^(e-7).
 *
 *   Partials: for a key range, (m, l, O) with m = max_j s_j * log2(e) (log2
 *   units), l = sum_j 2^(t_j - m), O = sum_j 2^(t_j - m) v_j, t_j = s_j log2(e);
 *   an empty range gives (-inf, 0, 0).  The merge ("fmhaReductionKernel",
 *   TensorRT-LLM PR #20380, "Description"): M = max_s m_s,
 *   w_s = 2^(m_s - M), O = sum_s w_s O_s / sum_s w_s l_s,
 *   LSE = ln 2 * (M + log2 sum_s w_s l_s); empty partials contribute nothing.
 *
 * Two passes over stored scores per row; no online rescaling, no blocking.
 *
 * KV append (the step that fills the paged cache; TensorRT-LLM PR #17273,
 * "Fuse the DSv4 MLA prologue": a latent row is quantized to FP8 and scattered
 * into the paged cache): each new 576-value row x of request b at token
 * position j is stored as code = e4m3(x / kv_scale) in slot j % 32 of page
 * page_table[b][j / 32].  The division is IEEE fp32 (the precision the
 * quantised code is decided in on the device); e4m3() is the nearest E4M3
 * value, ties to the even code, magnitudes beyond 448 saturate to 448, NaN
 * stays NaN.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_HEAD_DIM 576
#define ORC_LATENT_DIM 512
#define ORC_PAGE 32

/* Exact E4M3 decode from its bit fields. */
double mla_oracle_e4m3_decode(uint8_t code) {
  int sign = (code >> 7) & 1;
  int e = (code >> 3) & 15;
  int m = code & 7;
  double v;
  if (e == 15 && m == 7) return NAN;
  if (e == 0) {
    v = ldexp((double)m / 8.0, -6);
  } else {
    v = ldexp(1.0 + (double)m / 8.0, e - 7);
  }
  return sign ? -v : v;
}

static void build_lut(double lut[256]) {
  for (int c = 0; c < 256; ++c) lut[c] = mla_oracle_e4m3_decode((uint8_t)c);
}

int mla_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Visible key range of one row, intersected with [tok_begin, tok_end). */
static void row_range(int32_t L, int32_t q_len, int32_t qi, int32_t causal,
                      int64_t tok_begin, int64_t tok_end, int64_t* lo, int64_t* hi) {
  int64_t n = causal ? (int64_t)L - q_len + qi + 1 : (int64_t)L;
  if (n < 0) n = 0;
  int64_t a = tok_begin < 0 ? 0 : tok_begin;
  int64_t b = (tok_end < 0 || tok_end > n) ? n : tok_end;
  if (b < a) b = a;
  *lo = a;
  *hi = b;
}

/* Value d of the 576-value row at element index `row` of an array of
 * element type dtype: 0 = E4M3 codes (uint8), 1 = BF16 bit patterns (uint16,
 * widened exactly: the 16 bits are the top half of an IEEE float). */
static double elem(const void* base, int dtype, int64_t row, int d, const double lut[256]) {
  if (dtype == 0) return lut[((const uint8_t*)base)[row * ORC_HEAD_DIM + d]];
  uint32_t bits = (uint32_t)((const uint16_t*)base)[row * ORC_HEAD_DIM + d] << 16;
  float f;
  memcpy(&f, &bits, sizeof(f));
  return (double)f;
}

static int64_t key_index(const int32_t* page_table, int32_t max_pages, int32_t b, int64_t j) {
  int64_t page = page_table[(int64_t)b * max_pages + j / ORC_PAGE];
  return page * ORC_PAGE + (j % ORC_PAGE);
}

/*
 * Decode rows.  rows[i] is the flat row id (b*q_len + qi)*num_heads + h.
 * Keys are restricted to [tok_begin, tok_end) when those are >= 0.
 * mode 0: final outputs: out[i][512] = O, lse[i] = LSE (natural log);
 *         an empty row gives O = 0, LSE = -inf.
 * mode 1: partials: out[i][512] = unnormalised O, m_out[i] = m (log2 units),
 *         l_out[i] = l.
 * Returns 0, or -1 on an out-of-range page id, -2 on allocation failure.
 */
int mla_oracle_decode_rows_v2(const void* q, const void* kv, int32_t dtype, int64_t num_pages,
                              const int32_t* page_table, int32_t max_pages,
                              const int32_t* kv_lens, int32_t batch, int32_t q_len,
                              int32_t num_heads, int32_t causal, double q_scale,
                              double kv_scale, double softmax_scale, const double* sinks,
                              double output_scale, const int32_t* query_lens,
                              const int32_t* kv_bounds, const int32_t* block_idx, int32_t topk,
                              const int64_t* rows, int64_t n_rows, int64_t tok_begin,
                              int64_t tok_end, int32_t mode, double* out, double* lse,
                              double* m_out, double* l_out, int32_t n_threads);
int mla_oracle_decode_rows_ex(const void* q, const void* kv, int32_t dtype, int64_t num_pages,
                              const int32_t* page_table, int32_t max_pages,
                              const int32_t* kv_lens, int32_t batch, int32_t q_len,
                              int32_t num_heads, int32_t causal, double q_scale,
                              double kv_scale, double softmax_scale, const double* sinks,
                              double output_scale, const int64_t* rows, int64_t n_rows,
                              int64_t tok_begin, int64_t tok_end, int32_t mode, double* out,
                              double* lse, double* m_out, double* l_out, int32_t n_threads);

int mla_oracle_decode_rows(const uint8_t* q, const uint8_t* kv, int64_t num_pages,
                           const int32_t* page_table, int32_t max_pages,
                           const int32_t* kv_lens, int32_t batch, int32_t q_len,
                           int32_t num_heads, int32_t causal, double q_scale,
                           double kv_scale, double softmax_scale, const int64_t* rows,
                           int64_t n_rows, int64_t tok_begin, int64_t tok_end, int32_t mode,
                           double* out, double* lse, double* m_out, double* l_out,
                           int32_t n_threads) {
  return mla_oracle_decode_rows_ex(q, kv, 0, num_pages, page_table, max_pages, kv_lens, batch,
                                   q_len, num_heads, causal, q_scale, kv_scale, softmax_scale,
                                   NULL, 1.0, rows, n_rows, tok_begin, tok_end, mode, out, lse,
                                   m_out, l_out, n_threads);
}

/*
 * Same, with per-head attention sinks, an output scale, and the element type
 * of Q and KV (dtype 0: E4M3 codes; 1: BF16, the pages' BF16-KV kernel,
 * issue #20510 "Repro 2" comparison, same geometry).  A sink is a
 * virtual key of logit sinks[h] (natural-log units, compared with the scaled
 * scores s_j) and zero value: Z gains exp(sink - M), O shrinks accordingly,
 * LSE = ln(sum_j exp(s_j) + exp(sink)).  output_scale multiplies O only.
 * Sinks and output_scale apply to mode 0 (final outputs) only.
 */
int mla_oracle_decode_rows_ex(const void* q, const void* kv, int32_t dtype, int64_t num_pages,
                              const int32_t* page_table, int32_t max_pages,
                              const int32_t* kv_lens, int32_t batch, int32_t q_len,
                              int32_t num_heads, int32_t causal, double q_scale,
                              double kv_scale, double softmax_scale, const double* sinks,
                              double output_scale, const int64_t* rows, int64_t n_rows,
                              int64_t tok_begin, int64_t tok_end, int32_t mode, double* out,
                              double* lse, double* m_out, double* l_out, int32_t n_threads) {
  return mla_oracle_decode_rows_v2(q, kv, dtype, num_pages, page_table, max_pages, kv_lens, batch,
                                   q_len, num_heads, causal, q_scale, kv_scale, softmax_scale,
                                   sinks, output_scale, NULL, NULL, NULL, 0, rows, n_rows,
                                   tok_begin, tok_end, mode, out, lse, m_out, l_out, n_threads);
}

/*
 * The general form: mla_oracle_decode_rows_ex plus three restrictions of the
 * visible keys: the run() arguments is_var_q/query_lens and kv_bounds (issue
 * #20510, "Repro 1", arguments added after #19338), and the sparse decode over
 * selected pages (TensorRT-LLM PR #17441 "m3 decode perf": the sparse decode
 * kernel after the block selector, with E4M3 q widened inside the kernel).
 * The pages name these arguments without defining them; the readings are:
 *
 *   query_lens (int32 [B] or NULL): request b has q_b = query_lens[b] query
 *     tokens, 1 <= q_b <= q_len, in slots qi < q_b of the padded
 *     [B][q_len][H] row layout.  They are the last q_b positions of the
 *     request, so under causal query qi sees keys j <= L_b - q_b + qi.  Rows
 *     with qi >= q_b see no key (O = 0, LSE = -inf, or the sink).
 *   kv_bounds (int32 [B][2] or NULL): keys restricted to lo <= j < hi with
 *     (lo, hi) = kv_bounds[b] (a window of the request's keys).
 *   block_idx (int32 [B][topk] or NULL): keys restricted to the request's
 *     logical pages listed in block_idx[b] (page p holds keys [32p, 32p+32));
 *     negative entries are unused slots.  A page listed twice counts once.
 *
 * All restrictions intersect the causal range and [0, L_b).
 */
int mla_oracle_decode_rows_v2(const void* q, const void* kv, int32_t dtype, int64_t num_pages,
                              const int32_t* page_table, int32_t max_pages,
                              const int32_t* kv_lens, int32_t batch, int32_t q_len,
                              int32_t num_heads, int32_t causal, double q_scale,
                              double kv_scale, double softmax_scale, const double* sinks,
                              double output_scale, const int32_t* query_lens,
                              const int32_t* kv_bounds, const int32_t* block_idx, int32_t topk,
                              const int64_t* rows, int64_t n_rows, int64_t tok_begin,
                              int64_t tok_end, int32_t mode, double* out, double* lse,
                              double* m_out, double* l_out, int32_t n_threads) {
  double lut[256];
  int status = 0;
  build_lut(lut);
  (void)batch;
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
#else
  (void)n_threads;
#endif

#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < n_rows; ++i) {
    int64_t r = rows[i];
    int32_t h = (int32_t)(r % num_heads);
    int32_t qi = (int32_t)((r / num_heads) % q_len);
    int32_t b = (int32_t)(r / ((int64_t)num_heads * q_len));
    double qd[ORC_HEAD_DIM];
    double* o = out + i * ORC_LATENT_DIM;
    int64_t lo, hi;
    for (int d = 0; d < ORC_HEAD_DIM; ++d) qd[d] = q_scale * elem(q, dtype, r, d, lut);
    const int32_t qb = query_lens ? query_lens[b] : q_len;
    row_range(kv_lens[b], qb, qi, causal, tok_begin, tok_end, &lo, &hi);
    if (qi >= qb) hi = lo;  /* a padding slot of a shorter query block */
    if (kv_bounds) {
      if (lo < kv_bounds[2 * b]) lo = kv_bounds[2 * b];
      if (hi > kv_bounds[2 * b + 1]) hi = kv_bounds[2 * b + 1];
      if (hi < lo) hi = lo;
    }
    for (int d = 0; d < ORC_LATENT_DIM; ++d) o[d] = 0.0;
    const double sink = (sinks && mode == 0) ? sinks[h] : -INFINITY;
    /* Selected pages of this request (all pages when there is no selection). */
    unsigned char* sel = NULL;
    if (block_idx && hi > lo) {
      sel = (unsigned char*)calloc((size_t)max_pages, 1);
      if (!sel) {
#pragma omp atomic write
        status = -2;
        continue;
      }
      for (int32_t t = 0; t < topk; ++t) {
        int32_t pg = block_idx[(int64_t)b * topk + t];
        if (pg >= 0 && pg < max_pages) sel[pg] = 1;
      }
    }
    int64_t n_vis = 0;
    for (int64_t j = lo; j < hi; ++j) n_vis += (!sel || sel[j / ORC_PAGE]) ? 1 : 0;
    if (n_vis == 0) {
      free(sel);
      if (mode == 0) {
        lse[i] = sink;
      } else {
        m_out[i] = -INFINITY;
        l_out[i] = 0.0;
      }
      continue;
    }
    double* s = (double*)malloc(sizeof(double) * (size_t)(hi - lo));
    if (!s) {
      free(sel);
#pragma omp atomic write
      status = -2;
      continue;
    }
    int bad = 0;
    /* Pass 1: scores (keys outside the selection are not visible: -inf). */
    for (int64_t j = lo; j < hi; ++j) {
      if (sel && !sel[j / ORC_PAGE]) {
        s[j - lo] = -INFINITY;
        continue;
      }
      int64_t page = page_table[(int64_t)b * max_pages + j / ORC_PAGE];
      if (page < 0 || page >= num_pages) {
        bad = 1;
        s[j - lo] = 0.0;
        continue;
      }
      const int64_t kr = key_index(page_table, max_pages, b, j);
      double dot = 0.0;
      for (int d = 0; d < ORC_HEAD_DIM; ++d) dot += qd[d] * (kv_scale * elem(kv, dtype, kr, d, lut));
      s[j - lo] = softmax_scale * dot;
    }
    double M = sink;
    for (int64_t j = lo; j < hi; ++j)
      if (s[j - lo] > M) M = s[j - lo];
    /* Pass 2: weights and the weighted sum of values (the sink adds weight
       and no value). */
    double Z = (sink == -INFINITY) ? 0.0 : exp(sink - M);
    for (int64_t j = lo; j < hi; ++j) {
      if (sel && !sel[j / ORC_PAGE]) continue;
      double w = exp(s[j - lo] - M);
      int64_t page = page_table[(int64_t)b * max_pages + j / ORC_PAGE];
      Z += w;
      if (page < 0 || page >= num_pages) continue;
      const int64_t kr = key_index(page_table, max_pages, b, j);
      for (int d = 0; d < ORC_LATENT_DIM; ++d) o[d] += w * (kv_scale * elem(kv, dtype, kr, d, lut));
    }
    free(s);
    free(sel);
    if (bad) {
#pragma omp atomic write
      status = -1;
    }
    if (mode == 0) {
      for (int d = 0; d < ORC_LATENT_DIM; ++d) o[d] = output_scale * (o[d] / Z);
      lse[i] = M + log(Z);
    } else {
      m_out[i] = M * (1.0 / log(2.0));
      l_out[i] = Z;
    }
  }
  return status;
}

/*
 * Merge split partials (closed form).  ml: [rows][S][2] = (m, l);
 * o: [rows][S][512]; fp64 throughout (float32 partials widen exactly).
 * An empty slot (l == 0 or m == -inf) is skipped.  A row with no non-empty
 * slot gives O = 0 and LSE = -inf.
 */
void mla_oracle_merge(const double* ml, const double* o, int64_t rows, int32_t S, double* out,
                      double* lse) {
  for (int64_t r = 0; r < rows; ++r) {
    double M = -INFINITY;
    for (int32_t s = 0; s < S; ++s) {
      double m = ml[(r * S + s) * 2 + 0];
      double l = ml[(r * S + s) * 2 + 1];
      if (l > 0.0 && m > M) M = m;
    }
    double* dst = out + r * ORC_LATENT_DIM;
    for (int d = 0; d < ORC_LATENT_DIM; ++d) dst[d] = 0.0;
    if (M == -INFINITY) {
      lse[r] = -INFINITY;
      continue;
    }
    double den = 0.0;
    for (int32_t s = 0; s < S; ++s) {
      double m = ml[(r * S + s) * 2 + 0];
      double l = ml[(r * S + s) * 2 + 1];
      if (!(l > 0.0) || m == -INFINITY) continue;
      double w = exp2(m - M);
      den += w * l;
      const double* src = o + (r * S + s) * ORC_LATENT_DIM;
      for (int d = 0; d < ORC_LATENT_DIM; ++d) dst[d] += w * src[d];
    }
    for (int d = 0; d < ORC_LATENT_DIM; ++d) dst[d] /= den;
    lse[r] = log(2.0) * (M + log2(den));
  }
}

/* Nearest E4M3 code to v (ties to even), saturating at +-448; NaN -> 0x7F. */
uint8_t mla_oracle_e4m3_encode(float v) {
  double lut[256];
  build_lut(lut);
  if (v != v) return 0x7F;
  double x = (double)v;
  int neg = signbit(v) ? 1 : 0;
  double a = neg ? -x : x;
  if (a >= 448.0) return (uint8_t)(neg ? 0xFE : 0x7E);
  /* Positive codes 0x00..0x7E are increasing in value. */
  int best = 0;
  for (int c = 0; c <= 0x7E; ++c) {
    double d = fabs(lut[c] - a), db = fabs(lut[best] - a);
    if (d < db || (d == db && (c & 1) == 0 && (best & 1) == 1)) best = c;
  }
  return (uint8_t)(neg ? (best | 0x80) : best);
}

/* Append: rows[n][576] are bf16 bit patterns (widened exactly to float). */
int mla_oracle_kv_append(const uint16_t* rows_bf16, int64_t n, const int32_t* req,
                         const int32_t* pos, const int32_t* page_table, int32_t max_pages,
                         int32_t batch, uint8_t* kv, int64_t num_pages, float kv_scale) {
  int status = 0;
  for (int64_t i = 0; i < n; ++i) {
    int32_t b = req[i], j = pos[i];
    if (b < 0 || b >= batch || j < 0 || j / ORC_PAGE >= max_pages) {
      status = -1;
      continue;
    }
    int64_t page = page_table[(int64_t)b * max_pages + j / ORC_PAGE];
    if (page < 0 || page >= num_pages) {
      status = -1;
      continue;
    }
    uint8_t* dst = kv + (page * ORC_PAGE + j % ORC_PAGE) * ORC_HEAD_DIM;
    for (int d = 0; d < ORC_HEAD_DIM; ++d) {
      uint32_t bits = (uint32_t)rows_bf16[i * ORC_HEAD_DIM + d] << 16;
      float x;
      memcpy(&x, &bits, sizeof(x));
      volatile float q = x / kv_scale; /* IEEE fp32 division */
      dst[d] = mla_oracle_e4m3_encode(q);
    }
  }
  return status;
}
