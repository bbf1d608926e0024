/*
 * oracle.c -- plain, slow CPU oracle for the FP4 paged-MQA indexer prefill.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the tests, the smoke check and the benchmark's
 * CPU-baseline leg do.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes (method: "[FlyDSL] Add FP4 LiteTopK prefill operator",
 * ROCm/aiter#5309, Summary and Implementation; "[FlyDSL][DSv4] Prototype FP4
 * MQA streaming TopK", ROCm/aiter#5282, Changes and Scope):
 *
 *   logit[r,h,s] = sum_d q[r,h,d] * k[s,d]         exact (FP4 E2M1 x UE8M0)
 *   score[r,s]   = sum_{h=0..63} w[r,h] * max(logit[r,h,s], 0)   in float64,
 *                  heads in ascending order starting from +0.0
 *   out_raw[r]   = the topk window positions of row r under the total order
 *                  (score descending, logical index ascending; NaN below every
 *                  number; +0 above -0), or start..end-1 padded with -1 when
 *                  the window is not longer than topk (short-row contract,
 *                  aiter#5282 Changes);
 *   out_phys[r]  = page_table[req][raw / 64] * 64 + raw % 64, -1 stays -1
 *                  (aiter#5282 Changes: the raw C4 positions become physical
 *                  slots through the page table).
 *
 * Data formats: E2M1 as in the OCP Microscaling Formats (MX) v1.0 spec
 * (1 sign, 2 exponent bits with bias 1, 1 mantissa bit), two codes per byte
 * with the even element of D in the low nibble; UE8M0 scale byte e means
 * 2^(e-127), one per 32 consecutive elements of D; 255 is NaN and is outside
 * the input contract.
 *
 * Each per-head dot is computed exactly: per 32-element block the integer sum
 * of products in units of 1/4, then the blocks are brought to a common power
 * of two in 128-bit integers.  Every dot is reported together with whether it
 * is exactly representable in fp32.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define NH 64          /* heads */
#define ND 128         /* head dimension */
#define NPAGE 64       /* slots per page */
#define NDB (ND / 2)   /* bytes per head row / slot row */
#define NSF (ND / 32)  /* scale bytes per head row / slot row */

/* E2M1 magnitudes in units of 1/2: codes 0..7 are 0, 0.5, 1, 1.5, 2, 3, 4, 6;
 * bit 3 is the sign. */
static const int e2m1_half_units[16] = {0, 1, 2, 3, 4, 6, 8, 12,
                                        0, -1, -2, -3, -4, -6, -8, -12};

int oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

double oracle_e2m1_value(int code) {
  code &= 15;
  if (code == 8) return -0.0;
  return 0.5 * (double)e2m1_half_units[code];
}

double oracle_ue8m0_value(int byte) {
  if (byte == 255) return NAN;
  return ldexp(1.0, byte - 127);
}

/* Decoded operand row: 128 codes in half units and 4 block exponents. */
typedef struct {
  int8_t v[ND];
  int e[NSF];
} row_t;

static void decode_row(const uint8_t* bytes, const uint8_t* scales, row_t* out) {
  for (int d = 0; d < ND; ++d) {
    int code = (bytes[d / 2] >> (4 * (d & 1))) & 15;
    out->v[d] = (int8_t)e2m1_half_units[code];
  }
  for (int b = 0; b < NSF; ++b) out->e[b] = (int)scales[b];
}

/* Exact dot of two decoded rows.  Returns the value as a double (exact when
 * *dbl_exact is 1) and sets *f32_exact when it is also an fp32 value. */
static double exact_dot(const row_t* a, const row_t* b, int* f32_exact, int* dbl_exact) {
  long long blk[NSF];
  int ex[NSF];
  int have = 0, m = 0;
  for (int k = 0; k < NSF; ++k) {
    int acc = 0;
    for (int i = 0; i < 32; ++i) acc += (int)a->v[32 * k + i] * (int)b->v[32 * k + i];
    blk[k] = acc;
    /* product of two half-unit values is in units of 1/4 */
    ex[k] = (a->e[k] - 127) + (b->e[k] - 127) - 2;
    if (acc != 0) {
      if (!have || ex[k] < m) m = ex[k];
      have = 1;
    }
  }
  *f32_exact = 1;
  *dbl_exact = 1;
  if (!have) return 0.0;
  __int128 tot = 0;
  for (int k = 0; k < NSF; ++k) {
    if (blk[k] == 0) continue;
    int sh = ex[k] - m;
    if (sh > 100) { /* outside any input the generator makes */
      *f32_exact = 0;
      *dbl_exact = 0;
      return NAN;
    }
    tot += ((__int128)blk[k]) << sh;
  }
  if (tot == 0) return 0.0;
  while ((tot & 1) == 0) { tot >>= 1; ++m; }
  __int128 mag = tot < 0 ? -tot : tot;
  int bits = 0;
  for (__int128 t = mag; t; t >>= 1) ++bits;
  if (bits > 53) *dbl_exact = 0;
  /* fp32: 24-bit significand, smallest subnormal 2^-149, largest < 2^128 */
  if (bits > 24 || m < -149 || m + bits > 128) *f32_exact = 0;
  if (bits <= 62) return ldexp((double)(long long)tot, m);
  return ldexp((double)tot, m);
}

static int slot_row(const int32_t* page_table, int32_t max_pages, int32_t req, int32_t s,
                    int32_t num_pages, int64_t* phys_row) {
  int32_t p = s / NPAGE;
  if (p < 0 || p >= max_pages) return -1;
  int32_t page = page_table[(int64_t)req * max_pages + p];
  if (page < 0 || page >= num_pages) return -1;
  *phys_row = (int64_t)page * NPAGE + (s % NPAGE);
  return 0;
}

/*
 * Per-head logits of query row `row` against logical slots [s_begin, s_end)
 * of request `req`.  out is [(s_end - s_begin), 64] in slot-major order.
 * Returns the number of dots that are not exact in fp32, or -1 on a bad page.
 */
long long oracle_row_logits(const uint8_t* q_fp4, const uint8_t* q_scale,
                            const uint8_t* k_fp4, const uint8_t* k_scale,
                            const int32_t* page_table, int32_t max_pages, int32_t num_pages,
                            int32_t row, int32_t req, int32_t s_begin, int32_t s_end,
                            double* out) {
  row_t* qr = (row_t*)malloc(sizeof(row_t) * NH);
  for (int h = 0; h < NH; ++h)
    decode_row(q_fp4 + ((int64_t)row * NH + h) * NDB, q_scale + ((int64_t)row * NH + h) * NSF, &qr[h]);
  long long inexact = 0, bad = 0;
#pragma omp parallel for schedule(static) reduction(+ : inexact, bad)
  for (int32_t s = s_begin; s < s_end; ++s) {
    int64_t pr;
    if (slot_row(page_table, max_pages, req, s, num_pages, &pr)) { bad++; continue; }
    row_t kr;
    decode_row(k_fp4 + pr * NDB, k_scale + pr * NSF, &kr);
    for (int h = 0; h < NH; ++h) {
      int f32e, dble;
      out[(int64_t)(s - s_begin) * NH + h] = exact_dot(&qr[h], &kr, &f32e, &dble);
      inexact += !f32e;
    }
  }
  free(qr);
  return bad ? -1 : inexact;
}

/*
 * Scores of query row `row` over logical slots [s_begin, s_end) of `req`:
 * score = sum over heads h = 0..63, in that order from +0.0, of
 * w[row,h] * max(dot_h, 0), in float64.  Returns the number of dots that are
 * not exact in fp32, or -1 on a bad page.
 */
long long oracle_row_scores(const uint8_t* q_fp4, const uint8_t* q_scale,
                            const uint8_t* k_fp4, const uint8_t* k_scale, const float* weights,
                            const int32_t* page_table, int32_t max_pages, int32_t num_pages,
                            int32_t row, int32_t req, int32_t s_begin, int32_t s_end,
                            double* out) {
  row_t* qr = (row_t*)malloc(sizeof(row_t) * NH);
  double w[NH];
  for (int h = 0; h < NH; ++h) {
    decode_row(q_fp4 + ((int64_t)row * NH + h) * NDB, q_scale + ((int64_t)row * NH + h) * NSF, &qr[h]);
    w[h] = (double)weights[(int64_t)row * NH + h];
  }
  long long inexact = 0, bad = 0;
#pragma omp parallel for schedule(static) reduction(+ : inexact, bad)
  for (int32_t s = s_begin; s < s_end; ++s) {
    int64_t pr;
    if (slot_row(page_table, max_pages, req, s, num_pages, &pr)) { bad++; continue; }
    row_t kr;
    decode_row(k_fp4 + pr * NDB, k_scale + pr * NSF, &kr);
    double acc = 0.0;
    for (int h = 0; h < NH; ++h) {
      int f32e, dble;
      double dot = exact_dot(&qr[h], &kr, &f32e, &dble);
      inexact += !f32e;
      double relu = dot > 0.0 ? dot : 0.0;
      acc += w[h] * relu;
    }
    out[s - s_begin] = acc;
  }
  free(qr);
  return bad ? -1 : inexact;
}

/* ---- total order ---------------------------------------------------------
 * (score, idx) ranks first when: it is a number and the other is NaN; or both
 * numbers and score is larger; or scores compare equal and this one is +0
 * while the other is -0; otherwise the lower logical index ranks first. */
typedef struct {
  double score;
  int64_t idx;
} cand_t;

static int ranks_before(const cand_t* a, const cand_t* b) {
  int na = isnan(a->score), nb = isnan(b->score);
  if (na != nb) return nb;
  if (!na) {
    if (a->score > b->score) return 1;
    if (a->score < b->score) return 0;
    int sa = signbit(a->score) != 0, sb = signbit(b->score) != 0;
    if (sa != sb) return sb;
  }
  return a->idx < b->idx;
}

static int cand_cmp(const void* pa, const void* pb) {
  const cand_t* a = (const cand_t*)pa;
  const cand_t* b = (const cand_t*)pb;
  if (ranks_before(a, b)) return -1;
  if (ranks_before(b, a)) return 1;
  return 0;
}

/*
 * Exact TopK of n scores under the total order, by a full sort.  Entry i has
 * logical index base + i.  Writes the first min(n, k) indices in rank order
 * and pads the rest of out_idx[0..k) with -1.  Returns the count written.
 */
int64_t oracle_select(const double* scores, int64_t n, int64_t base, int32_t k, int32_t* out_idx) {
  cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (size_t)(n > 0 ? n : 1));
  for (int64_t i = 0; i < n; ++i) {
    c[i].score = scores[i];
    c[i].idx = base + i;
  }
  qsort(c, (size_t)n, sizeof(cand_t), cand_cmp);
  int64_t m = n < k ? n : k;
  for (int64_t i = 0; i < k; ++i) out_idx[i] = i < m ? (int32_t)c[i].idx : -1;
  free(c);
  return m;
}

/*
 * The whole prefill for the listed rows.  out_phys and out_raw are
 * [n_rows, topk].  kth_score (nullable) receives each row's topk-th selected
 * score (NaN for short rows); n_inexact (nullable) the count of dots not exact
 * in fp32.  Returns 0, or 1 for bad row metadata, 2 for a bad page entry.
 */
int oracle_prefill_rows(const uint8_t* q_fp4, const uint8_t* q_scale,
                        const uint8_t* k_fp4, const uint8_t* k_scale, const float* weights,
                        const int32_t* page_table, int32_t num_req, int32_t max_pages,
                        int32_t num_pages, const int32_t* row_req, const int32_t* row_start,
                        const int32_t* row_end, const int32_t* rows, int32_t n_rows,
                        int32_t topk, int32_t* out_phys, int32_t* out_raw,
                        double* kth_score, long long* n_inexact) {
  long long inexact_total = 0;
  for (int32_t i = 0; i < n_rows; ++i) {
    int32_t r = rows[i];
    int32_t req = row_req[r], s0 = row_start[r], s1 = row_end[r];
    int32_t* raw = out_raw + (int64_t)i * topk;
    int32_t* phys = out_phys + (int64_t)i * topk;
    if (req < 0 || req >= num_req || s0 < 0 || s1 < s0 || (int64_t)s1 > (int64_t)max_pages * NPAGE)
      return 1;
    int64_t len = (int64_t)s1 - s0;
    if (kth_score) kth_score[i] = NAN;
    if (len <= topk) {
      for (int64_t j = 0; j < topk; ++j) raw[j] = j < len ? (int32_t)(s0 + j) : -1;
    } else {
      double* sc = (double*)malloc(sizeof(double) * (size_t)len);
      long long ie = oracle_row_scores(q_fp4, q_scale, k_fp4, k_scale, weights, page_table,
                                       max_pages, num_pages, r, req, s0, s1, sc);
      if (ie < 0) { free(sc); return 2; }
      inexact_total += ie;
      oracle_select(sc, len, s0, topk, raw);
      if (kth_score) kth_score[i] = sc[raw[topk - 1] - s0];
      free(sc);
    }
    for (int64_t j = 0; j < topk; ++j) {
      if (raw[j] < 0) { phys[j] = -1; continue; }
      int64_t pr;
      if (slot_row(page_table, max_pages, req, raw[j], num_pages, &pr)) return 2;
      phys[j] = (int32_t)pr;
    }
  }
  if (n_inexact) *n_inexact = inexact_total;
  return 0;
}
