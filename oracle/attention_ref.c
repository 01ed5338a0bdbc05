/*
 * attention_ref.c -- fp64 CPU oracle for exact attention (forward pass).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file.  Only the test suite, the smoke check and the bench's CPU
 * baseline leg use it.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * What it computes is the plain definition of attention, written out row by
 * row with the score row S and the probability row P materialised:
 *
 *   S = Q K^T * scale                     (page "llm-infra-atlas / 01 IO
 *                                          awareness", section 1; page
 *                                          "lumenova research-attention",
 *                                          section 01)
 *   P = row-softmax(S), computed safely: m = max_j S_j, e_j = exp(S_j - m),
 *       l = sum_j e_j, P_j = e_j / l       (page "jianzhnie flash-attention",
 *                                          section 4.3, equations (2)-(4))
 *   O = P V
 *   LSE = m + ln(l)                       (page "llm-infra-atlas / 01",
 *                                          sections 3 and 5: the statistic
 *                                          that lets P = exp(S - LSE) be
 *                                          rebuilt in the backward pass)
 *
 * Readings taken where the pages are silent:
 *   - causal masking keeps key j for query row i iff j <= i (top-left
 *     alignment); a masked key is left out of the row entirely, which is the
 *     same as exp(-inf) = 0;
 *   - a sliding window (the "sliding" mask named beside "causal" in the
 *     tiled loop of page "llm-infra-atlas / FlashAttention 01", section 3)
 *     keeps key j for row i iff  i + s - wl <= j <= i + s + wr  with
 *     s = Nk - Nq (the window's diagonal ends at the last query and the last
 *     key: bottom-right alignment) and wl or wr < 0 meaning unbounded on that
 *     side; causal is the window (-1, 0);
 *   - the scale multiplies the fp64 dot product (never a pre-scaled Q);
 *   - LSE is a natural logarithm, in scaled-logit units;
 *   - a row with no allowed key (possible only under a window with Nq > Nk)
 *     gives O = 0 and LSE = -inf.
 *
 * No tiling, no exp2, no online recurrence, no lazy rescaling: the sums run
 * over j in ascending order, in double precision.  bf16 inputs are widened to
 * double exactly (a bf16 value is the upper half of an IEEE binary32).
 *
 * Compiled with -ffp-contract=off so that no multiply-add is fused and the
 * result is the same on x86-64 and AArch64 hosts.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F64 = 0, ORACLE_BF16 = 1 };

/* Exact bf16 -> double: the 16 bits are the high half of a binary32. */
static double bf16_bits_to_double(uint16_t h) {
  uint32_t w = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static double load_elem(const void* base, int dtype, size_t idx) {
  if (dtype == ORACLE_BF16) return bf16_bits_to_double(((const uint16_t*)base)[idx]);
  return ((const double*)base)[idx];
}

/*
 * One query row.  s_row and p_row are caller-provided scratch of length Nk.
 * q_base: offset of this row's query vector; kv_base: offset of key/value
 * row 0 of this (b, h).
 */
static void attend_one_row(const void* q, const void* k, const void* v, int dtype,
                           size_t q_base, size_t kv_base, long i, long Nk, long d,
                           double scale, long j_first, long j_last, double* s_row, double* p_row,
                           double* o_row, double* lse_out) {
  /* visible keys: j_first <= j <= j_last, clipped to [0, Nk) */
  if (j_first < 0) j_first = 0;
  if (j_last > Nk - 1) j_last = Nk - 1;
  const long n_keys = j_last - j_first + 1;
  (void)i;

  for (long c = 0; c < d; ++c) o_row[c] = 0.0;
  if (n_keys <= 0) {
    *lse_out = -INFINITY;
    return;
  }

  /* S row: s_j = scale * <q_i, k_j>, stored at index j - j_first */
  for (long j = j_first; j <= j_last; ++j) {
    double dot = 0.0;
    size_t krow = kv_base + (size_t)j * (size_t)d;
    for (long c = 0; c < d; ++c)
      dot += load_elem(q, dtype, q_base + (size_t)c) * load_elem(k, dtype, krow + (size_t)c);
    s_row[j - j_first] = scale * dot;
  }

  /* safe softmax: pass 1 max, pass 2 sum of exp(s - m), pass 3 normalise */
  double m = s_row[0];
  for (long t = 1; t < n_keys; ++t)
    if (s_row[t] > m) m = s_row[t];
  double l = 0.0;
  for (long t = 0; t < n_keys; ++t) {
    p_row[t] = exp(s_row[t] - m);
    l += p_row[t];
  }
  for (long t = 0; t < n_keys; ++t) p_row[t] = p_row[t] / l;

  /* O row = P row times V */
  for (long t = 0; t < n_keys; ++t) {
    size_t vrow = kv_base + (size_t)(j_first + t) * (size_t)d;
    double pj = p_row[t];
    for (long c = 0; c < d; ++c) o_row[c] += pj * load_elem(v, dtype, vrow + (size_t)c);
  }
  *lse_out = m + log(l);
}

/* Visible key range of row i.  mode 0: all keys; mode 1: causal, top-left
 * (j <= i); mode 2: window (wl, wr), bottom-right aligned. */
static void key_range(long i, long Nq, long Nk, int mode, long long wl, long long wr, long* j_first,
                      long* j_last) {
  *j_first = 0;
  *j_last = Nk - 1;
  if (mode == 1) {
    *j_last = i;
  } else if (mode == 2) {
    const long long diag = (long long)i + (long long)Nk - (long long)Nq;
    if (wl >= 0) *j_first = (long)(diag - wl > -1 ? diag - wl : -1);
    if (wr >= 0) *j_last = (long)(diag + wr < (long long)Nk ? diag + wr : (long long)Nk);
  }
}

int oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Rows given by flat index r in [0, B*H*Nq): (b*H + h)*Nq + i.
 * Outputs: o[n_rows * d] and lse[n_rows], in the order of rows[].
 * Inputs laid out [B, H, Nq, d] (q) and [B, H, Nk, d] (k, v), contiguous.
 * Returns 0 on success, a negative value on bad arguments or no memory.
 */
static int rows_impl(const void* q, const void* k, const void* v, int dtype, const long long* rows,
                     long long n_rows, double* o, double* lse, long long B, long long H, long long Nq,
                     long long Nk, long long d, double scale, int mode, long long wl, long long wr,
                     int nthreads);

int oracle_attention_rows(const void* q, const void* k, const void* v, int dtype,
                          const long long* rows, long long n_rows, double* o, double* lse,
                          long long B, long long H, long long Nq, long long Nk, long long d,
                          double scale, int causal, int nthreads) {
  return rows_impl(q, k, v, dtype, rows, n_rows, o, lse, B, H, Nq, Nk, d, scale, causal ? 1 : 0, -1, -1,
                   nthreads);
}

/* Selected rows under a window (wl, wr) aligned bottom-right; < 0 = unbounded. */
int oracle_attention_rows_window(const void* q, const void* k, const void* v, int dtype,
                                 const long long* rows, long long n_rows, double* o, double* lse,
                                 long long B, long long H, long long Nq, long long Nk, long long d,
                                 double scale, long long wl, long long wr, int nthreads) {
  return rows_impl(q, k, v, dtype, rows, n_rows, o, lse, B, H, Nq, Nk, d, scale, 2, wl, wr, nthreads);
}

static int rows_impl(const void* q, const void* k, const void* v, int dtype, const long long* rows,
                     long long n_rows, double* o, double* lse, long long B, long long H, long long Nq,
                     long long Nk, long long d, double scale, int mode, long long wl, long long wr,
                     int nthreads) {
  if (!q || !k || !v || !o || !lse || (!rows && n_rows > 0)) return -1;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0 || n_rows < 0) return -2;
  if (dtype != ORACLE_F64 && dtype != ORACLE_BF16) return -3;
  long long total = B * H * Nq;
  for (long long r = 0; r < n_rows; ++r)
    if (rows[r] < 0 || rows[r] >= total) return -4;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  int failed = 0;
#pragma omp parallel
  {
    size_t nbuf = (size_t)(Nk > 0 ? Nk : 1);
    double* s_row = (double*)malloc(nbuf * sizeof(double));
    double* p_row = (double*)malloc(nbuf * sizeof(double));
    if (!s_row || !p_row) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (long long r = 0; r < n_rows; ++r) {
        long long flat = rows[r];
        long long bh = flat / Nq;
        long long i = flat % Nq;
        size_t q_base = (size_t)flat * (size_t)d;
        size_t kv_base = (size_t)bh * (size_t)Nk * (size_t)d;
        long jf, jl;
        key_range((long)i, (long)Nq, (long)Nk, mode, wl, wr, &jf, &jl);
        attend_one_row(q, k, v, dtype, q_base, kv_base, (long)i, (long)Nk, (long)d, scale, jf, jl,
                       s_row, p_row, o + (size_t)r * (size_t)d, lse + r);
      }
    }
    free(s_row);
    free(p_row);
  }
  return failed ? -5 : 0;
}

static int fwd_impl(const void* q, const void* k, const void* v, int dtype, double* o, double* lse,
                    long long B, long long H, long long Nq, long long Nk, long long d, double scale,
                    int mode, long long wl, long long wr, int nthreads);

/* All rows: o[B*H*Nq*d], lse[B*H*Nq]. */
int oracle_attention_fwd(const void* q, const void* k, const void* v, int dtype, double* o,
                         double* lse, long long B, long long H, long long Nq, long long Nk,
                         long long d, double scale, int causal, int nthreads) {
  return fwd_impl(q, k, v, dtype, o, lse, B, H, Nq, Nk, d, scale, causal ? 1 : 0, -1, -1, nthreads);
}

/* All rows under a window (wl, wr) aligned bottom-right; < 0 = unbounded. */
int oracle_attention_fwd_window(const void* q, const void* k, const void* v, int dtype, double* o,
                                double* lse, long long B, long long H, long long Nq, long long Nk,
                                long long d, double scale, long long wl, long long wr, int nthreads) {
  return fwd_impl(q, k, v, dtype, o, lse, B, H, Nq, Nk, d, scale, 2, wl, wr, nthreads);
}

static int fwd_impl(const void* q, const void* k, const void* v, int dtype, double* o, double* lse,
                    long long B, long long H, long long Nq, long long Nk, long long d, double scale,
                    int mode, long long wl, long long wr, int nthreads) {
  if (!q || !k || !v || !o || !lse) return -1;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0) return -2;
  if (dtype != ORACLE_F64 && dtype != ORACLE_BF16) return -3;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  long long total = B * H * Nq;
  int failed = 0;
#pragma omp parallel
  {
    size_t nbuf = (size_t)(Nk > 0 ? Nk : 1);
    double* s_row = (double*)malloc(nbuf * sizeof(double));
    double* p_row = (double*)malloc(nbuf * sizeof(double));
    if (!s_row || !p_row) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (long long flat = 0; flat < total; ++flat) {
        long long bh = flat / Nq;
        long long i = flat % Nq;
        size_t q_base = (size_t)flat * (size_t)d;
        size_t kv_base = (size_t)bh * (size_t)Nk * (size_t)d;
        long jf, jl;
        key_range((long)i, (long)Nq, (long)Nk, mode, wl, wr, &jf, &jl);
        attend_one_row(q, k, v, dtype, q_base, kv_base, (long)i, (long)Nk, (long)d, scale, jf, jl,
                       s_row, p_row, o + (size_t)flat * (size_t)d, lse + flat);
      }
    }
    free(s_row);
    free(p_row);
  }
  return failed ? -5 : 0;
}
