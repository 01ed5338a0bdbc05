/*
 * attention_bwd_ref.c -- fp64 CPU oracle for the exact-attention backward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may include, link or
 * call this file.  It shares no code, header, table or constant with the
 * CUDA library.
 *
 * With the forward pass S = Q K^T * scale, P = row-softmax(S), O = P V and a
 * loss whose gradient with respect to O is dO, the gradients follow from the
 * chain rule through the three operations (page "llm-infra-atlas /
 * FlashAttention 01", section 5, written out here in my own notation):
 *
 *   dV = P^T dO
 *   dP = dO V^T
 *   dS = P (elementwise) (dP - D),   D_i = sum_c dO_ic O_ic  (the softmax Jacobian
 *                                                             applied row by row)
 *   dQ = dS K * scale
 *   dK = dS^T Q * scale
 *
 * Masked scores have P = 0 and therefore dS = 0.  Masks: causal (key j kept
 * for row i iff j <= i), or a sliding window (wl, wr) aligned bottom-right as
 * in the forward oracle: key j kept iff i + s - wl <= j <= i + s + wr with
 * s = Nk - Nq, a negative bound leaving that side open.  A row that keeps no
 * key has P = 0, O = 0 and D = 0, so it adds nothing to any gradient and its
 * dQ is 0.  Everything is recomputed from Q, K, V and dO in double
 * precision: S, P, O and D of each row are materialised, no tiling, sums in
 * ascending index order.  bf16 inputs are widened exactly.
 *
 * Compiled with -ffp-contract=off (same results on x86-64 and AArch64).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { BWD_F64 = 0, BWD_BF16 = 1 };

static double bf16_to_f64(uint16_t h) {
  uint32_t w = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &w, sizeof f);
  return (double)f;
}

static double elem(const void* base, int dtype, size_t idx) {
  if (dtype == BWD_BF16) return bf16_to_f64(((const uint16_t*)base)[idx]);
  return ((const double*)base)[idx];
}

enum { MASK_NONE = 0, MASK_CAUSAL = 1, MASK_WINDOW = 2 };

/* The keys query row i keeps: [*lo_out, returned end). */
static long visible_keys(long i, long Nq, long Nk, int mask, long wl, long wr, long* lo_out) {
  const int causal = (mask == MASK_CAUSAL);
  long lo = 0, n = Nk;
  if (causal && i + 1 < Nk) n = i + 1;
  if (mask == MASK_WINDOW) {
    const long s = Nk - Nq;
    if (wl >= 0 && i + s - wl > lo) lo = i + s - wl;
    if (wr >= 0 && i + s + wr + 1 < n) n = i + s + wr + 1;
  }
  if (n < lo) n = lo;
  *lo_out = lo;
  return n;
}

/*
 * P row, dP row, O row and D of query row i of one head (base offsets of the
 * head given), over its visible keys [lo, n).  p_row, dp_row: length Nk
 * scratch indexed by key; o_row: length d scratch.
 */
static void row_state(const void* q, const void* k, const void* v, const void* dout, int dtype, size_t q_base,
                      size_t kv_base, long lo, long n, long d, double scale, double* p_row, double* dp_row,
                      double* o_row, double* D_out) {
  if (n <= lo) {
    for (long c = 0; c < d; ++c) o_row[c] = 0.0;
    *D_out = 0.0;
    return;
  }
  /* S row and its safe softmax */
  for (long j = lo; j < n; ++j) {
    double dot = 0.0;
    for (long c = 0; c < d; ++c)
      dot += elem(q, dtype, q_base + (size_t)c) * elem(k, dtype, kv_base + (size_t)j * (size_t)d + (size_t)c);
    p_row[j] = scale * dot;
  }
  double m = p_row[lo];
  for (long j = lo + 1; j < n; ++j)
    if (p_row[j] > m) m = p_row[j];
  double l = 0.0;
  for (long j = lo; j < n; ++j) {
    p_row[j] = exp(p_row[j] - m);
    l += p_row[j];
  }
  for (long j = lo; j < n; ++j) p_row[j] /= l;
  /* O row = P V; dP row = dO_i V^T; D = dO_i . O_i */
  for (long c = 0; c < d; ++c) o_row[c] = 0.0;
  for (long j = lo; j < n; ++j) {
    double dp = 0.0;
    for (long c = 0; c < d; ++c) {
      const double vjc = elem(v, dtype, kv_base + (size_t)j * (size_t)d + (size_t)c);
      o_row[c] += p_row[j] * vjc;
      dp += elem(dout, dtype, q_base + (size_t)c) * vjc;
    }
    dp_row[j] = dp;
  }
  double D = 0.0;
  for (long c = 0; c < d; ++c) D += elem(dout, dtype, q_base + (size_t)c) * o_row[c];
  *D_out = D;
}

int oracle_bwd_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * All gradients: dq [B,H,Nq,d], dk, dv [B,H,Nk,d] (double), from q [B,H,Nq,d],
 * k, v [B,H,Nk,d], dout [B,H,Nq,d].  Heads run in parallel; inside a head the
 * rows are visited in order and dK, dV accumulate in that order.
 */
static int bwd_all(const void* q, const void* k, const void* v, const void* dout, int dtype, double* dq,
                   double* dk, double* dv, long long B, long long H, long long Nq, long long Nk, long long d,
                   double scale, int mask, long wl, long wr, int nthreads) {
  if (!q || !k || !v || !dout || !dq || !dk || !dv) return -1;
  if (B < 0 || H < 0 || Nq < 0 || Nk < 0 || d <= 0) return -2;
  if (dtype != BWD_F64 && dtype != BWD_BF16) return -3;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  const long long BH = B * H;
  int failed = 0;
#pragma omp parallel
  {
    double* p_row = (double*)malloc((size_t)(Nk > 0 ? Nk : 1) * sizeof(double));
    double* dp_row = (double*)malloc((size_t)(Nk > 0 ? Nk : 1) * sizeof(double));
    double* o_row = (double*)malloc((size_t)d * sizeof(double));
    if (!p_row || !dp_row || !o_row) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 1)
      for (long long bh = 0; bh < BH; ++bh) {
        const size_t kv_base = (size_t)bh * (size_t)Nk * (size_t)d;
        double* dk_h = dk + kv_base;
        double* dv_h = dv + kv_base;
        for (size_t x = 0; x < (size_t)Nk * (size_t)d; ++x) dk_h[x] = dv_h[x] = 0.0;
        for (long long i = 0; i < Nq; ++i) {
          const size_t q_base = ((size_t)bh * (size_t)Nq + (size_t)i) * (size_t)d;
          double D;
          long lo;
          const long n = visible_keys((long)i, (long)Nq, (long)Nk, mask, wl, wr, &lo);
          row_state(q, k, v, dout, dtype, q_base, kv_base, lo, n, (long)d, scale, p_row, dp_row, o_row, &D);
          double* dq_row = dq + q_base;
          for (long c = 0; c < d; ++c) dq_row[c] = 0.0;
          for (long j = lo; j < n; ++j) {
            const double ds = p_row[j] * (dp_row[j] - D);
            const size_t krow = kv_base + (size_t)j * (size_t)d;
            for (long c = 0; c < d; ++c) {
              dq_row[c] += ds * elem(k, dtype, krow + (size_t)c);
              dk_h[(size_t)j * (size_t)d + (size_t)c] += ds * elem(q, dtype, q_base + (size_t)c);
              dv_h[(size_t)j * (size_t)d + (size_t)c] += p_row[j] * elem(dout, dtype, q_base + (size_t)c);
            }
          }
          for (long c = 0; c < d; ++c) dq_row[c] *= scale;
        }
        for (size_t x = 0; x < (size_t)Nk * (size_t)d; ++x) dk_h[x] *= scale;
      }
    }
    free(p_row);
    free(dp_row);
    free(o_row);
  }
  return failed ? -5 : 0;
}

/*
 * dQ for selected query rows (flat index (b*H + h)*Nq + i): dq_rows [n_rows, d].
 */
static int bwd_dq_rows(const void* q, const void* k, const void* v, const void* dout, int dtype,
                       const long long* rows, long long n_rows, double* dq_rows, long long B, long long H,
                       long long Nq, long long Nk, long long d, double scale, int mask, long wl, long wr,
                       int nthreads) {
  if (!q || !k || !v || !dout || !dq_rows || (!rows && n_rows > 0)) return -1;
  const long long total = B * H * Nq;
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
    double* p_row = (double*)malloc((size_t)(Nk > 0 ? Nk : 1) * sizeof(double));
    double* dp_row = (double*)malloc((size_t)(Nk > 0 ? Nk : 1) * sizeof(double));
    double* o_row = (double*)malloc((size_t)d * sizeof(double));
    if (!p_row || !dp_row || !o_row) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (long long r = 0; r < n_rows; ++r) {
        const long long bh = rows[r] / Nq, i = rows[r] % Nq;
        const size_t kv_base = (size_t)bh * (size_t)Nk * (size_t)d;
        const size_t q_base = (size_t)rows[r] * (size_t)d;
        double D;
        long lo;
        const long n = visible_keys((long)i, (long)Nq, (long)Nk, mask, wl, wr, &lo);
        row_state(q, k, v, dout, dtype, q_base, kv_base, lo, n, (long)d, scale, p_row, dp_row, o_row, &D);
        double* out = dq_rows + (size_t)r * (size_t)d;
        for (long c = 0; c < d; ++c) out[c] = 0.0;
        for (long j = lo; j < n; ++j) {
          const double ds = p_row[j] * (dp_row[j] - D);
          for (long c = 0; c < d; ++c) out[c] += ds * elem(k, dtype, kv_base + (size_t)j * (size_t)d + (size_t)c);
        }
        for (long c = 0; c < d; ++c) out[c] *= scale;
      }
    }
    free(p_row);
    free(dp_row);
    free(o_row);
  }
  return failed ? -5 : 0;
}

/*
 * dK and dV for selected key rows of ONE head bh: keys[n_keys] are key
 * indices inside that head; dk_rows, dv_rows [n_keys, d].  Every query row of
 * the head is visited (its P row, dP row and D recomputed), and the selected
 * columns are accumulated in query order.
 */
static int bwd_dkdv_keys(const void* q, const void* k, const void* v, const void* dout, int dtype, long long bh,
                         const long long* keys, long long n_keys, double* dk_rows, double* dv_rows, long long B,
                         long long H, long long Nq, long long Nk, long long d, double scale, int mask, long wl,
                         long wr, int nthreads) {
  if (!q || !k || !v || !dout || !dk_rows || !dv_rows || (!keys && n_keys > 0)) return -1;
  if (bh < 0 || bh >= B * H) return -4;
  for (long long t = 0; t < n_keys; ++t)
    if (keys[t] < 0 || keys[t] >= Nk) return -4;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
  const size_t kv_base = (size_t)bh * (size_t)Nk * (size_t)d;
  /* per-query dS and P of the selected keys, computed in parallel over queries */
  double* ds_sel = (double*)malloc((size_t)(Nq > 0 ? Nq : 1) * (size_t)(n_keys > 0 ? n_keys : 1) * sizeof(double));
  double* p_sel = (double*)malloc((size_t)(Nq > 0 ? Nq : 1) * (size_t)(n_keys > 0 ? n_keys : 1) * sizeof(double));
  if (!ds_sel || !p_sel) {
    free(ds_sel);
    free(p_sel);
    return -5;
  }
  int failed = 0;
#pragma omp parallel
  {
    double* p_row = (double*)malloc((size_t)(Nk > 0 ? Nk : 1) * sizeof(double));
    double* dp_row = (double*)malloc((size_t)(Nk > 0 ? Nk : 1) * sizeof(double));
    double* o_row = (double*)malloc((size_t)d * sizeof(double));
    if (!p_row || !dp_row || !o_row) {
#pragma omp atomic write
      failed = 1;
    } else {
#pragma omp for schedule(dynamic, 16)
      for (long long i = 0; i < Nq; ++i) {
        const size_t q_base = ((size_t)bh * (size_t)Nq + (size_t)i) * (size_t)d;
        double D;
        long lo;
        const long n = visible_keys((long)i, (long)Nq, (long)Nk, mask, wl, wr, &lo);
        row_state(q, k, v, dout, dtype, q_base, kv_base, lo, n, (long)d, scale, p_row, dp_row, o_row, &D);
        for (long long t = 0; t < n_keys; ++t) {
          const long j = (long)keys[t];
          const int kept = j >= lo && j < n;
          const double pj = kept ? p_row[j] : 0.0;
          p_sel[(size_t)i * (size_t)n_keys + (size_t)t] = pj;
          ds_sel[(size_t)i * (size_t)n_keys + (size_t)t] = kept ? pj * (dp_row[j] - D) : 0.0;
        }
      }
    }
    free(p_row);
    free(dp_row);
    free(o_row);
  }
  if (!failed) {
    for (long long t = 0; t < n_keys; ++t) {
      double* dkr = dk_rows + (size_t)t * (size_t)d;
      double* dvr = dv_rows + (size_t)t * (size_t)d;
      for (long c = 0; c < d; ++c) dkr[c] = dvr[c] = 0.0;
      for (long long i = 0; i < Nq; ++i) {
        const size_t q_base = ((size_t)bh * (size_t)Nq + (size_t)i) * (size_t)d;
        const double ds = ds_sel[(size_t)i * (size_t)n_keys + (size_t)t];
        const double pj = p_sel[(size_t)i * (size_t)n_keys + (size_t)t];
        for (long c = 0; c < d; ++c) {
          dkr[c] += ds * elem(q, dtype, q_base + (size_t)c);
          dvr[c] += pj * elem(dout, dtype, q_base + (size_t)c);
        }
      }
      for (long c = 0; c < d; ++c) dkr[c] *= scale;
    }
  }
  free(ds_sel);
  free(p_sel);
  return failed ? -5 : 0;
}

/* Public entry points.  causal: 0 or 1.  The _window forms take the window
 * (wl, wr) aligned bottom-right; a negative bound leaves that side open. */
int oracle_attention_bwd(const void* q, const void* k, const void* v, const void* dout, int dtype, double* dq,
                         double* dk, double* dv, long long B, long long H, long long Nq, long long Nk,
                         long long d, double scale, int causal, int nthreads) {
  return bwd_all(q, k, v, dout, dtype, dq, dk, dv, B, H, Nq, Nk, d, scale, causal ? MASK_CAUSAL : MASK_NONE, -1,
                 -1, nthreads);
}

int oracle_attention_bwd_window(const void* q, const void* k, const void* v, const void* dout, int dtype,
                                double* dq, double* dk, double* dv, long long B, long long H, long long Nq,
                                long long Nk, long long d, double scale, long long wl, long long wr,
                                int nthreads) {
  return bwd_all(q, k, v, dout, dtype, dq, dk, dv, B, H, Nq, Nk, d, scale, MASK_WINDOW, (long)wl, (long)wr,
                 nthreads);
}

int oracle_attention_bwd_dq_rows(const void* q, const void* k, const void* v, const void* dout, int dtype,
                                 const long long* rows, long long n_rows, double* dq_rows, long long B,
                                 long long H, long long Nq, long long Nk, long long d, double scale, int causal,
                                 int nthreads) {
  return bwd_dq_rows(q, k, v, dout, dtype, rows, n_rows, dq_rows, B, H, Nq, Nk, d, scale,
                     causal ? MASK_CAUSAL : MASK_NONE, -1, -1, nthreads);
}

int oracle_attention_bwd_dq_rows_window(const void* q, const void* k, const void* v, const void* dout, int dtype,
                                        const long long* rows, long long n_rows, double* dq_rows, long long B,
                                        long long H, long long Nq, long long Nk, long long d, double scale,
                                        long long wl, long long wr, int nthreads) {
  return bwd_dq_rows(q, k, v, dout, dtype, rows, n_rows, dq_rows, B, H, Nq, Nk, d, scale, MASK_WINDOW, (long)wl,
                     (long)wr, nthreads);
}

int oracle_attention_bwd_dkdv_keys(const void* q, const void* k, const void* v, const void* dout, int dtype,
                                   long long bh, const long long* keys, long long n_keys, double* dk_rows,
                                   double* dv_rows, long long B, long long H, long long Nq, long long Nk,
                                   long long d, double scale, int causal, int nthreads) {
  return bwd_dkdv_keys(q, k, v, dout, dtype, bh, keys, n_keys, dk_rows, dv_rows, B, H, Nq, Nk, d, scale,
                       causal ? MASK_CAUSAL : MASK_NONE, -1, -1, nthreads);
}

int oracle_attention_bwd_dkdv_keys_window(const void* q, const void* k, const void* v, const void* dout,
                                          int dtype, long long bh, const long long* keys, long long n_keys,
                                          double* dk_rows, double* dv_rows, long long B, long long H,
                                          long long Nq, long long Nk, long long d, double scale, long long wl,
                                          long long wr, int nthreads) {
  return bwd_dkdv_keys(q, k, v, dout, dtype, bh, keys, n_keys, dk_rows, dv_rows, B, H, Nq, Nk, d, scale,
                       MASK_WINDOW, (long)wl, (long)wr, nthreads);
}
