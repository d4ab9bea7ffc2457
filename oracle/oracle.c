/*
 * Oracle for frame-aligned window-sparse attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * cpu_baseline / reference legs of bench.py may build, load or call this.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Plain, slow, obviously correct fp64 code.  Every function restates a
 * passage of the Google Developers Blog post "HeyGen x Google Cloud:
 * Bringing Avatar IV to TPUs" (cited by section):
 *
 *   orc_mask            section "Deleting the mask", Fig. 3: each frame's
 *                       tokens attend a window of nearby frames plus one
 *                       global reference frame; the mask is frame-aligned.
 *   orc_blockmap        same section: blocks whose sizes are multiples of 16
 *                       dividing the frame token span are either fully inside
 *                       or fully outside the mask.
 *   orc_prepare         section "Breaking softmax's dependency chain": key
 *                       mean-centering, each row's Cauchy-Schwarz bound
 *                       (query norm times the max key norm), per-head
 *                       eligibility (a bound far above the true max makes the
 *                       exponentials underflow).
 *   orc_prepare_window  the same with each row's bound over the keys it
 *                       attends (the window, not all keys).
 *   orc_attention_rows  the plain definition: masked softmax(q k^T * scale) v
 *                       over the element-by-element mask, max-subtracted.
 *   orc_attention_rows_fixed   Fig. 4 bottom: the row bound as a fixed max.
 *   orc_attention_rows_online  Fig. 4 top: the flash-style running max with
 *                              accumulator rescaling, key block by key block.
 *
 * Readings of points the pages leave open (token order, what reference rows
 * see, which keys the mean covers, tau, the underflow clause) are listed with
 * each function.
 *
 * Inputs are fp64 arrays laid out [nbh][N][D] (the caller upcasts bf16
 * exactly).  Token i belongs to frame floor(i / T); frames [0, R) are the
 * reference frames (a prefix), frame R + f is video frame f.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* Mask element M[i, j] (1 = query token i attends key token j).
 * Reading: every query attends every reference key; reference queries are
 * global and attend every key; video queries attend video keys whose frame
 * index differs by at most w (clipped at the ends, no wrap-around).
 * Variants of the same family (flags, or-ed; 0 = the reading above):
 *   1  causal window: video frame f attends video frames f - w .. f;
 *   2  the reference frames follow the F video frames in token order;
 *   4  reference queries attend only reference keys. */
int orc_mask(long F, long T, long w, long R, long flags, long i, long j) {
  long fi = i / T, fj = j / T;
  int ref_i, ref_j;
  long vi, vj;
  if (flags & 2) {
    ref_i = fi >= F;
    ref_j = fj >= F;
    vi = fi;
    vj = fj;
  } else {
    ref_i = fi < R;
    ref_j = fj < R;
    vi = fi - R;
    vj = fj - R;
  }
  if (ref_i) return (flags & 4) ? ref_j : 1;
  if (ref_j) return 1;
  long d = vi - vj;
  if (flags & 1) return (d >= 0 && d <= w) ? 1 : 0;
  if (d < 0) d = -d;
  return d <= w ? 1 : 0;
}

/* The whole N x N mask, element by element (small shapes only). */
void orc_mask_dense(long F, long T, long w, long R, long flags, uint8_t* out) {
  long n = (F + R) * T;
  for (long i = 0; i < n; ++i)
    for (long j = 0; j < n; ++j) out[i * n + j] = (uint8_t)orc_mask(F, T, w, R, flags, i, j);
}

/* Classifies every bq x bk block of the element mask.
 * bitmap[qb * nkb + kb] = 1 when the block holds any active element.
 * CSR lists those blocks row by row in increasing kb.
 * counts[0..3] = full, empty, partial blocks, nonzero blocks.
 * Returns 0, or -1 when col_cap is too small or the sizes do not tile N. */
int orc_blockmap(long F, long T, long w, long R, long flags, long bq, long bk, uint8_t* bitmap,
                 int32_t* row_ptr, int32_t* col, long col_cap, long* counts) {
  long n = (F + R) * T;
  if (bq <= 0 || bk <= 0 || n % bq != 0 || n % bk != 0) return -1;
  long nqb = n / bq, nkb = n / bk;
  long n_full = 0, n_empty = 0, n_partial = 0;
#pragma omp parallel for reduction(+ : n_full, n_empty, n_partial) schedule(dynamic, 1)
  for (long qb = 0; qb < nqb; ++qb) {
    for (long kb = 0; kb < nkb; ++kb) {
      long active = 0;
      for (long i = qb * bq; i < (qb + 1) * bq; ++i)
        for (long j = kb * bk; j < (kb + 1) * bk; ++j) active += orc_mask(F, T, w, R, flags, i, j);
      if (active == 0) {
        n_empty++;
        bitmap[qb * nkb + kb] = 0;
      } else {
        if (active == bq * bk)
          n_full++;
        else
          n_partial++;
        bitmap[qb * nkb + kb] = 1;
      }
    }
  }
  long nnz = 0;
  row_ptr[0] = 0;
  for (long qb = 0; qb < nqb; ++qb) {
    for (long kb = 0; kb < nkb; ++kb) {
      if (bitmap[qb * nkb + kb]) {
        if (nnz >= col_cap) return -1;
        col[nnz++] = (int32_t)kb;
      }
    }
    row_ptr[qb + 1] = (int32_t)nnz;
  }
  counts[0] = n_full;
  counts[1] = n_empty;
  counts[2] = n_partial;
  counts[3] = nnz;
  return 0;
}

/* Per-head statistics of the fixed-max method, in fp64.
 *   mu[h][d]  = mean over all N keys of head h      (reading: the mean runs
 *               over every key of the head, reference frame included)
 *   kmax[h]   = max_j || k_j - mu ||                (the global max key norm
 *               of the head: valid for any key slice a row sees)
 *   qn[h][i]  = || q_i ||
 *   b[h][i]   = scale * qn[h][i] * kmax[h]          (the row's bound, in
 *               scaled-logit units)
 *   bmax[h]   = max_i b[h][i]
 *   elig[h]   = 1 iff bmax[h] <= tau and every row has 2 * b_i < 126 ln 2
 *               (reading: every exponent s' - b_i lies in [-2 b_i, 0], so
 *               it stays an fp32 normal; tau comes from the library, 40). */
void orc_prepare(const double* q, const double* k, long nbh, long n, long d, double scale,
                 double tau, double* mu, double* kmax, double* qn, double* b, double* bmax,
                 uint8_t* elig) {
  const double underflow_limit = 126.0 * log(2.0);
#pragma omp parallel for schedule(dynamic, 1)
  for (long h = 0; h < nbh; ++h) {
    const double* kh = k + h * n * d;
    const double* qh = q + h * n * d;
    double* m = mu + h * d;
    for (long c = 0; c < d; ++c) m[c] = 0.0;
    for (long j = 0; j < n; ++j)
      for (long c = 0; c < d; ++c) m[c] += kh[j * d + c];
    for (long c = 0; c < d; ++c) m[c] /= (double)n;
    double km = 0.0;
    for (long j = 0; j < n; ++j) {
      double s = 0.0;
      for (long c = 0; c < d; ++c) {
        double x = kh[j * d + c] - m[c];
        s += x * x;
      }
      double nk = sqrt(s);
      if (nk > km) km = nk;
    }
    kmax[h] = km;
    double bm = 0.0;
    int rows_ok = 1;
    for (long i = 0; i < n; ++i) {
      double s = 0.0;
      for (long c = 0; c < d; ++c) s += qh[i * d + c] * qh[i * d + c];
      qn[h * n + i] = sqrt(s);
      b[h * n + i] = scale * qn[h * n + i] * km;
      if (b[h * n + i] > bm) bm = b[h * n + i];
      if (!(2.0 * b[h * n + i] < underflow_limit)) rows_ok = 0;
    }
    bmax[h] = bm;
    elig[h] = (uint8_t)((bm <= tau) && rows_ok);
  }
}

/* The same statistics with the window bound (the tighter variant of the
 * section "Breaking softmax's dependency chain": any key set that contains a
 * row's active keys bounds its logits, and the smallest is the row's own):
 *   mu, kmax, qn  as in orc_prepare (kmax stays the global maximum);
 *   b[h][i]  = scale * qn[h][i] * max_{j : M[i, j] = 1} || k_j - mu ||
 *              (the mask walked element by element for every row);
 *   bmax, elig    from these b as in orc_prepare. */
void orc_prepare_window(const double* q, const double* k, long nbh, long n, long d, long F,
                        long T, long w, long R, long flags, double scale, double tau, double* mu,
                        double* kmax, double* qn, double* b, double* bmax, uint8_t* elig) {
  const double underflow_limit = 126.0 * log(2.0);
  double* knorm = (double*)malloc(sizeof(double) * (size_t)n * (size_t)nbh);
  if (!knorm) return;
#pragma omp parallel for schedule(dynamic, 1)
  for (long h = 0; h < nbh; ++h) {
    const double* kh = k + h * n * d;
    const double* qh = q + h * n * d;
    double* m = mu + h * d;
    double* kn = knorm + h * n;
    for (long c = 0; c < d; ++c) m[c] = 0.0;
    for (long j = 0; j < n; ++j)
      for (long c = 0; c < d; ++c) m[c] += kh[j * d + c];
    for (long c = 0; c < d; ++c) m[c] /= (double)n;
    double km = 0.0;
    for (long j = 0; j < n; ++j) {
      double s = 0.0;
      for (long c = 0; c < d; ++c) {
        double x = kh[j * d + c] - m[c];
        s += x * x;
      }
      kn[j] = sqrt(s);
      if (kn[j] > km) km = kn[j];
    }
    kmax[h] = km;
    double bm = 0.0;
    int rows_ok = 1;
    for (long i = 0; i < n; ++i) {
      double s = 0.0;
      for (long c = 0; c < d; ++c) s += qh[i * d + c] * qh[i * d + c];
      qn[h * n + i] = sqrt(s);
      double kw = 0.0;
      for (long j = 0; j < n; ++j)
        if (orc_mask(F, T, w, R, flags, i, j) && kn[j] > kw) kw = kn[j];
      b[h * n + i] = scale * qn[h * n + i] * kw;
      if (b[h * n + i] > bm) bm = b[h * n + i];
      if (!(2.0 * b[h * n + i] < underflow_limit)) rows_ok = 0;
    }
    bmax[h] = bm;
    elig[h] = (uint8_t)((bm <= tau) && rows_ok);
  }
  free(knorm);
}

/* Scratch of N doubles per thread for the logits of one row. */
static double* row_scratch(long n) { return (double*)malloc((size_t)n * sizeof(double)); }

/* o_i = sum_{j in A(i)} exp(s_ij - max_A s) v_j / sum_{j in A(i)} exp(s_ij - max_A s),
 * s_ij = scale * q_i . k_j, A(i) = { j : M[i, j] = 1 }, for the listed
 * (head, row) pairs.  out is [npairs][D]. */
void orc_attention_rows(const double* q, const double* k, const double* v, long n, long d,
                        long F, long T, long w, long R, long flags, double scale, long npairs,
                        const int64_t* head, const int64_t* row, double* out) {
#pragma omp parallel
  {
    double* s = row_scratch(n);
#pragma omp for schedule(dynamic, 4)
    for (long p = 0; p < npairs; ++p) {
      const long h = (long)head[p], i = (long)row[p];
      const double* qi = q + (h * n + i) * d;
      const double* kh = k + h * n * d;
      const double* vh = v + h * n * d;
      double mx = -INFINITY;
      for (long j = 0; j < n; ++j) {
        if (!orc_mask(F, T, w, R, flags, i, j)) continue;
        double acc = 0.0;
        for (long c = 0; c < d; ++c) acc += qi[c] * kh[j * d + c];
        s[j] = scale * acc;
        if (s[j] > mx) mx = s[j];
      }
      double den = 0.0;
      double* o = out + p * d;
      for (long c = 0; c < d; ++c) o[c] = 0.0;
      for (long j = 0; j < n; ++j) {
        if (!orc_mask(F, T, w, R, flags, i, j)) continue;
        double e = exp(s[j] - mx);
        den += e;
        for (long c = 0; c < d; ++c) o[c] += e * vh[j * d + c];
      }
      for (long c = 0; c < d; ++c) o[c] /= den;
    }
    free(s);
  }
}

/* Fixed-max formulation: logits against the centered keys k_j - mu, and the
 * row bound b_i used in place of the row max: p_ij = exp(s'_ij - b_i).
 * mu is [nbh][D], b is [nbh][N] (from orc_prepare). */
void orc_attention_rows_fixed(const double* q, const double* k, const double* v,
                              const double* mu, const double* b, long n, long d, long F,
                              long T, long w, long R, long flags, double scale, long npairs,
                              const int64_t* head, const int64_t* row, double* out) {
#pragma omp parallel for schedule(dynamic, 4)
  for (long p = 0; p < npairs; ++p) {
    const long h = (long)head[p], i = (long)row[p];
    const double* qi = q + (h * n + i) * d;
    const double* kh = k + h * n * d;
    const double* vh = v + h * n * d;
    const double* m = mu + h * d;
    const double bi = b[h * n + i];
    double den = 0.0;
    double* o = out + p * d;
    for (long c = 0; c < d; ++c) o[c] = 0.0;
    for (long j = 0; j < n; ++j) {
      if (!orc_mask(F, T, w, R, flags, i, j)) continue;
      double acc = 0.0;
      for (long c = 0; c < d; ++c) acc += qi[c] * (kh[j * d + c] - m[c]);
      double e = exp(scale * acc - bi);
      den += e;
      for (long c = 0; c < d; ++c) o[c] += e * vh[j * d + c];
    }
    for (long c = 0; c < d; ++c) o[c] /= den;
  }
}

/* Online (flash-style) formulation: active keys visited in blocks of bk
 * consecutive key indices; a running max m, and the running sum and output
 * rescaled by exp(m_old - m_new) whenever a block raises the max. */
void orc_attention_rows_online(const double* q, const double* k, const double* v, long n,
                               long d, long F, long T, long w, long R, long flags, double scale,
                               long bk,
                               long npairs, const int64_t* head, const int64_t* row,
                               double* out) {
#pragma omp parallel
  {
    double* s = row_scratch(n);
#pragma omp for schedule(dynamic, 4)
    for (long p = 0; p < npairs; ++p) {
      const long h = (long)head[p], i = (long)row[p];
      const double* qi = q + (h * n + i) * d;
      const double* kh = k + h * n * d;
      const double* vh = v + h * n * d;
      double* o = out + p * d;
      for (long c = 0; c < d; ++c) o[c] = 0.0;
      double m = -INFINITY, l = 0.0;
      for (long j0 = 0; j0 < n; j0 += bk) {
        long j1 = j0 + bk < n ? j0 + bk : n;
        double bm = -INFINITY;
        int any = 0;
        for (long j = j0; j < j1; ++j) {
          if (!orc_mask(F, T, w, R, flags, i, j)) continue;
          double acc = 0.0;
          for (long c = 0; c < d; ++c) acc += qi[c] * kh[j * d + c];
          s[j] = scale * acc;
          if (s[j] > bm) bm = s[j];
          any = 1;
        }
        if (!any) continue;
        double m_new = bm > m ? bm : m;
        double alpha = exp(m - m_new); /* 0 on the first block */
        l *= alpha;
        for (long c = 0; c < d; ++c) o[c] *= alpha;
        for (long j = j0; j < j1; ++j) {
          if (!orc_mask(F, T, w, R, flags, i, j)) continue;
          double e = exp(s[j] - m_new);
          l += e;
          for (long c = 0; c < d; ++c) o[c] += e * vh[j * d + c];
        }
        m = m_new;
      }
      for (long c = 0; c < d; ++c) o[c] /= l;
    }
    free(s);
  }
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
