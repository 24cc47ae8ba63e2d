/*
 * attn_oracle.c -- fp64 CPU oracle for the scaled-dot-product attention
 * forward  O = softmax(scale * Q K^T) V  and its log-sum-exp.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent reference that the
 * CUDA path is checked against.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load it.  It shares no code, header,
 * table or helper with the CUDA library, and it never calls into it.
 *
 * What it computes (the plain definition, nothing streamed, nothing fused):
 * the problem statement of "Learning FlashAttention the Hard Way -- Part 2"
 * (the SDPA_P / SDPA_L shapes: F.scaled_dot_product_attention on fp16
 * [B,H,N,D] tensors) and the two-kernel naive lowering of its
 * section "Move 0 -- Scalar Streaming Kernel": every score of a query row is
 * materialised, then a max pass, a sum-of-exponentials pass and a
 * normalise-and-multiply-by-V pass.  Per query row i of head (b,h):
 *
 *   J_i    = { j : 0 <= j < Nk }            (non-causal)
 *          = { j : 0 <= j < Nk, j <= i }    (causal, top-left: key j is
 *                                            masked when j > i)
 *   s_j    = scale * sum_d q[i,d] * k[j,d]                 for j in J_i
 *   m      = max_{j in J_i} s_j
 *   dsum   = sum_{j in J_i} exp(s_j - m)
 *   O[i,:] = sum_{j in J_i} (exp(s_j - m) / dsum) * v[j,:]
 *   LSE[i] = m + ln(dsum)                   (natural log)
 *
 * Differences from that naive lowering, all of them precision only: scores
 * are never rounded to fp16 (the page's score kernel stores fp16; here every
 * intermediate is an IEEE double), and the score matrix is held one query
 * row at a time (Nk doubles) instead of as the whole N x N array, which is
 * the same definition row by row.  The inputs are the fp16 bit patterns the
 * GPU reads; each is converted to double exactly.
 *
 * Layout (the pages' listings index q[b*H*N*D + h*N*D + n*D + d], e.g. the
 * head stride 8192 and batch stride 32768 of SDPA_L in "Move 1 -- Tensor
 * Cores"): Q and O are contiguous [B,H,Nq,D], K and V are [B,H,Nk,D], LSE is
 * [B,H,Nq].  Rows are addressed by the flat index r = (b*H + h)*Nq + i.
 *
 * Loop order: for each row the score accumulation runs d-outer / j-inner
 * and the P.V accumulation j-outer / c-inner.  Every individual sum is still
 * taken in ascending index order exactly as written above; only the nesting
 * of independent sums differs, so that the compiler can vectorise them.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* IEEE 754 binary16 -> double, exact (every binary16 value is a double). */
double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int f = h & 0x3ff;
  double mag;
  if (e == 0) {
    mag = ldexp((double)f, -24); /* subnormal: f * 2^-24 */
  } else if (e == 31) {
    mag = (f == 0) ? INFINITY : NAN;
  } else {
    mag = ldexp((double)(1024 + f), e - 25); /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -mag : mag;
}

typedef struct {
  const uint16_t *q;
  const double *kt; /* this head's K, transposed to [D][Nk], as doubles */
  const double *vd; /* this head's V, [Nk][D], as doubles */
  int64_t Nq, Nk, D;
  double scale;
  int causal;
  const int64_t *rows; /* flat row ids of this head */
  int64_t nrows;
  int64_t head_q_offset; /* element offset of this head's Q */
  const int64_t *out_index; /* position of each row in the caller's output */
  double *o_out;   /* [n_total][D] */
  double *lse_out; /* [n_total] */
  double *p_out;   /* [n_total][Nk] or NULL */
  int tid, nthreads;
} work_t;

static void *row_worker(void *arg) {
  work_t *w = (work_t *)arg;
  const int64_t Nk = w->Nk, D = w->D;
  double *s = (double *)malloc(sizeof(double) * (size_t)(Nk > 0 ? Nk : 1));
  double *qrow = (double *)malloc(sizeof(double) * (size_t)D);
  for (int64_t t = w->tid; t < w->nrows; t += w->nthreads) {
    const int64_t r = w->rows[t];
    const int64_t i = r % w->Nq;
    const int64_t slot = w->out_index[t];
    double *o = w->o_out + slot * D;
    /* admissible keys J_i = [0, nval) */
    int64_t nval = Nk;
    if (w->causal && i + 1 < nval) nval = i + 1;

    const uint16_t *qh = w->q + w->head_q_offset + i * D;
    for (int64_t d = 0; d < D; ++d) qrow[d] = oracle_half_to_double(qh[d]);

    /* scores: s_j = scale * sum_d q[i,d] k[j,d] */
    for (int64_t j = 0; j < nval; ++j) s[j] = 0.0;
    for (int64_t d = 0; d < D; ++d) {
      const double qd = qrow[d];
      const double *kd = w->kt + d * Nk;
      for (int64_t j = 0; j < nval; ++j) s[j] += qd * kd[j];
    }
    for (int64_t j = 0; j < nval; ++j) s[j] *= w->scale;

    /* pass 1: row max */
    double m = -INFINITY;
    for (int64_t j = 0; j < nval; ++j)
      if (s[j] > m) m = s[j];
    /* pass 2: denominator; s_j is replaced by exp(s_j - m) */
    double dsum = 0.0;
    for (int64_t j = 0; j < nval; ++j) {
      s[j] = exp(s[j] - m);
      dsum += s[j];
    }
    /* pass 3: normalise and multiply by V */
    for (int64_t c = 0; c < D; ++c) o[c] = 0.0;
    for (int64_t j = 0; j < nval; ++j) {
      const double pj = s[j] / dsum;
      const double *vj = w->vd + j * D;
      for (int64_t c = 0; c < D; ++c) o[c] += pj * vj[c];
    }
    w->lse_out[slot] = m + log(dsum);
    if (w->p_out) {
      double *p = w->p_out + slot * Nk;
      for (int64_t j = 0; j < Nk; ++j) p[j] = (j < nval) ? s[j] / dsum : 0.0;
    }
  }
  free(qrow);
  free(s);
  return NULL;
}

static int cmp_row(const void *a, const void *b) {
  const int64_t x = ((const int64_t *)a)[0], y = ((const int64_t *)b)[0];
  return (x > y) - (x < y);
}

/*
 * Compute O and LSE for a set of query rows.
 *   q  : fp16 bits, [B,H,Nq,D];  k, v : fp16 bits, [B,H,Nk,D]
 *   rows, nrows : flat row ids r = (b*H+h)*Nq + i; rows == NULL means all
 *                 B*H*Nq rows in order (nrows is then ignored).
 *   o_out  : [n][D] doubles, lse_out : [n] doubles, in the order of `rows`.
 *   p_out  : optional [n][Nk] doubles, the softmax row (0 where masked).
 *   nthreads <= 0 uses every online core.
 * Returns the number of threads used, or a negative value on a bad argument.
 */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     int64_t B, int64_t H, int64_t Nq, int64_t Nk, int64_t D,
                     double scale, int causal, const int64_t *rows,
                     int64_t nrows, double *o_out, double *lse_out,
                     double *p_out, int nthreads) {
  if (!q || !k || !v || !o_out || !lse_out) return -1;
  if (B < 1 || H < 1 || Nq < 1 || Nk < 1 || D < 1) return -2;
  if (nthreads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = n > 0 ? (int)n : 1;
  }
  const int64_t total = B * H * Nq;
  if (!rows) nrows = total;
  if (nrows < 0) return -3;

  /* (row id, output slot) pairs sorted by row id so that rows of one head
   * are contiguous and that head's K/V is converted once. */
  int64_t *pairs = (int64_t *)malloc(sizeof(int64_t) * 2 * (size_t)(nrows + 1));
  for (int64_t t = 0; t < nrows; ++t) {
    const int64_t r = rows ? rows[t] : t;
    if (r < 0 || r >= total) {
      free(pairs);
      return -4;
    }
    pairs[2 * t] = r;
    pairs[2 * t + 1] = t;
  }
  qsort(pairs, (size_t)nrows, 2 * sizeof(int64_t), cmp_row);

  double *kt = (double *)malloc(sizeof(double) * (size_t)(Nk * D));
  double *vd = (double *)malloc(sizeof(double) * (size_t)(Nk * D));
  int64_t *hrows = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nrows + 1));
  int64_t *hslot = (int64_t *)malloc(sizeof(int64_t) * (size_t)(nrows + 1));
  pthread_t *th = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
  work_t *ws = (work_t *)malloc(sizeof(work_t) * (size_t)nthreads);

  int64_t t0 = 0;
  while (t0 < nrows) {
    const int64_t head = pairs[2 * t0] / Nq;
    int64_t t1 = t0;
    while (t1 < nrows && pairs[2 * t1] / Nq == head) {
      hrows[t1 - t0] = pairs[2 * t1];
      hslot[t1 - t0] = pairs[2 * t1 + 1];
      ++t1;
    }
    const uint16_t *kh = k + head * Nk * D;
    const uint16_t *vh = v + head * Nk * D;
    for (int64_t j = 0; j < Nk; ++j)
      for (int64_t d = 0; d < D; ++d) {
        kt[d * Nk + j] = oracle_half_to_double(kh[j * D + d]);
        vd[j * D + d] = oracle_half_to_double(vh[j * D + d]);
      }
    const int64_t n_here = t1 - t0;
    const int nt = (int64_t)nthreads < n_here ? nthreads : (int)n_here;
    for (int w = 0; w < nt; ++w) {
      ws[w] = (work_t){q, kt, vd, Nq, Nk, D, scale, causal, hrows, n_here,
                       head * Nq * D, hslot, o_out, lse_out, p_out, w, nt};
      if (nt == 1)
        row_worker(&ws[w]);
      else
        pthread_create(&th[w], NULL, row_worker, &ws[w]);
    }
    if (nt > 1)
      for (int w = 0; w < nt; ++w) pthread_join(th[w], NULL);
    t0 = t1;
  }
  free(ws);
  free(th);
  free(hslot);
  free(hrows);
  free(vd);
  free(kt);
  free(pairs);
  return nthreads;
}
