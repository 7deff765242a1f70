/*
 * ORACLE — test infrastructure only.
 *
 * A plain, slow, fp64 CPU statement of the Palimpsa dual-state recurrence
 * (metaplastic linear attention). Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg may load this file's library. The CUDA
 * library shares no code, header or table with it.
 *
 * Source: Bonnet, Lohoff, Finkbeiner, Shiqerukaj, Neftci, "Learning to
 * Remember, Learn, and Forget in Attention-Based Models" — the slide deck on
 * it (slides 4, 5 and 7: Eqs. (2), (5) and the gate alpha_t = exp(-A d_t)),
 * and the Chinese reading notes on it (sections 2.1, 2.2 and 2.5).
 *
 * For every head (b, h) and value row i (rows are independent: row i sees
 * only beta_{t,i}, v_{t,i} and the shared key/query), for t = 0..T-1 in order:
 *
 *   alpha_t = exp(-A_h * d_t)                                   (slide 5)
 *   I_t     = alpha_t I_{t-1} + (1 - alpha_t) I_prior + beta_{t,i} k_t^2
 *   mu_t    = alpha_t (I_{t-1} / I_t) mu_{t-1}
 *             + (1 / I_t) (beta_{t,i} v_{t,i}) k_t              (slide 7, Eq. 5)
 *   y_{t,i} = sum_j mu_{t,ij} q_{t,j}      (read after the write; slide 4, Eq. 2)
 *
 * v* variant (slide 11, "preserve writes while introducing importance"): the
 * caller supplies v*_t = beta_t (.) v_t as the input itself, so the content
 * write is (1 / I_t) v*_{t,i} k_t while beta_t still feeds I_t. Selected by
 * v_star = 1 in the *_ex entry points; v then holds v*.
 *
 * Squares, products and divisions are elementwise over the key index j.
 * Nothing is blocked, fused or reordered beyond those definitions. The only
 * parallelism is an OpenMP loop over the independent (b, h, i) rows, which
 * leaves every row's arithmetic in the order written above.
 *
 * Layouts (row-major, contiguous):
 *   q, k        [B, H, T, dk]
 *   v, beta     [B, H, T, dv]
 *   d_t         [B, H, T]
 *   A           [H]
 *   I_prior     [H] when prior_full == 0, [H, dv, dk] when prior_full == 1
 *   mu0, I0     [B, H, dv, dk]; NULL means mu0 = 0 and I0 = I_prior
 *   y           [B, H, T, dv]
 *   muT, IT     [B, H, dv, dk]
 */
#include <math.h>
#include <stddef.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double prior_at(const double *I_prior, int prior_full, long h, long i,
                       long j, long dv, long dk) {
  if (prior_full) return I_prior[(h * dv + i) * dk + j];
  return I_prior[h];
}

/* One value row of one head over all T tokens. mu and I (length dk) hold the
 * state on entry and on exit. y_row has stride dv between tokens. */
static void row_scan(const double *q, const double *k, const double *v,
                     const double *beta, const double *d_t, double A,
                     const double *I_prior, int prior_full, int v_star, long h,
                     long i, long T, long dk, long dv, double *mu, double *I,
                     double *y_row) {
  for (long t = 0; t < T; ++t) {
    const double *kt = k + t * dk;
    const double *qt = q + t * dk;
    const double b = beta[t * dv + i];
    const double vi = v[t * dv + i];
    const double write = v_star ? vi : b * vi; /* the content written to row i */
    const double alpha = exp(-A * d_t[t]);
    double y = 0.0;
    for (long j = 0; j < dk; ++j) {
      const double Ip = prior_at(I_prior, prior_full, h, i, j, dv, dk);
      const double I_prev = I[j];
      const double I_new = alpha * I_prev + (1.0 - alpha) * Ip + b * kt[j] * kt[j];
      const double mu_new = alpha * (I_prev / I_new) * mu[j] + (1.0 / I_new) * write * kt[j];
      I[j] = I_new;
      mu[j] = mu_new;
      y += mu_new * qt[j];
    }
    if (y_row) y_row[t * dv] = y;
  }
}

/* Returns 0 on success, -1 on a bad argument, -2 on allocation failure. */
int oracle_forward_ex(const double *q, const double *k, const double *v,
                      const double *beta, const double *d_t, const double *A,
                      const double *I_prior, int prior_full, int v_star,
                      const double *mu0, const double *I0, double *y,
                      double *muT, double *IT, long B, long H, long T, long dk,
                      long dv, int nthreads) {
  if (!q || !k || !v || !beta || !d_t || !A || !I_prior || !muT || !IT) return -1;
  if (B < 0 || H < 0 || T < 0 || dk <= 0 || dv <= 0) return -1;
  const long rows = B * H * dv;
  int failed = 0;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
#pragma omp parallel for schedule(dynamic, 1) reduction(| : failed)
  for (long r = 0; r < rows; ++r) {
    const long bh = r / dv, i = r % dv, h = bh % H;
    double *mu = (double *)malloc(sizeof(double) * dk);
    double *I = (double *)malloc(sizeof(double) * dk);
    if (!mu || !I) {
      free(mu);
      free(I);
      failed |= 1;
      continue;
    }
    for (long j = 0; j < dk; ++j) {
      const long s = (bh * dv + i) * dk + j;
      mu[j] = mu0 ? mu0[s] : 0.0;
      I[j] = I0 ? I0[s] : prior_at(I_prior, prior_full, h, i, j, dv, dk);
    }
    row_scan(q + bh * T * dk, k + bh * T * dk, v + bh * T * dv,
             beta + bh * T * dv, d_t + bh * T, A[h], I_prior, prior_full, v_star,
             h, i, T, dk, dv, mu, I, y ? y + bh * T * dv + i : NULL);
    for (long j = 0; j < dk; ++j) {
      const long s = (bh * dv + i) * dk + j;
      muT[s] = mu[j];
      IT[s] = I[j];
    }
    free(mu);
    free(I);
  }
  return failed ? -2 : 0;
}

/* The recurrent inference step: Eq. (5) and the readout for one token, with
 * the state (mu, I) read and written in place. This is the same update as one
 * iteration of the scan above (slide 22 / App. A.13 describe the recurrent
 * kernel as the per-token dual-state update). Layouts: q, k [B, H, dk];
 * v, beta [B, H, dv]; d_t [B, H]; mu, I [B, H, dv, dk]; y [B, H, dv]. */
int oracle_forward(const double *q, const double *k, const double *v,
                   const double *beta, const double *d_t, const double *A,
                   const double *I_prior, int prior_full, const double *mu0,
                   const double *I0, double *y, double *muT, double *IT,
                   long B, long H, long T, long dk, long dv, int nthreads) {
  return oracle_forward_ex(q, k, v, beta, d_t, A, I_prior, prior_full, 0, mu0,
                           I0, y, muT, IT, B, H, T, dk, dv, nthreads);
}

int oracle_step_ex(const double *q, const double *k, const double *v,
                   const double *beta, const double *d_t, const double *A,
                   const double *I_prior, int prior_full, int v_star,
                   double *mu, double *I, double *y, long B, long H, long dk,
                   long dv, int nthreads) {
  return oracle_forward_ex(q, k, v, beta, d_t, A, I_prior, prior_full, v_star,
                           mu, I, y, mu, I, B, H, 1, dk, dv, nthreads);
}

int oracle_step(const double *q, const double *k, const double *v,
                const double *beta, const double *d_t, const double *A,
                const double *I_prior, int prior_full, double *mu, double *I,
                double *y, long B, long H, long dk, long dv, int nthreads) {
  return oracle_step_ex(q, k, v, beta, d_t, A, I_prior, prior_full, 0, mu, I,
                        y, B, H, dk, dv, nthreads);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
