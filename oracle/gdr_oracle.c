/*
 * Float64 CPU oracle of the gated delta rule: the plain token recurrence.
 *
 * TEST INFRASTRUCTURE ONLY. Used by tests/, __graft_entry__.smoke() and the
 * CPU-baseline legs of bench.py through oracle/native.py. The CUDA library
 * never links or calls this file, and this file includes nothing of it.
 *
 * What it computes (Gated DeltaNet-2 notes, key design 1, in the d_k x d_v
 * orientation of LLMs from scratch ch. 11 section 11.1; order of steps as the
 * KDA derivation, section 3, requires: forget, predict, correct, write, read):
 *
 *   alpha_t = exp(g_t)                       scalar, or per key channel
 *   S~      = Diag(alpha_t) S_{t-1}
 *   r_t     = S~^T e_t
 *   S_t     = S~ + k_t (z_t - r_t)^T
 *   o_t     = S_t^T (scale q_t)
 *
 * with x_t = k_t + lam_t q_t under QMIX (Q-Delta notes, key design 3), else
 * x_t = k_t; e_t = b_t (.) x_t under ERASE_CHANNEL, else beta_t x_t;
 * z_t = w_t (.) v_t under WRITE_CHANNEL, else beta_t v_t.
 *
 * Under BETA_CHANNEL (the README variant of LLMs from scratch ch. 11, section
 * 11.3: a write strength per value channel scaling the prediction error)
 * beta is [B, T, H, d_v], e_t = k_t, z_t = v_t and the write is
 * S_t = S~ + k_t (beta_t (.) (v_t - r_t))^T.
 *
 * Layout: every per-token array is [B, T, H, d] row-major (d fastest); scalar
 * gates are [B, T, H]; states are [B, H, d_k, d_v] (d_v fastest). All double.
 * Each (batch, head) sequence is independent; OpenMP runs them in parallel.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_DECAY_CHANNEL 1u
#define OR_ERASE_CHANNEL 2u
#define OR_WRITE_CHANNEL 4u
#define OR_QMIX 8u
#define OR_BETA_CHANNEL 16u

static void one_sequence(int B, int T, int H, int dk, int dv, unsigned flags,
                         double scale, int bi, int h, const double* q,
                         const double* k, const double* v, const double* g,
                         const double* beta, const double* lam, const double* b,
                         const double* w, const double* h0, double* o,
                         double* hT, double* S, double* x, double* e,
                         double* z, double* alpha, double* r) {
  (void)B;
  if (h0)
    memcpy(S, h0 + ((size_t)bi * H + h) * dk * dv, sizeof(double) * dk * dv);
  else
    memset(S, 0, sizeof(double) * dk * dv);

  for (int t = 0; t < T; ++t) {
    size_t tok = (size_t)bi * T * H + (size_t)t * H + h; /* token-head index */
    const double* qt = q + tok * dk;
    const double* kt = k + tok * dk;
    const double* vt = v + tok * dv;

    /* decay factors */
    for (int i = 0; i < dk; ++i)
      alpha[i] = exp((flags & OR_DECAY_CHANNEL) ? g[tok * dk + i] : g[tok]);

    /* erase direction and write vector */
    for (int i = 0; i < dk; ++i)
      x[i] = (flags & OR_QMIX) ? kt[i] + lam[tok] * qt[i] : kt[i];
    for (int i = 0; i < dk; ++i) {
      if (flags & OR_BETA_CHANNEL)
        e[i] = kt[i];
      else
        e[i] = (flags & OR_ERASE_CHANNEL) ? b[tok * dk + i] * x[i] : beta[tok] * x[i];
    }
    for (int j = 0; j < dv; ++j) {
      if (flags & OR_BETA_CHANNEL)
        z[j] = vt[j];
      else
        z[j] = (flags & OR_WRITE_CHANNEL) ? w[tok * dv + j] * vt[j] : beta[tok] * vt[j];
    }

    /* forget: S~ = Diag(alpha) S */
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[i * dv + j] *= alpha[i];

    /* predict: r = S~^T e */
    for (int j = 0; j < dv; ++j) r[j] = 0.0;
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) r[j] += S[i * dv + j] * e[i];

    /* correct and write: S = S~ + k (z - r)^T, the error scaled per value
     * channel under BETA_CHANNEL */
    if (flags & OR_BETA_CHANNEL)
      for (int j = 0; j < dv; ++j) r[j] = beta[tok * dv + j] * (z[j] - r[j]);
    else
      for (int j = 0; j < dv; ++j) r[j] = z[j] - r[j];
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) S[i * dv + j] += kt[i] * r[j];

    /* read: o = S^T (scale q) */
    double* ot = o + tok * dv;
    for (int j = 0; j < dv; ++j) ot[j] = 0.0;
    for (int i = 0; i < dk; ++i)
      for (int j = 0; j < dv; ++j) ot[j] += S[i * dv + j] * (scale * qt[i]);
  }
  if (hT) memcpy(hT + ((size_t)bi * H + h) * dk * dv, S, sizeof(double) * dk * dv);
}

/* Runs every (batch, head) sequence. Returns 0, or -1 on bad arguments or
 * allocation failure. nthreads <= 0 uses the OpenMP default. */
int gdr_oracle_recurrence(int B, int T, int H, int dk, int dv, unsigned flags,
                          double scale, const double* q, const double* k,
                          const double* v, const double* g, const double* beta,
                          const double* lam, const double* b, const double* w,
                          const double* h0, double* o, double* hT,
                          int nthreads) {
  if (B <= 0 || T <= 0 || H <= 0 || dk <= 0 || dv <= 0) return -1;
  if (!q || !k || !v || !g || !o) return -1;
  if (!((flags & OR_ERASE_CHANNEL) && (flags & OR_WRITE_CHANNEL)) && !beta) return -1;
  if ((flags & OR_QMIX) && !lam) return -1;
  if ((flags & OR_ERASE_CHANNEL) && !b) return -1;
  if ((flags & OR_WRITE_CHANNEL) && !w) return -1;
  int failed = 0;
  int nseq = B * H;
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel
#endif
  {
    size_t per = (size_t)dk * dv + 3 * (size_t)dk + 2 * (size_t)dv + (size_t)dk;
    double* buf = (double*)malloc(sizeof(double) * per);
    double* S = buf;
    double* x = buf ? S + (size_t)dk * dv : NULL;
    double* e = buf ? x + dk : NULL;
    double* alpha = buf ? e + dk : NULL;
    double* z = buf ? alpha + dk : NULL;
    double* r = buf ? z + dv : NULL;
    /* every thread reaches the work-sharing loop, so none waits forever */
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
    for (int s = 0; s < nseq; ++s) {
      if (!buf) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
        failed = 1;
        continue;
      }
      one_sequence(B, T, H, dk, dv, flags, scale, s / H, s % H, q, k, v, g,
                   beta, lam, b, w, h0, o, hT, S, x, e, z, alpha, r);
    }
    free(buf);
  }
  return failed ? -1 : 0;
}

/* Number of threads an OpenMP parallel region would use (1 without OpenMP). */
int gdr_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
