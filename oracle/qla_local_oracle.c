/*
 * ORACLE -- test infrastructure only.
 *
 * The per-segment local pass that produces the inputs of the context-parallel
 * state correction: for every segment of a long sequence, the segment-local
 * state H_i ("ht") and the propagation matrix M_i ("mt") of Antarx Memos,
 * "一次 TileLang Warp Specialization 数值错误的定位与修复：从双缓冲竞争到 membar",
 * section "从版本升级后的数值偏差开始", which names the two quantities (the
 * correction kernel consumes them) but does not say how they are computed.
 *
 * Reading (from outside the pages): the token recurrence of the gated delta
 * rule (S. Yang, J. Kautz, A. Hatamizadeh, "Gated Delta Networks: Improving
 * Mamba2 with Delta Rule", ICLR 2025), written for a K x V state ("kv" view):
 *
 *     X_t = alpha_t (I - beta_t k_t k_t^T) X_{t-1} + beta_t k_t v_t^T,
 *     alpha_t = exp(g_t)
 *
 * with k_t in R^K, v_t in R^V, a write strength beta_t and a log-space decay
 * g_t per token.  The map from the state entering a segment to the state
 * leaving it is affine, X_end = M_i X_start + H_i, with
 *
 *     H_i = the state after the segment's tokens from X = 0,
 *     M_i = A_{last} ... A_{first},  A_t = alpha_t (I - beta_t k_t k_t^T),
 *
 * which is exactly the recurrence the correction pass composes across
 * segments (forward, kv: X_{i+1} = M_i X_i + H_i).  In the vk view the state
 * is stored transposed (H is V x K) and M is the same matrix.
 *
 * Arithmetic: the bf16 keys and values are widened exactly to fp64, beta and
 * g (fp32) likewise, alpha_t = exp(g_t) in fp64.  Token by token, in order:
 * r = k_t^T X (one fp64 dot product per column, row index ascending), then
 * X = alpha_t (X - beta_t k_t r) + beta_t k_t v_t^T, and the same for the
 * propagation matrix P (from the identity, without the write term).  One
 * thread per (chain, segment); OpenMP does not reorder any sum.
 *
 * This is the plain definition, not the chunked form a fast kernel uses.  Its
 * parity is pinned by the tests (explicit matrix products, the delta rule's
 * write-then-read property, orthogonal-key closed forms, composition of
 * sub-segments, a hand-derived example), not by values on the pages.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static inline double bf16_to_double(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/*
 * k [chains][T][K] and v [chains][T][V] bf16 bit patterns; beta, g
 * [chains][T] fp32; T = S * L.  Writes H [chains][S][K][V] (layout 0) or
 * [chains][S][V][K] (layout 1) and M [chains][S][K][K], fp64 (either may be
 * NULL).  Returns the thread count used.
 */
int qla_oracle_local_pass(const uint16_t* k, const uint16_t* v, const float* beta, const float* g, double* H,
                          double* M, int64_t chains, int T, int S, int K, int V, int layout, int nthreads) {
  const int L = T / S;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
  nthreads = 1;
#endif
  const int64_t units = chains * S;
#pragma omp parallel num_threads(nthreads)
  {
    double* X = (double*)malloc(sizeof(double) * (size_t)K * V);
    double* P = (double*)malloc(sizeof(double) * (size_t)K * K);
    double* kt = (double*)malloc(sizeof(double) * (size_t)K);
    double* vt = (double*)malloc(sizeof(double) * (size_t)V);
    double* r = (double*)malloc(sizeof(double) * (size_t)(K > V ? K : V));
#pragma omp for schedule(dynamic, 1)
    for (int64_t u = 0; u < units; ++u) {
      const int64_t c = u / S;
      const int i = (int)(u % S);
      memset(X, 0, sizeof(double) * (size_t)K * V);
      for (int a = 0; a < K; ++a)
        for (int b = 0; b < K; ++b) P[(int64_t)a * K + b] = (a == b) ? 1.0 : 0.0;
      for (int t = i * L; t < (i + 1) * L; ++t) {
        const int64_t tok = c * T + t;
        for (int a = 0; a < K; ++a) kt[a] = bf16_to_double(k[tok * K + a]);
        for (int b = 0; b < V; ++b) vt[b] = bf16_to_double(v[tok * V + b]);
        const double bt = (double)beta[tok];
        const double at = exp((double)g[tok]);
        /* state: r = k^T X, then X = a (X - b k r^T) + b k v^T */
        for (int col = 0; col < V; ++col) {
          double acc = 0.0;
          for (int a = 0; a < K; ++a) acc += kt[a] * X[(int64_t)a * V + col];
          r[col] = acc;
        }
        for (int a = 0; a < K; ++a)
          for (int col = 0; col < V; ++col) {
            double* x = &X[(int64_t)a * V + col];
            *x = at * (*x - bt * kt[a] * r[col]) + bt * kt[a] * vt[col];
          }
        /* propagation matrix: the same transition without the write */
        for (int col = 0; col < K; ++col) {
          double acc = 0.0;
          for (int a = 0; a < K; ++a) acc += kt[a] * P[(int64_t)a * K + col];
          r[col] = acc;
        }
        for (int a = 0; a < K; ++a)
          for (int col = 0; col < K; ++col) {
            double* p = &P[(int64_t)a * K + col];
            *p = at * (*p - bt * kt[a] * r[col]);
          }
      }
      if (H) {
        double* h = H + u * (int64_t)K * V;
        for (int a = 0; a < K; ++a)
          for (int col = 0; col < V; ++col)
            h[layout == 0 ? (int64_t)a * V + col : (int64_t)col * K + a] = X[(int64_t)a * V + col];
      }
      if (M) memcpy(M + u * (int64_t)K * K, P, sizeof(double) * (size_t)K * K);
    }
    free(X);
    free(P);
    free(kt);
    free(vt);
    free(r);
  }
  return nthreads;
}
