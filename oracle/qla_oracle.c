/*
 * ORACLE -- test infrastructure only.
 *
 * A plain, slow, fp64 restatement of the context-parallel (CP) state
 * correction.  Only the tests, the smoke check and the benchmark's CPU-baseline
 * leg may call it; the library's CUDA path never does, and the two share no
 * code.
 *
 * What it computes.  Antarx Memos, "一次 TileLang Warp Specialization 数值错误的
 * 定位与修复：从双缓冲竞争到 membar":
 *   - section "从版本升级后的数值偏差开始": a long sequence is split into
 *     segments; each segment yields a local state ht (= H_i) and a propagation
 *     matrix mt (= M_i); one kernel corrects the segment-initial states on the
 *     forward pass and the segment-terminal states on the reverse pass; the
 *     state is stored K x V ("kv") or V x K ("vk").
 *   - section "理解三个缓冲区，才能判断哪里需要同步": the simplified state
 *     recurrence, whose printed formula did not survive text extraction.  The
 *     buffer table beside it fixes the roles: H_i seeds the accumulator, the
 *     GEMM reads M_i and the previous state.  The plainest reading is
 *         X_0 = h_init,  X_{i+1} = propagate(M_i, X_i) + H_i,
 *     with propagate = M_i X (kv), X M_i^T (vk) going forward and the
 *     transpose of M_i going in reverse.
 *
 * Outputs (exclusive states, one per segment, the shape of H):
 *   forward: out[i] = X_i for i = 0..S-1 (the initial state of segment i).
 *   reverse: G = h_init; for i = S-1 down to 0: out[i] = G, then (i > 0)
 *            G = propagate_rev(M_i, G) + H_i, i.e. out[i] is the terminal
 *            state of segment i and out[i] = M_{i+1}^T out[i+1] + H_{i+1}
 *            in the kv view.
 *   final_state (optional): the state after the last segment as well, i.e.
 *            X_S (forward) or M_0^T out[0] + H_0 (reverse).
 *
 * Arithmetic: inputs are the fp32 arrays widened exactly to fp64; each output
 * element is one dot product accumulated in fp64 with the summation index
 * ascending, plus H.  kv and vk go through the same loop on index-transposed
 * views, so the oracle's kv and vk results are exact transposes of each other.
 * Chains (b, h) are independent; OpenMP splits chains across threads and does
 * not reorder any sum.
 *
 * Parity of this code is pinned by the tests (unrolled products, closed forms,
 * layout and direction identities, exact integer cases), not by printed values:
 * the pages print none for this computation.
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Element (k, v) of a kv-view state, stored kv ([k][v]) or vk ([v][k]). */
static inline int64_t st_idx(int layout, int K, int V, int k, int v) {
  return layout == 0 ? (int64_t)k * V + v : (int64_t)v * K + k;
}

/* Y = A X + Hseg in the kv view, A = M (forward) or M^T (reverse).
 * X, Y: K x V row-major fp64 scratch.  Hseg may be NULL (no local state). */
static void step(const float* Mseg, const float* Hseg, const double* X, double* Y, int K, int V,
                 int layout, int reverse) {
  for (int k = 0; k < K; ++k) {
    for (int v = 0; v < V; ++v) {
      double acc = 0.0;
      for (int c = 0; c < K; ++c) {
        double a = reverse ? (double)Mseg[(int64_t)c * K + k] : (double)Mseg[(int64_t)k * K + c];
        acc += a * X[(int64_t)c * V + v];
      }
      if (Hseg) acc += (double)Hseg[st_idx(layout, K, V, k, v)];
      Y[(int64_t)k * V + v] = acc;
    }
  }
}

/*
 * H      [nchains][S][state]  fp32 (state = K x V kv or V x K vk)
 * M      [nchains][S][K][K]   fp32
 * h_init [nchains][state]     fp32, NULL means zeros
 * out    [nchains][S][state]  fp64, may be NULL
 * final  [nchains][state]     fp64, may be NULL
 * layout 0 = kv, 1 = vk; direction 0 = forward, 1 = reverse.
 * nthreads <= 0 uses the OpenMP default.  Returns the thread count used.
 */
int qla_oracle_cp_correct(const float* H, const float* M, const float* h_init, double* out,
                          double* final_state, int64_t nchains, int S, int K, int V, int layout,
                          int direction, int nthreads) {
  const int64_t st = (int64_t)K * V;
  int used = 1;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#else
  nthreads = 1;
#endif
#pragma omp parallel num_threads(nthreads)
  {
#ifdef _OPENMP
#pragma omp single
    used = omp_get_num_threads();
#endif
    double* X = (double*)malloc(sizeof(double) * (size_t)st);
    double* Y = (double*)malloc(sizeof(double) * (size_t)st);
#pragma omp for schedule(dynamic, 1)
    for (int64_t c = 0; c < nchains; ++c) {
      const float* Hc = H + c * S * st;
      const float* Mc = M + c * S * (int64_t)K * K;
      for (int k = 0; k < K; ++k)
        for (int v = 0; v < V; ++v)
          X[(int64_t)k * V + v] = h_init ? (double)h_init[c * st + st_idx(layout, K, V, k, v)] : 0.0;
      for (int j = 0; j < S; ++j) {
        /* Step j visits segment i: ascending going forward, descending in reverse. */
        const int i = direction == 0 ? j : S - 1 - j;
        if (out) {
          double* o = out + (c * S + i) * st;
          for (int k = 0; k < K; ++k)
            for (int v = 0; v < V; ++v) o[st_idx(layout, K, V, k, v)] = X[(int64_t)k * V + v];
        }
        const int last = (j == S - 1);
        if (last && !final_state) break;
        step(Mc + (int64_t)i * K * K, Hc + (int64_t)i * st, X, Y, K, V, layout, direction);
        double* t = X;
        X = Y;
        Y = t;
      }
      if (final_state) {
        double* f = final_state + c * st;
        for (int k = 0; k < K; ++k)
          for (int v = 0; v < V; ++v) f[st_idx(layout, K, V, k, v)] = X[(int64_t)k * V + v];
      }
    }
    free(X);
    free(Y);
  }
  return used;
}
