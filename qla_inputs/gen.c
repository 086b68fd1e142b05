/*
 * Seeded synthetic inputs for the context-parallel state-correction pass.
 *
 * This file makes input tensors only.  It holds none of the recurrence's
 * arithmetic: both the fp64 oracle and the CUDA path consume the fp32 arrays
 * written here.
 *
 * Random numbers: SplitMix64 (Steele, Lea and Flood, "Fast splittable
 * pseudorandom number generators", OOPSLA 2014) with one independent stream
 * per (seed, tensor id, block index).  A block is one matrix of a tensor, e.g.
 * H[b][h][i] or M[b][h][i], so any block can be regenerated on its own.
 * Gaussians: Box-Muller on two uniforms.  Orthogonal matrices: modified
 * Gram-Schmidt on the columns of a Gaussian matrix, which equals the Q of a QR
 * decomposition with a positive diagonal in R (the Haar convention).
 *
 * Every value is generated in fp64 and rounded to fp32 once.
 * Build with -ffp-contract=off so x86-64 and aarch64 hosts agree.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct { uint64_t s; } qla_rng;

static inline uint64_t sm64_mix(uint64_t z) {
  z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ULL;
  z = (z ^ (z >> 27)) * 0x94d049bb133111ebULL;
  return z ^ (z >> 31);
}

static inline uint64_t rng_next(qla_rng* r) {
  r->s += 0x9e3779b97f4a7c15ULL;
  return sm64_mix(r->s);
}

/* Uniform in [0, 1) with 53 random bits. */
static inline double rng_uniform(qla_rng* r) {
  return (double)(rng_next(r) >> 11) * (1.0 / 9007199254740992.0);
}

static qla_rng stream_for(uint64_t seed, uint64_t tensor_id, int64_t block) {
  qla_rng r;
  uint64_t k = sm64_mix(seed + 0x632be59bd9b4e019ULL);
  k = sm64_mix(k ^ (tensor_id * 0x8cb92ba72f3d8dd7ULL + 0x1ULL));
  k = sm64_mix(k ^ ((uint64_t)block * 0xd6e8feb86659fd93ULL + 0x2ULL));
  r.s = k;
  return r;
}

/* Fills n values with N(0,1) draws, two per Box-Muller pair. */
static void fill_gauss(qla_rng* r, double* dst, int64_t n) {
  const double two_pi = 6.283185307179586476925286766559;
  for (int64_t e = 0; e < n; e += 2) {
    double u1 = 1.0 - rng_uniform(r); /* (0, 1] so the log is finite */
    double u2 = rng_uniform(r);
    double rad = sqrt(-2.0 * log(u1));
    dst[e] = rad * cos(two_pi * u2);
    if (e + 1 < n) dst[e + 1] = rad * sin(two_pi * u2);
  }
}

/* Blocks of block_elems values ~ N(0,1) * scale. */
void qla_gen_gaussian(float* out, int64_t nblocks, int64_t block_elems, uint64_t seed,
                      uint64_t tensor_id, int64_t block0, double scale) {
#pragma omp parallel
  {
    double* tmp = (double*)malloc(sizeof(double) * (size_t)block_elems);
#pragma omp for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
      qla_rng r = stream_for(seed, tensor_id, block0 + b);
      fill_gauss(&r, tmp, block_elems);
      float* o = out + b * block_elems;
      for (int64_t e = 0; e < block_elems; ++e) o[e] = (float)(tmp[e] * scale);
    }
    free(tmp);
  }
}

/* K x K blocks M = g * (I - beta * u u^T): u a unit Gaussian vector,
 * beta ~ U(0,1), g ~ U(gmin, gmax).  Draw order per block: K Gaussians for u,
 * then beta, then g. */
void qla_gen_householder(float* out, int64_t nblocks, int K, uint64_t seed, uint64_t tensor_id,
                         int64_t block0, double gmin, double gmax) {
#pragma omp parallel
  {
    double* u = (double*)malloc(sizeof(double) * (size_t)K);
#pragma omp for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
      qla_rng r = stream_for(seed, tensor_id, block0 + b);
      fill_gauss(&r, u, K);
      double nrm = 0.0;
      for (int k = 0; k < K; ++k) nrm += u[k] * u[k];
      nrm = sqrt(nrm);
      for (int k = 0; k < K; ++k) u[k] /= nrm;
      double beta = rng_uniform(&r);
      double g = gmin + (gmax - gmin) * rng_uniform(&r);
      float* o = out + b * (int64_t)K * K;
      for (int rr = 0; rr < K; ++rr)
        for (int c = 0; c < K; ++c)
          o[(int64_t)rr * K + c] = (float)(g * ((rr == c ? 1.0 : 0.0) - beta * u[rr] * u[c]));
    }
    free(u);
  }
}

/* K x K blocks M = scale * Q, Q orthogonal: modified Gram-Schmidt over the
 * columns of a row-major Gaussian K x K matrix. */
void qla_gen_orthogonal(float* out, int64_t nblocks, int K, uint64_t seed, uint64_t tensor_id,
                        int64_t block0, double scale) {
#pragma omp parallel
  {
    double* a = (double*)malloc(sizeof(double) * (size_t)K * K); /* row-major */
    double* q = (double*)malloc(sizeof(double) * (size_t)K * K); /* q[j*K + r]: column j */
#pragma omp for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
      qla_rng r = stream_for(seed, tensor_id, block0 + b);
      fill_gauss(&r, a, (int64_t)K * K);
      for (int j = 0; j < K; ++j) {
        double* v = q + (int64_t)j * K;
        for (int rr = 0; rr < K; ++rr) v[rr] = a[(int64_t)rr * K + j];
        for (int i = 0; i < j; ++i) {
          const double* qi = q + (int64_t)i * K;
          double d = 0.0;
          for (int rr = 0; rr < K; ++rr) d += qi[rr] * v[rr];
          for (int rr = 0; rr < K; ++rr) v[rr] -= d * qi[rr];
        }
        double nrm = 0.0;
        for (int rr = 0; rr < K; ++rr) nrm += v[rr] * v[rr];
        nrm = sqrt(nrm);
        for (int rr = 0; rr < K; ++rr) v[rr] /= nrm;
      }
      float* o = out + b * (int64_t)K * K;
      for (int rr = 0; rr < K; ++rr)
        for (int c = 0; c < K; ++c) o[(int64_t)rr * K + c] = (float)(scale * q[(int64_t)c * K + rr]);
    }
    free(a);
    free(q);
  }
}

/* K x K signed permutation blocks: one +-1 per row and per column
 * (Fisher-Yates shuffle, then one sign bit per row). */
void qla_gen_signed_perm(float* out, int64_t nblocks, int K, uint64_t seed, uint64_t tensor_id,
                         int64_t block0) {
#pragma omp parallel
  {
    int* perm = (int*)malloc(sizeof(int) * (size_t)K);
#pragma omp for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
      qla_rng r = stream_for(seed, tensor_id, block0 + b);
      for (int k = 0; k < K; ++k) perm[k] = k;
      for (int k = K - 1; k > 0; --k) {
        int j = (int)(rng_next(&r) % (uint64_t)(k + 1));
        int t = perm[k];
        perm[k] = perm[j];
        perm[j] = t;
      }
      float* o = out + b * (int64_t)K * K;
      memset(o, 0, sizeof(float) * (size_t)K * K);
      for (int rr = 0; rr < K; ++rr) o[(int64_t)rr * K + perm[rr]] = (rng_next(&r) >> 63) ? -1.0f : 1.0f;
    }
    free(perm);
  }
}

/* Blocks of integers drawn uniformly from [-maxabs, maxabs]. */
void qla_gen_small_int(float* out, int64_t nblocks, int64_t block_elems, uint64_t seed,
                       uint64_t tensor_id, int64_t block0, int maxabs) {
  const uint64_t span = (uint64_t)(2 * maxabs + 1);
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nblocks; ++b) {
    qla_rng r = stream_for(seed, tensor_id, block0 + b);
    float* o = out + b * block_elems;
    for (int64_t e = 0; e < block_elems; ++e) o[e] = (float)((int64_t)(rng_next(&r) % span) - maxabs);
  }
}

/* ------------------------------------------------------------------ local pass inputs
 * Token-level inputs of the per-segment local pass: keys and values in bf16
 * (bit patterns), write strengths and log-space decays in fp32. */

/* bf16 bit pattern of x: rounded to fp32, then to bf16 with ties to even. */
static uint16_t to_bf16(double x) {
  float f = (float)x;
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  u += 0x7fffu + ((u >> 16) & 1u);
  return (uint16_t)(u >> 16);
}

/* Blocks of `dim` values: a Gaussian vector scaled to unit length, in bf16. */
void qla_gen_unit_bf16(uint16_t* out, int64_t nblocks, int dim, uint64_t seed, uint64_t tensor_id,
                       int64_t block0) {
#pragma omp parallel
  {
    double* tmp = (double*)malloc(sizeof(double) * (size_t)dim);
#pragma omp for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
      qla_rng r = stream_for(seed, tensor_id, block0 + b);
      fill_gauss(&r, tmp, dim);
      double nrm = 0.0;
      for (int e = 0; e < dim; ++e) nrm += tmp[e] * tmp[e];
      nrm = sqrt(nrm);
      uint16_t* o = out + b * (int64_t)dim;
      for (int e = 0; e < dim; ++e) o[e] = to_bf16(tmp[e] / nrm);
    }
    free(tmp);
  }
}

/* Blocks of block_elems values ~ N(0,1) * scale, in bf16. */
void qla_gen_gaussian_bf16(uint16_t* out, int64_t nblocks, int64_t block_elems, uint64_t seed,
                           uint64_t tensor_id, int64_t block0, double scale) {
#pragma omp parallel
  {
    double* tmp = (double*)malloc(sizeof(double) * (size_t)block_elems);
#pragma omp for schedule(static)
    for (int64_t b = 0; b < nblocks; ++b) {
      qla_rng r = stream_for(seed, tensor_id, block0 + b);
      fill_gauss(&r, tmp, block_elems);
      uint16_t* o = out + b * block_elems;
      for (int64_t e = 0; e < block_elems; ++e) o[e] = to_bf16(tmp[e] * scale);
    }
    free(tmp);
  }
}

/* Blocks of block_elems values ~ U(lo, hi); with `log_space` set, the natural
 * logarithm of such a draw (a log-space decay), rounded to fp32 once. */
void qla_gen_uniform(float* out, int64_t nblocks, int64_t block_elems, uint64_t seed, uint64_t tensor_id,
                     int64_t block0, double lo, double hi, int log_space) {
#pragma omp parallel for schedule(static)
  for (int64_t b = 0; b < nblocks; ++b) {
    qla_rng r = stream_for(seed, tensor_id, block0 + b);
    float* o = out + b * block_elems;
    for (int64_t e = 0; e < block_elems; ++e) {
      const double x = lo + (hi - lo) * rng_uniform(&r);
      o[e] = (float)(log_space ? log(x) : x);
    }
  }
}
