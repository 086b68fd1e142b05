// Sequential state correction, plain FFMA engine (no TMA, no warp roles).
//
// Computes the recurrence of Antarx Memos, "一次 TileLang Warp Specialization 数
// 值错误的定位与修复", section "理解三个缓冲区，才能判断哪里需要同步":
// X_{i+1} = propagate(M_i, X_i) + H_i, with out[seg] = the state entering seg.
// It plays the role of that page's WS-off kernel (section "先恢复正确性：只关闭
// 问题 kernel 的 WS"): one thread group does the loads and the math, so there
// is no slot handoff to get wrong.  It serves every supported shape and is the
// reference point for the warp-specialised engines.
//
// One CTA owns a 32-column tile of the kv-view state of one unit (chain,
// group) for all of that unit's segments.  Per step it streams the
// propagation matrix through shared memory in 32-wide k chunks of A (A = M
// going forward, M^T in reverse), keeps the state tile in shared memory, and
// each of its 256 threads accumulates R x 4 outputs (R = K / 32 rows spaced 32
// apart, 4 adjacent columns) in registers.  The chunks go through a ring of
// NST stages filled with cp.async NST - 1 chunks ahead, across step boundaries
// too (M does not depend on the state), so a chunk's global latency overlaps
// the arithmetic of the chunks before it.  NST is 8 for K <= 64, where a step
// has only one or two chunks and their latency dominates (config of 1 head,
// K = V = 64, S = 4: 8.92 -> 8.56 us per call), and 2 above: at K = 128 with
// 32 heads five stages measured up to 9 % slower (the larger shared-memory
// carve-out leaves less L1 to the 4-byte cp.async copies and the H loads).
//
// In-place (out == H): a thread reads its H_seg elements before it writes
// out[seg] over the same addresses, and no other thread touches them.
#include "qla_internal.h"

namespace qla {
namespace {

constexpr int kThreads = 256;
constexpr int kTileV = 32;
constexpr int kXsLd = kTileV + 4;  // padded row of the state tile (bank spread, keeps float4 alignment)

__device__ __forceinline__ int64_t state_index(int layout, int K, int V, int k, int v) {
  return layout == 0 ? (int64_t)k * V + v : (int64_t)v * K + k;
}

__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Floats of one chunk stage: forward [K rows m][33] (row m of A, 32 k + pad),
// reverse [32 rows k][K + 1] (row k of M = column of A, + pad).  Both pads keep
// the compute's shared loads free of bank conflicts.
template <int K>
__host__ __device__ constexpr int stage_floats() {
  return K * 33 > 32 * (K + 1) ? K * 33 : 32 * (K + 1);
}

// Ring stages for K (75 KB of shared memory at most, with the state tile).
template <int K>
__host__ __device__ constexpr int ring_stages() {
  return K <= 64 ? 8 : 2;
}

template <int R, int LAYOUT>
__global__ void __launch_bounds__(kThreads) seq_simt_kernel(const SeqJob j) {
  constexpr int K = R * 32;
  constexpr int CH = K / 32;  // chunks per step
  constexpr int SF = stage_floats<K>();
  constexpr int NST = ring_stages<K>();  // ring stages
  constexpr int D = NST - 1;             // chunks in flight ahead of the one in use
  extern __shared__ __align__(16) float smem[];
  float* Xs = smem;                 // [K][kXsLd]    state tile, kv view
  float* As = smem + K * kXsLd;     // [NST][SF]     chunk ring

  const int t = threadIdx.x;
  // kv: 8 column groups across a warp, so float4 global accesses along v coalesce.
  // vk: 32 consecutive rows across a warp, so scalar global accesses along k coalesce.
  const int cg = LAYOUT == 0 ? (t & 7) : (t >> 5);
  const int rg = LAYOUT == 0 ? (t >> 3) : (t & 31);
  const int V = j.V;
  int u, tile;
  if (!unit_and_tile(j, u, tile)) return;
  const int v0 = tile * kTileV + cg * 4;

  const int chain = u / j.G;
  const int g = u - chain * j.G;
  int64_t cbase;  // the chain's first segment in the packed arrays
  int S;
  griddep_wait();  // (before the first global access: the offsets may be the previous kernel's output)
  if (!chain_span(j, chain, cbase, S)) return;
  const int s_lo = g * j.L;
  const int n = min(j.L, S - s_lo);
  const int64_t st = (int64_t)K * V;
  const bool fwd = j.direction == 0;

  const float* Hc = j.H ? j.H + cbase * st : nullptr;
  float* Oc = j.out ? j.out + cbase * st : nullptr;
  const float* Mc = j.M + cbase * K * K;

  float x[R][4];
#pragma unroll
  for (int q = 0; q < R; ++q) {
    const int k = rg + 32 * q;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      float val = 0.f;
      if (j.init_mode == kInitPointer)
        val = j.init[u * j.init_unit_stride + state_index(LAYOUT, K, V, k, v0 + e)];
      else if (j.init_mode == kInitIdentity)
        val = (k == v0 + e) ? 1.f : 0.f;
      x[q][e] = val;
    }
  }

  const int nsteps = n - 1 + (j.fin ? 1 : 0);
  const int total = nsteps > 0 ? nsteps * CH : 0;  // chunks over all steps
  auto seg_of = [&](int jj) { return fwd ? s_lo + jj : s_lo + n - 1 - jj; };
  // Chunk c (step c / CH, k block c % CH) -> stage c % NST, one 4-byte cp.async
  // per element: forward A[m][kc + kk] = M[m][kc + kk], reverse A[m][kc + kk] =
  // M[kc + kk][m]; consecutive threads read consecutive global floats.
  auto issue_chunk = [&](int c) {
    const float* Ms = Mc + (int64_t)seg_of(c / CH) * K * K;
    const int kc = (c % CH) * 32;
    float* dst = As + (c % NST) * SF;
    for (int e = t; e < 32 * K; e += kThreads) {
      if (fwd) {
        const int m = e >> 5, kk = e & 31;
        cp_async4(dst + m * 33 + kk, Ms + (int64_t)m * K + kc + kk);
      } else {
        const int kk = e / K, m = e - kk * K;
        cp_async4(dst + kk * (K + 1) + m, Ms + (int64_t)(kc + kk) * K + m);
      }
    }
  };
  // One commit group per chunk, empty past the last: D groups ahead of the loop.
#pragma unroll
  for (int c = 0; c < D; ++c) {
    if (c < total) issue_chunk(c);
    cp_async_commit();
  }

  for (int jj = 0; jj < n; ++jj) {
    const int seg = seg_of(jj);
    const bool do_step = jj < nsteps;
    float h[R][4];
#pragma unroll
    for (int q = 0; q < R; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) h[q][e] = 0.f;
    if (do_step && Hc) {
      const float* Hs = Hc + seg * st;
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const int k = rg + 32 * q;
        if (LAYOUT == 0) {
          const float4 hv = *reinterpret_cast<const float4*>(Hs + (int64_t)k * V + v0);
          h[q][0] = hv.x; h[q][1] = hv.y; h[q][2] = hv.z; h[q][3] = hv.w;
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) h[q][e] = Hs[(int64_t)(v0 + e) * K + k];
        }
      }
    }
    if (Oc) {
      float* Os = Oc + seg * st;
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const int k = rg + 32 * q;
        if (LAYOUT == 0) {
          *reinterpret_cast<float4*>(Os + (int64_t)k * V + v0) = make_float4(x[q][0], x[q][1], x[q][2], x[q][3]);
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) Os[(int64_t)(v0 + e) * K + k] = x[q][e];
        }
      }
    }
    if (!do_step) break;

    __syncthreads();  // the previous step's readers of Xs are done
#pragma unroll
    for (int q = 0; q < R; ++q)
      *reinterpret_cast<float4*>(Xs + (rg + 32 * q) * kXsLd + cg * 4) =
          make_float4(x[q][0], x[q][1], x[q][2], x[q][3]);

    float acc[R][4];
#pragma unroll
    for (int q = 0; q < R; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[q][e] = 0.f;

    for (int kb = 0; kb < CH; ++kb) {
      const int c = jj * CH + kb;
      __syncthreads();  // every thread is done with chunk c - 1, whose stage chunk c + D reuses; Xs written
      if (c + D < total) issue_chunk(c + D);
      cp_async_commit();
      cp_async_wait<D>();  // this thread's copies of chunk c have landed
      __syncthreads();     // everyone's have
      const float* A = As + (c % NST) * SF;
      const int kc = kb * 32;
#pragma unroll 8
      for (int kk = 0; kk < 32; ++kk) {
        const float4 xv = *reinterpret_cast<const float4*>(Xs + (kc + kk) * kXsLd + cg * 4);
#pragma unroll
        for (int q = 0; q < R; ++q) {
          const float a = fwd ? A[(rg + 32 * q) * 33 + kk] : A[kk * (K + 1) + rg + 32 * q];
          acc[q][0] = fmaf(a, xv.x, acc[q][0]);
          acc[q][1] = fmaf(a, xv.y, acc[q][1]);
          acc[q][2] = fmaf(a, xv.z, acc[q][2]);
          acc[q][3] = fmaf(a, xv.w, acc[q][3]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < R; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[q][e] = acc[q][e] + h[q][e];
  }
  cp_async_wait<0>();  // no copy may land after the CTA is gone
  griddep_launch_dependents();

  if (j.fin) {
    float* F = j.fin + u * j.fin_unit_stride;
#pragma unroll
    for (int q = 0; q < R; ++q) {
      const int k = rg + 32 * q;
#pragma unroll
      for (int e = 0; e < 4; ++e) F[state_index(LAYOUT, K, V, k, v0 + e)] = x[q][e];
    }
  }
}

template <int R, int LAYOUT>
cudaError_t launch_one(const SeqJob& j, cudaStream_t stream) {
  constexpr int K = R * 32;
  const size_t smem = sizeof(float) * ((size_t)K * kXsLd + (size_t)ring_stages<K>() * stage_floats<K>());
  auto kern = seq_simt_kernel<R, LAYOUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid = job_grid(j, j.V / kTileV);
  e = launch_kernel(kern, grid, kThreads, smem, stream, j.pdl != 0, j);
  return e != cudaSuccess ? e : cudaGetLastError();
}

template <int LAYOUT>
cudaError_t dispatch_r(const SeqJob& j, cudaStream_t s) {
  switch (j.K / 32) {
    case 1: return launch_one<1, LAYOUT>(j, s);
    case 2: return launch_one<2, LAYOUT>(j, s);
    case 3: return launch_one<3, LAYOUT>(j, s);
    case 4: return launch_one<4, LAYOUT>(j, s);
    case 5: return launch_one<5, LAYOUT>(j, s);
    case 6: return launch_one<6, LAYOUT>(j, s);
    case 7: return launch_one<7, LAYOUT>(j, s);
    case 8: return launch_one<8, LAYOUT>(j, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

cudaError_t launch_seq_simt(const SeqJob& job, cudaStream_t stream) {
  if (job.K % 32 || job.K < 32 || job.K > 256 || job.V % kTileV) return cudaErrorInvalidValue;
  if (job_grid(job, job.V / kTileV).x == 0) return cudaErrorInvalidValue;
  return job.layout == 0 ? dispatch_r<0>(job, stream) : dispatch_r<1>(job, stream);
}

}  // namespace qla
