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
// each of its 256 threads accumulates R x 4 outputs (R = K / 32 consecutive
// rows, 4 adjacent columns) in registers.  A reverse chunk is stored k-major,
// so per k a thread reads its R values of A and its 4 of the state with vector
// loads; a forward chunk is stored m-major (16-byte copies of M's rows either
// way), read as R rows x 4 k per step of four k.
// The chunks go through a ring of three stages filled with cp.async two
// chunks ahead, across step boundaries too (M does not depend on the state),
// so a chunk's global latency overlaps the arithmetic of the two chunks before
// it; one barrier per chunk hands a landed chunk to every thread and frees the
// stage of the chunk before.  This form serves K > 128; K <= 128 runs the
// k-split form below.  At K = V = 256 (32 heads, S = 8) three stages with one
// barrier per chunk measured 252.5 / 211.4 us forward / reverse against
// 262.8 / 221.7 for two stages with two barriers per chunk.
//
// In-place (out == H): a thread reads its H_seg elements before it writes
// out[seg] over the same addresses, and no other thread touches them.
#include "qla_internal.h"

namespace qla {
namespace {

constexpr int kThreads = 256;
constexpr int kTileV = 32;
constexpr int kXsLd = kTileV + 4;  // padded row of the state tile (bank spread, keeps float4 alignment)

__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async16(float* dst, const float* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
               "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// A reverse chunk stage holds A[m][kc + kk] = M[kc + kk][m] k-major, as
// [32 rows kk][K + 4]: a thread's R consecutive rows m of one kk are adjacent,
// so the compute reads them with vector loads; the 4-float pad keeps those
// loads 16-byte aligned.
template <int K>
__host__ __device__ constexpr int stage_ld() {
  return K + 4;
}
// A forward stage holds A[m][kc + kk] = M[m][kc + kk] m-major instead: K rows
// of the chunk's 32 k, padded to 36 (both copies are 16-byte copies of M's
// rows, no transposition on the way in).
constexpr int kStageMLd = 36;
template <int K>
__host__ __device__ constexpr int stage_floats() {
  return 32 * stage_ld<K>() > K * kStageMLd ? 32 * stage_ld<K>() : K * kStageMLd;
}

// R consecutive floats from / to p (aligned to 4 R bytes): float4 pieces when
// R is a multiple of 4, float2 when even, scalars otherwise.
template <int R>
__device__ __forceinline__ void load_run(const float* p, float (&a)[R]) {
  if constexpr (R % 4 == 0) {
#pragma unroll
    for (int i = 0; i < R; i += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + i);
      a[i] = v.x; a[i + 1] = v.y; a[i + 2] = v.z; a[i + 3] = v.w;
    }
  } else if constexpr (R % 2 == 0) {
#pragma unroll
    for (int i = 0; i < R; i += 2) {
      const float2 v = *reinterpret_cast<const float2*>(p + i);
      a[i] = v.x; a[i + 1] = v.y;
    }
  } else {
#pragma unroll
    for (int i = 0; i < R; ++i) a[i] = p[i];
  }
}
template <int R>
__device__ __forceinline__ void store_run(float* p, const float (&a)[R]) {
  if constexpr (R % 4 == 0) {
#pragma unroll
    for (int i = 0; i < R; i += 4) *reinterpret_cast<float4*>(p + i) = make_float4(a[i], a[i + 1], a[i + 2], a[i + 3]);
  } else if constexpr (R % 2 == 0) {
#pragma unroll
    for (int i = 0; i < R; i += 2) *reinterpret_cast<float2*>(p + i) = make_float2(a[i], a[i + 1]);
  } else {
#pragma unroll
    for (int i = 0; i < R; ++i) p[i] = a[i];
  }
}

// Ring stages: three, so two chunks are in flight while one is in use (at
// K = 256, 108 KB of ring plus the 36 KB state tile; one CTA per SM).
template <int K>
__host__ __device__ constexpr int ring_stages() {
  return 3;
}

template <int R, int LAYOUT>
__global__ void __launch_bounds__(kThreads, 1) seq_simt_kernel(const SeqJob j) {
  constexpr int K = R * 32;
  constexpr int CH = K / 32;  // chunks per step
  constexpr int SL = stage_ld<K>();
  constexpr int SF = stage_floats<K>();
  constexpr int NST = ring_stages<K>();  // ring stages
  constexpr int D = NST - 1;             // chunks in flight ahead of the one in use
  extern __shared__ __align__(16) float smem[];
  float* Xs = smem;                 // [K][kXsLd]    state tile, kv view
  float* As = smem + K * kXsLd;     // [NST][SF]     chunk ring

  // Thread t owns rows R rg .. R rg + R - 1 and columns 4 cg .. 4 cg + 3 of
  // the 32-column tile: 8 column groups across a warp, so kv global accesses
  // are float4 runs along v; vk ones are runs of R along k.
  const int t = threadIdx.x;
  const int cg = t & 7;
  const int rg = t >> 3;
  const int k0 = R * rg;
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

  // This thread's R x 4 block of a state (k-major in registers) from / to a
  // [K][V] (kv) or [V][K] (vk) array.
  auto load_block = [&](const float* src, float (&b)[R][4]) {
    if (LAYOUT == 0) {
#pragma unroll
      for (int q = 0; q < R; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(src + (int64_t)(k0 + q) * V + v0);
        b[q][0] = v.x; b[q][1] = v.y; b[q][2] = v.z; b[q][3] = v.w;
      }
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float r[R];
        load_run<R>(src + (int64_t)(v0 + e) * K + k0, r);
#pragma unroll
        for (int q = 0; q < R; ++q) b[q][e] = r[q];
      }
    }
  };
  auto store_block = [&](float* dst, const float (&b)[R][4]) {
    if (LAYOUT == 0) {
#pragma unroll
      for (int q = 0; q < R; ++q)
        *reinterpret_cast<float4*>(dst + (int64_t)(k0 + q) * V + v0) = make_float4(b[q][0], b[q][1], b[q][2], b[q][3]);
    } else {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float r[R];
#pragma unroll
        for (int q = 0; q < R; ++q) r[q] = b[q][e];
        store_run<R>(dst + (int64_t)(v0 + e) * K + k0, r);
      }
    }
  };

  float x[R][4];
  if (j.init_mode == kInitPointer) {
    load_block(j.init + u * j.init_unit_stride, x);
  } else {
#pragma unroll
    for (int q = 0; q < R; ++q)
#pragma unroll
      for (int e = 0; e < 4; ++e) x[q][e] = (j.init_mode == kInitIdentity && k0 + q == v0 + e) ? 1.f : 0.f;
  }

  const int nsteps = n - 1 + (j.fin ? 1 : 0);
  const int total = nsteps > 0 ? nsteps * CH : 0;  // chunks over all steps
  auto seg_of = [&](int jj) { return fwd ? s_lo + jj : s_lo + n - 1 - jj; };
  // Chunk c (step c / CH, k block c % CH) -> stage c % NST, with 16-byte
  // cp.async copies of M's rows either way.  Reverse: A[m][kc + kk] =
  // M[kc + kk][m], kept k-major as [kk][m].  Forward: A[m][kc + kk] =
  // M[m][kc + kk], kept m-major as [m][kk] (rows of kStageMLd); the compute
  // then reads R rows x 4 k per step of four k.
  auto issue_chunk = [&](int c) {
    const float* Ms = Mc + (int64_t)seg_of(c / CH) * K * K;
    const int kc = (c % CH) * 32;
    float* dst = As + (c % NST) * SF;
    if (fwd) {  // m-major: row m holds A[m][kc .. kc + 32), 16-byte copies of M's rows
      for (int e = t; e < 8 * K; e += kThreads) {
        const int m = e >> 3, p4 = 4 * (e & 7);
        cp_async16(dst + m * kStageMLd + p4, Ms + (int64_t)m * K + kc + p4);
      }
    } else {  // k-major: row kk holds M[kc + kk][0 .. K), 16-byte copies
      for (int e = t; e < 8 * K; e += kThreads) {
        const int kk = e / (K / 4), m4 = 4 * (e - kk * (K / 4));
        cp_async16(dst + kk * SL + m4, Ms + (int64_t)(kc + kk) * K + m4);
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
    if (do_step && Hc) {
      load_block(Hc + seg * st, h);
    } else {
#pragma unroll
      for (int q = 0; q < R; ++q)
#pragma unroll
        for (int e = 0; e < 4; ++e) h[q][e] = 0.f;
    }
    if (Oc) store_block(Oc + seg * st, x);
    if (!do_step) break;

    __syncthreads();  // the previous step's readers of Xs are done
#pragma unroll
    for (int q = 0; q < R; ++q)
      *reinterpret_cast<float4*>(Xs + (k0 + q) * kXsLd + cg * 4) = make_float4(x[q][0], x[q][1], x[q][2], x[q][3]);

    // acc[q][p] holds columns 2p, 2p + 1 of row q: packed fma.rn.f32x2, each
    // half rounded as a scalar FMA
    float2 acc[R][2];
#pragma unroll
    for (int q = 0; q < R; ++q) acc[q][0] = acc[q][1] = make_float2(0.f, 0.f);

    for (int kb = 0; kb < CH; ++kb) {
      const int c = jj * CH + kb;
      // D + c groups are committed, chunk c's is the (c + 1)-th: with D - 1
      // pending, this thread's copies of chunk c have landed.
      cp_async_wait<D - 1>();
      // Everyone's have, Xs is written, and every thread is done with chunk
      // c - 1, whose stage chunk c + D reuses.
      __syncthreads();
      if (c + D < total) issue_chunk(c + D);
      cp_async_commit();
      const int kc = kb * 32;
      if (fwd) {  // m-major stage: R rows x 4 k per step of four k
        const float* Am = As + (c % NST) * SF + k0 * kStageMLd;
#pragma unroll 2
        for (int kk4 = 0; kk4 < 32; kk4 += 4) {
          float4 a4[R];
#pragma unroll
          for (int q = 0; q < R; ++q) a4[q] = *reinterpret_cast<const float4*>(Am + q * kStageMLd + kk4);
#pragma unroll
          for (int j4 = 0; j4 < 4; ++j4) {
            const float4 xv = *reinterpret_cast<const float4*>(Xs + (kc + kk4 + j4) * kXsLd + cg * 4);
            const float2 x01 = make_float2(xv.x, xv.y), x23 = make_float2(xv.z, xv.w);
#pragma unroll
            for (int q = 0; q < R; ++q) {
              const float a = j4 == 0 ? a4[q].x : j4 == 1 ? a4[q].y : j4 == 2 ? a4[q].z : a4[q].w;
              const float2 aq = make_float2(a, a);
              acc[q][0] = __ffma2_rn(aq, x01, acc[q][0]);
              acc[q][1] = __ffma2_rn(aq, x23, acc[q][1]);
            }
          }
        }
        continue;
      }
      const float* A = As + (c % NST) * SF + k0;
#pragma unroll 8
      for (int kk = 0; kk < 32; ++kk) {
        const float4 xv = *reinterpret_cast<const float4*>(Xs + (kc + kk) * kXsLd + cg * 4);
        const float2 x01 = make_float2(xv.x, xv.y), x23 = make_float2(xv.z, xv.w);
        float a[R];
        load_run<R>(A + kk * SL, a);  // A[k0 .. k0 + R - 1][kc + kk]
#pragma unroll
        for (int q = 0; q < R; ++q) {
          const float2 aq = make_float2(a[q], a[q]);
          acc[q][0] = __ffma2_rn(aq, x01, acc[q][0]);
          acc[q][1] = __ffma2_rn(aq, x23, acc[q][1]);
        }
      }
    }
#pragma unroll
    for (int q = 0; q < R; ++q) {
      x[q][0] = acc[q][0].x + h[q][0];
      x[q][1] = acc[q][0].y + h[q][1];
      x[q][2] = acc[q][1].x + h[q][2];
      x[q][3] = acc[q][1].y + h[q][3];
    }
  }
  cp_async_wait<0>();  // no copy may land after the CTA is gone
  griddep_launch_dependents();

  if (j.fin) store_block(j.fin + u * j.fin_unit_stride, x);
}

// ---------------------------------------------------------------- k-split form (K <= 128)
//
// The same recurrence with the contraction split four ways: 2K threads in
// four k-groups of K/2; a thread of k-group g computes an 8-row x 8-column
// block of sum over k in [g K/4, (g+1) K/4) of A[m][k] X[k][v], so every value
// it reads from shared memory feeds four FMAs (the R x 4 tiles above feed two;
// at K = 128 those make the shared-memory reads, not the FMAs, the bound).
// The four partial blocks meet in shared memory once per step, where the
// thread that owns an output (a row and 16 columns) adds them and H.  A step's
// whole A (K x K, k-major) is copied in with cp.async during the step before.
constexpr int kKG = 4;          // k-groups
constexpr int kPld = kTileV + 4;  // padded row of the state tile

// Partial blocks are [kKG][K][kPld] (padded rows, so consecutive rows start in
// different banks) with the two 16-byte groups of each pair swapped in odd
// 8-row blocks: a warp's writes (8-row blocks of 8 columns, two row blocks
// per quarter-warp) and the owners' reads (one row, 16 columns) then fall in
// distinct banks.
__device__ __forceinline__ int pidx(int row, int col) {
  return row * kPld + ((((col >> 2) ^ (row >> 3)) & 1) | ((col >> 2) & 6)) * 4 + (col & 3);
}

// Forward A (= M) is kept m-major, A[m][k] in row m, with the 16-byte chunks of
// odd 8-row blocks swapped in pairs: the two row blocks a quarter-warp reads
// then fall in different banks (rows a multiple of 16 bytes apart would not).
template <int AL>
__device__ __forceinline__ int amx(int m, int k) {
  return m * AL + ((((k >> 2) ^ (m >> 3)) & 1) | ((k >> 2) & ~1)) * 4 + (k & 3);
}

template <int K>
__host__ __device__ constexpr int ks_threads() {
  return 2 * K;
}
template <int K>
__host__ __device__ constexpr int ks_ald() {
  return K + 4;  // padded row (one k) of the A copy
}
template <int K>
__host__ __device__ constexpr size_t ks_smem_floats() {
  // state tile [K][kPld] + two A copies [K][K + 4] + partials [kKG][K][kPld]
  return (size_t)K * kPld + 2 * (size_t)K * ks_ald<K>() + (size_t)kKG * K * kPld;
}

template <int K, int LAYOUT>
__global__ void __launch_bounds__(2 * K) seq_simt_ksplit_kernel(const SeqJob j) {
  constexpr int NT = ks_threads<K>();
  constexpr int KR = K / kKG;    // k per group
  constexpr int AL = ks_ald<K>();
  extern __shared__ __align__(16) float smem[];
  float* Xs = smem;                      // [K][kPld]   state tile, kv view
  float* As0 = Xs + K * kPld;            // [2][K][AL]  A copies, As[k][m] = A[m][k]
  float* Ps = As0 + 2 * K * AL;          // [kKG][K][kPld] partial blocks (pidx)

  const int t = threadIdx.x;
  const int kg = t / (K / 2);            // k-group
  const int w = t - kg * (K / 2);
  const int rb = w >> 2, cb = w & 3;     // 8-row block, 8-column block
  // owner of outputs: one row and 16 columns (kv: lanes pair up along a row;
  // vk: lanes run down a column, so global accesses are runs along k)
  const int orow = LAYOUT == 0 ? (t >> 1) : (t % K);
  const int oc0 = LAYOUT == 0 ? (t & 1) * 16 : (t / K) * 16;
  const int V = j.V;
  int u, tile;
  if (!unit_and_tile(j, u, tile)) return;
  const int vt = tile * kTileV;          // the tile's first column
  const int chain = u / j.G;
  const int g = u - chain * j.G;
  int64_t cbase;
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

  // this thread's owned outputs of a [K][V] (kv) or [V][K] (vk) state
  auto load_own = [&](const float* src, float (&b)[16]) {
    if (LAYOUT == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float4 v = *reinterpret_cast<const float4*>(src + (int64_t)orow * V + vt + oc0 + 4 * q);
        b[4 * q] = v.x; b[4 * q + 1] = v.y; b[4 * q + 2] = v.z; b[4 * q + 3] = v.w;
      }
    } else {
#pragma unroll
      for (int c = 0; c < 16; ++c) b[c] = src[(int64_t)(vt + oc0 + c) * K + orow];
    }
  };
  auto store_own = [&](float* dst, const float (&b)[16]) {
    if (LAYOUT == 0) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<float4*>(dst + (int64_t)orow * V + vt + oc0 + 4 * q) =
            make_float4(b[4 * q], b[4 * q + 1], b[4 * q + 2], b[4 * q + 3]);
    } else {
#pragma unroll
      for (int c = 0; c < 16; ++c) dst[(int64_t)(vt + oc0 + c) * K + orow] = b[c];
    }
  };
  auto put_state = [&](const float (&b)[16]) {
#pragma unroll
    for (int q = 0; q < 4; ++q)
      *reinterpret_cast<float4*>(Xs + orow * kPld + oc0 + 4 * q) =
          make_float4(b[4 * q], b[4 * q + 1], b[4 * q + 2], b[4 * q + 3]);
  };

  float x[16];
  if (j.init_mode == kInitPointer) {
    load_own(j.init + u * j.init_unit_stride, x);
  } else {
#pragma unroll
    for (int c = 0; c < 16; ++c) x[c] = (j.init_mode == kInitIdentity && orow == vt + oc0 + c) ? 1.f : 0.f;
  }
  const int nsteps = n - 1 + (j.fin ? 1 : 0);
  auto seg_of = [&](int jj) { return fwd ? s_lo + jj : s_lo + n - 1 - jj; };
  // A of step jj into copy jj & 1, with 16-byte copies of M's rows either
  // way: reverse A = M^T is kept k-major, As[k][m] = M[k][m]; forward A = M is
  // kept m-major, As[m][k] = M[m][k] (amx).
  auto issue_a = [&](int jj) {
    const float* Ms = Mc + (int64_t)seg_of(jj) * K * K;
    float* dst = As0 + (jj & 1) * K * AL;
    if (fwd) {
      for (int e = t; e < K * K / 4; e += NT) {
        const int m = e / (K / 4), k4 = 4 * (e - m * (K / 4));
        cp_async16(dst + amx<AL>(m, k4), Ms + (int64_t)m * K + k4);
      }
    } else {
      for (int e = t; e < K * K / 4; e += NT) {
        const int k = e / (K / 4), m4 = e - k * (K / 4);
        cp_async16(dst + k * AL + 4 * m4, Ms + (int64_t)k * K + 4 * m4);
      }
    }
    cp_async_commit();
  };
  if (nsteps > 0) issue_a(0);
  // vk: H of the next step is read one step ahead (its owners' reads are
  // K-strided, so their latency is long), under the current step's FMAs.  In
  // place (out == H): each thread reads its H_seg elements before it writes
  // out[seg] over the same addresses; no other thread touches them.
  float hn[16];
  if (LAYOUT == 1 && nsteps > 0 && Hc) {
    load_own(Hc + seg_of(0) * st, hn);
  } else {
#pragma unroll
    for (int c = 0; c < 16; ++c) hn[c] = 0.f;
  }

  for (int jj = 0; jj < n; ++jj) {
    const int seg = seg_of(jj);
    const bool do_step = jj < nsteps;
    float h[16];
    if (LAYOUT == 1) {
#pragma unroll
      for (int c = 0; c < 16; ++c) h[c] = hn[c];
    } else if (do_step && Hc) {
      load_own(Hc + seg * st, h);
    } else {
#pragma unroll
      for (int c = 0; c < 16; ++c) h[c] = 0.f;
    }
    if (Oc) store_own(Oc + seg * st, x);
    if (!do_step) break;
    if (LAYOUT == 1 && jj + 1 < nsteps && Hc) load_own(Hc + seg_of(jj + 1) * st, hn);
    put_state(x);
    cp_async_wait<0>();  // this thread's copies of step jj's A have landed
    // Everyone's have, and the state tile is written.  Every thread is also past
    // step jj-1: done with copy (jj+1)&1 (refilled next) and with its reads of
    // the partial blocks (rewritten after this step's FMAs), so one barrier
    // covers both hand-overs.
    __syncthreads();
    if (jj + 1 < nsteps) issue_a(jj + 1);

    // acc[r][p] holds columns 2p, 2p + 1 of row r: packed fma.rn.f32x2, each
    // half rounded as a scalar FMA, half the FMA instructions
    float2 acc[8][4];
#pragma unroll
    for (int r = 0; r < 8; ++r)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[r][c] = make_float2(0.f, 0.f);
    const float* X = Xs + kg * KR * kPld + cb * 8;
    if (fwd) {  // A m-major: 8 rows x 4 k per step of four k
      const float* Am = As0 + (jj & 1) * K * AL;
#pragma unroll
      for (int k4 = 0; k4 < KR; k4 += 4) {
        float4 ar[8];
#pragma unroll
        for (int r = 0; r < 8; ++r) ar[r] = *reinterpret_cast<const float4*>(Am + amx<AL>(rb * 8 + r, kg * KR + k4));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const float4 x0 = *reinterpret_cast<const float4*>(X + (k4 + kk) * kPld);
          const float4 x1 = *reinterpret_cast<const float4*>(X + (k4 + kk) * kPld + 4);
          const float2 xp[4] = {make_float2(x0.x, x0.y), make_float2(x0.z, x0.w), make_float2(x1.x, x1.y),
                                make_float2(x1.z, x1.w)};
#pragma unroll
          for (int r = 0; r < 8; ++r) {
            const float a = kk == 0 ? ar[r].x : kk == 1 ? ar[r].y : kk == 2 ? ar[r].z : ar[r].w;
            const float2 ap = make_float2(a, a);
#pragma unroll
            for (int c = 0; c < 4; ++c) acc[r][c] = __ffma2_rn(ap, xp[c], acc[r][c]);
          }
        }
      }
    } else {  // A k-major: 8 rows of one k per step
    const float* A = As0 + (jj & 1) * K * AL + kg * KR * AL + rb * 8;
#pragma unroll
    for (int k = 0; k < KR; ++k) {
      const float4 a0 = *reinterpret_cast<const float4*>(A + k * AL);
      const float4 a1 = *reinterpret_cast<const float4*>(A + k * AL + 4);
      const float4 x0 = *reinterpret_cast<const float4*>(X + k * kPld);
      const float4 x1 = *reinterpret_cast<const float4*>(X + k * kPld + 4);
      const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
      const float2 xp[4] = {make_float2(x0.x, x0.y), make_float2(x0.z, x0.w), make_float2(x1.x, x1.y),
                            make_float2(x1.z, x1.w)};
#pragma unroll
      for (int r = 0; r < 8; ++r) {
        const float2 ar = make_float2(av[r], av[r]);
#pragma unroll
        for (int c = 0; c < 4; ++c) acc[r][c] = __ffma2_rn(ar, xp[c], acc[r][c]);
      }
    }
    }
    // partial blocks -> shared memory; the owners add them (k-groups in order) and H
    float* P = Ps + kg * K * kPld;
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      *reinterpret_cast<float4*>(P + pidx(rb * 8 + r, cb * 8)) =
          make_float4(acc[r][0].x, acc[r][0].y, acc[r][1].x, acc[r][1].y);
      *reinterpret_cast<float4*>(P + pidx(rb * 8 + r, cb * 8 + 4)) =
          make_float4(acc[r][2].x, acc[r][2].y, acc[r][3].x, acc[r][3].y);
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int pi = pidx(orow, oc0 + 4 * q);
      float4 sum = *reinterpret_cast<const float4*>(Ps + pi);
#pragma unroll
      for (int gg = 1; gg < kKG; ++gg) {
        const float4 p = *reinterpret_cast<const float4*>(Ps + gg * K * kPld + pi);
        sum.x += p.x; sum.y += p.y; sum.z += p.z; sum.w += p.w;
      }
      x[4 * q] = sum.x + h[4 * q];
      x[4 * q + 1] = sum.y + h[4 * q + 1];
      x[4 * q + 2] = sum.z + h[4 * q + 2];
      x[4 * q + 3] = sum.w + h[4 * q + 3];
    }
  }
  cp_async_wait<0>();  // no copy may land after the CTA is gone
  griddep_launch_dependents();
  if (j.fin) store_own(j.fin + u * j.fin_unit_stride, x);
}

template <int K, int LAYOUT>
cudaError_t launch_ksplit(const SeqJob& j, cudaStream_t stream) {
  const size_t smem = sizeof(float) * ks_smem_floats<K>();
  auto kern = seq_simt_ksplit_kernel<K, LAYOUT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const dim3 grid = job_grid(j, j.V / kTileV);
  e = launch_kernel(kern, grid, ks_threads<K>(), smem, stream, j.pdl != 0, j);
  return e != cudaSuccess ? e : cudaGetLastError();
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
    case 1: return launch_ksplit<32, LAYOUT>(j, s);
    case 2: return launch_ksplit<64, LAYOUT>(j, s);
    case 3: return launch_ksplit<96, LAYOUT>(j, s);
    case 4: return launch_ksplit<128, LAYOUT>(j, s);
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
