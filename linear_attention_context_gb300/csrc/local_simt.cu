// Per-segment local pass: the inputs (H_i, M_i) of the context-parallel state
// correction, computed from token-level keys, values, write strengths and
// decays.  Antarx Memos, "一次 TileLang Warp Specialization 数值错误的定位与修复：
// 从双缓冲竞争到 membar", section "从版本升级后的数值偏差开始", names the two
// per-segment quantities (the local state "ht" and the propagation matrix
// "mt") without defining them; the reading implemented here is the token
// recurrence of the gated delta rule (Yang, Kautz, Hatamizadeh, "Gated Delta
// Networks: Improving Mamba2 with Delta Rule", ICLR 2025) in the kv view:
//
//     X_t = a_t (I - b_t k_t k_t^T) X_{t-1} + b_t k_t v_t^T,   a_t = exp(g_t)
//
// and for each segment of L tokens H = the state after its tokens from zero,
// M = A_last ... A_first with A_t = a_t (I - b_t k_t k_t^T), so that the state
// leaving a segment is M X_enter + H -- the recurrence the correction composes.
//
// Work split.  The columns of Y = [H | M] (V columns of the local state, K of
// the propagation matrix, which starts at the identity) evolve independently
// under the same left multiplications, so each warp owns a block of columns of
// one segment for the whole segment: a lane holds R rows x NC columns in
// registers and G = K / R lanes share a column group (the dot product k^T Y is
// a partial sum per lane, then a shuffle reduction over those G lanes).  Per
// token and lane: NC R FMAs for the dot products and NC R for the update, as
// packed two-row FMAs (fma.rn.f32x2: each half rounds as a scalar FMA would);
// every key value read from shared memory (a broadcast) feeds NC FMAs.  No
// synchronisation between tokens.
//
// Decay as a scale.  Y = s Yhat with s = exp(sum of g since a reference
// token), so the update is Yhat += k c^T with c = b (v / s - d), d = k^T Yhat:
// the decays never multiply the state element by element, so their fp32
// roundings do not compound over the segment.  The running log-decay sum is
// kept in fp64 by the staging warp; 1 / s per token comes from it in fp32 (exp
// of the high part, corrected to first order by the low part).  When the sum
// has moved more than 16 away from the reference at some token, the state is
// rescaled by s once, before that token's update, and the reference moves there.
//
// Staging.  Tokens go through shared memory in tiles of kTT: keys and values
// widened from bf16 to fp32, write strengths, 1 / s and the rescale factors.
// The next tile's raw inputs are copied in (cp.async) while the current tile
// computes; widening them is a shared-to-shared pass at the tile's start.
#include <cuda_runtime.h>
#include <stdint.h>

#include "qla_internal.h"

namespace qla {
namespace {

constexpr int kLocalWarps = 4;
constexpr int kLocalThreads = 32 * kLocalWarps;
constexpr int kTT = 32;              // tokens per staged tile (one per lane of the staging warp)
constexpr double kRescaleLog = 16.0;  // rescale when |log s| would exceed this

struct LocalParams {
  LocalJob j;
  int col_begin;     // first column of Y = [H | M] computed (0, or V when H is not wanted)
  int col_end;       // one past the last (V when M is not wanted, else V + K)
  int cols_per_cta;  // columns of Y per CTA
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// exp(x) for an fp64 x: exp of the fp32 high part times (1 + the low part).
__device__ __forceinline__ float exp_split(double x) {
  const float hi = (float)x;
  const float lo = (float)(x - (double)hi);
  return expf(hi) * (1.0f + lo);
}

__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async4(void* dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)), "l"(src)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }

// Issues the copies of a tile's raw inputs (bf16 keys and values, fp32 write
// strengths and log-decays) into shared memory.
__device__ __forceinline__ void issue_tile(const LocalJob& j, int64_t tok, int n, bool need_v, uint16_t* kraw,
                                           uint16_t* vraw, float* braw, float* graw) {
  const int kc = n * j.K / 8, vc = need_v ? n * j.V / 8 : 0;
  const uint4* ks = reinterpret_cast<const uint4*>(j.k + tok * j.K);
  const uint4* vs = reinterpret_cast<const uint4*>(j.v + tok * j.V);
  for (int i = threadIdx.x; i < kc; i += kLocalThreads) cp_async16(reinterpret_cast<uint4*>(kraw) + i, ks + i);
  for (int i = threadIdx.x; i < vc; i += kLocalThreads) cp_async16(reinterpret_cast<uint4*>(vraw) + i, vs + i);
  if (threadIdx.x < n) cp_async4(braw + threadIdx.x, j.beta + tok + threadIdx.x);
  else if (threadIdx.x >= 32 && threadIdx.x - 32 < n) cp_async4(graw + threadIdx.x - 32, j.g + tok + threadIdx.x - 32);
  cp_async_commit();
}

// Widens n rows of `width` bf16 values to fp32, shared memory to shared memory.
__device__ __forceinline__ void widen_rows(const uint16_t* src, float* dst, int n, int width) {
  const int total = n * width / 8;
  const uint4* s4 = reinterpret_cast<const uint4*>(src);
  float4* d4 = reinterpret_cast<float4*>(dst);
  for (int i = threadIdx.x; i < total; i += kLocalThreads) {
    const uint4 w = s4[i];
    d4[2 * i] = make_float4(bf16_lo(w.x), bf16_hi(w.x), bf16_lo(w.y), bf16_hi(w.y));
    d4[2 * i + 1] = make_float4(bf16_lo(w.z), bf16_hi(w.z), bf16_lo(w.w), bf16_hi(w.w));
  }
}

// Reduces a lane's partial dot products over the G lanes sharing its columns.
template <int CW, int NC>
__device__ __forceinline__ void reduce_parts(float (&d)[NC]) {
#pragma unroll
  for (int m = CW; m < 32; m <<= 1)
#pragma unroll
    for (int c = 0; c < NC; ++c) d[c] += __shfl_xor_sync(0xffffffffu, d[c], m);
}

// One pass over the registers: optionally Yhat += k_i c^T (token i's update),
// then optionally d = k_n^T Yhat (the next token's dot products, partial over
// this lane's rows); each key value read feeds NC FMAs per use.  The state is
// held as pairs of rows and every FMA is a packed fma.rn.f32x2 (two rows per
// instruction, each rounded as a scalar FMA): the pass issues half the
// instructions of scalar FMAs.
template <int R, int NC, bool UPD, bool DOT>
__device__ __forceinline__ void token_pass(float2 (&y)[NC][R / 2], const float* kc, const float (&cc)[NC],
                                           const float* kn, float (&d)[NC]) {
  float2 a[NC][2];
  float2 cp[NC];
#pragma unroll
  for (int c = 0; c < NC; ++c) {
    a[c][0] = a[c][1] = make_float2(0.f, 0.f);
    cp[c] = make_float2(cc[c], cc[c]);
  }
#pragma unroll
  for (int r = 0; r < R; r += 4) {
    if constexpr (UPD) {
      const float4 kk = *reinterpret_cast<const float4*>(kc + r);
      const float2 k01 = make_float2(kk.x, kk.y), k23 = make_float2(kk.z, kk.w);
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        y[c][r / 2] = __ffma2_rn(k01, cp[c], y[c][r / 2]);
        y[c][r / 2 + 1] = __ffma2_rn(k23, cp[c], y[c][r / 2 + 1]);
      }
    }
    if constexpr (DOT) {
      const float4 kq = *reinterpret_cast<const float4*>(kn + r);
      const float2 q01 = make_float2(kq.x, kq.y), q23 = make_float2(kq.z, kq.w);
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        a[c][0] = __ffma2_rn(q01, y[c][r / 2], a[c][0]);
        a[c][1] = __ffma2_rn(q23, y[c][r / 2 + 1], a[c][1]);
      }
    }
  }
  if constexpr (DOT) {
#pragma unroll
    for (int c = 0; c < NC; ++c) d[c] = (a[c][0].x + a[c][1].x) + (a[c][0].y + a[c][1].y);
  }
}

// Element r of a lane's column c held as row pairs.
template <int R, int NC>
__device__ __forceinline__ float yat(const float2 (&y)[NC][R / 2], int c, int r) {
  return (r & 1) ? y[c][r >> 1].y : y[c][r >> 1].x;
}

// y *= f, two rows per packed multiply.
template <int R, int NC>
__device__ __forceinline__ void scale_state(float2 (&y)[NC][R / 2], float f) {
  const float2 ff = make_float2(f, f);
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int m = 0; m < R / 2; ++m) y[c][m] = __fmul2_rn(y[c][m], ff);
}

// Two CTAs of four warps per SM at K = V = 128: the registers (~180 per
// thread for the packed state) allow two, and the staging (keys and values of
// 32 tokens, fp32 and raw, ~49 KB of shared memory per CTA) four.  Four warps
// per CTA share each tile's staging (widening and the log-decay prefix) over
// 128 columns: measured 2.4 % faster per call than two warps at four CTAs per
// SM, the same eight warps per SM.
template <int R, int G, int NC>
__global__ void __launch_bounds__(kLocalThreads, 2) local_pass_kernel(const LocalParams p) {
  constexpr int CW = 32 / G;  // column groups (of NC columns) per warp
  const LocalJob& j = p.j;
  const int K = j.K, V = j.V, L = j.L;
  const int64_t unit = blockIdx.z == 0 ? (int64_t)blockIdx.y : (int64_t)blockIdx.z * gridDim.y + blockIdx.y;
  if (unit >= (int64_t)j.nchains * j.S) return;
  const int64_t chain = unit / j.S;
  const int seg = (int)(unit - chain * j.S);

  extern __shared__ __align__(16) float smem[];
  float* ks = smem;               // [kTT][K] keys, fp32
  float* vs = ks + kTT * K;       // [kTT][V] values, fp32
  float* bs = vs + kTT * V;       // [kTT] write strength
  float* inv_s = bs + kTT;        // [kTT] 1 / s for the token's update
  float* fac_s = inv_s + kTT;     // [kTT] rescale factor after the previous token (1 = none)
  float* s_end = fac_s + kTT;     // [4] s after the segment's last token
  float* braw = s_end + 4;        // [kTT] next tile's write strengths, as loaded
  float* graw = braw + kTT;       // [kTT] next tile's log-decays, as loaded
  uint16_t* kraw = reinterpret_cast<uint16_t*>(graw + kTT);  // [kTT][K] next tile's keys, bf16
  uint16_t* vraw = kraw + kTT * K;                           // [kTT][V] next tile's values, bf16

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int part = lane / CW;  // which block of R rows
  const int q = lane - part * CW;
  const int row0 = part * R;
  const int cta_c0 = p.col_begin + (int)blockIdx.x * p.cols_per_cta;
  const int gc = cta_c0 + warp * (NC * CW) + NC * q;  // this lane's first column of Y (then gc + 1 .. gc + NC - 1)
  const bool live = gc < p.col_end;
  const bool is_h = gc < V;          // NC divides V: a lane's columns are all of H or all of M
  const int mc = gc - V;             // its first column of M when !is_h
  const bool need_v = cta_c0 < V;    // the CTA holds a column of H

  float2 y[NC][R / 2];
#pragma unroll
  for (int c = 0; c < NC; ++c)
#pragma unroll
    for (int m = 0; m < R / 2; ++m)
      y[c][m] = make_float2((!is_h && row0 + 2 * m == mc + c) ? 1.0f : 0.0f,
                            (!is_h && row0 + 2 * m + 1 == mc + c) ? 1.0f : 0.0f);

  // Let a dependent kernel (the correction) launch now; it reads H and M only
  // after its griddepcontrol.wait, i.e. after this grid has completed.
  griddep_launch_dependents();
  griddep_wait();

  const int64_t tok0 = chain * j.T + (int64_t)seg * L;
  issue_tile(j, tok0, min(kTT, L), need_v, kraw, vraw, braw, graw);
  double gsum = 0.0, gref = 0.0;  // staging warp: log-decay after the previous tile, and the reference
  for (int t0 = 0; t0 < L; t0 += kTT) {
    const int n = min(kTT, L - t0);
    cp_async_wait_all();
    __syncthreads();  // this tile's raw inputs have landed; every warp is done with the previous tile
    widen_rows(kraw, ks, n, K);
    if (need_v) widen_rows(vraw, vs, n, V);
    if (warp == 0) {
      // lane i <-> token t0 + i: inclusive prefix sum of the log-decays, fp64
      double Gs = lane < n ? (double)graw[lane] : 0.0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const double yv = __shfl_up_sync(0xffffffffu, Gs, o);
        if (lane >= o) Gs += yv;
      }
      Gs += gsum;
      // Reference moves: the first token whose sum is more than kRescaleLog
      // from the reference rescales the state before its update and becomes
      // the reference; tokens before it keep the old one.
      double ref = gref;
      bool done = lane >= n;
      float fac = 1.0f, inv = 1.0f;
      for (;;) {
        const unsigned far = __ballot_sync(0xffffffffu, !done && fabs(Gs - ref) > kRescaleLog);
        if (!far) break;
        const int f = __ffs(far) - 1;
        const double Gf = __shfl_sync(0xffffffffu, Gs, f);
        if (!done && lane < f) {
          inv = exp_split(ref - Gs);
          done = true;
        }
        if (lane == f) {
          fac = exp_split(Gf - ref);
          inv = 1.0f;
          done = true;
        }
        ref = Gf;
      }
      if (!done) inv = exp_split(ref - Gs);
      if (lane < n) {
        bs[lane] = braw[lane];
        inv_s[lane] = inv;
        fac_s[lane] = fac;
      }
      if (lane == n - 1) s_end[0] = exp_split(Gs - ref);
      gsum = __shfl_sync(0xffffffffu, Gs, n - 1);
      gref = ref;
    }
    __syncthreads();  // the widened tile is ready and the raw buffers are free
    if (t0 + kTT < L) issue_tile(j, tok0 + t0 + kTT, min(kTT, L - t0 - kTT), need_v, kraw, vraw, braw, graw);

    // Token i's update and token i + 1's dot products share one pass over the
    // registers: d_{i+1} = k_{i+1}^T (Yhat + k_i c_i^T).
    float d[NC];
    float cz[NC] = {};
    {
      const float fac = fac_s[0];
      if (fac != 1.0f) scale_state<R, NC>(y, fac);  // same for every thread of the CTA
      token_pass<R, NC, false, true>(y, nullptr, cz, ks + row0, d);
      reduce_parts<CW, NC>(d);
    }
    for (int i = 0; i < n; ++i) {
      float v[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) v[c] = 0.f;
      if (is_h && live) {
        if constexpr (NC == 4) {
          const float4 vv = *reinterpret_cast<const float4*>(vs + i * V + gc);
          v[0] = vv.x; v[1] = vv.y; v[2] = vv.z; v[3] = vv.w;
        } else {
#pragma unroll
          for (int c = 0; c < NC; ++c) v[c] = vs[i * V + gc + c];
        }
      }
      const float b = bs[i], inv = inv_s[i];
      float cc[NC];
#pragma unroll
      for (int c = 0; c < NC; ++c) cc[c] = b * fmaf(v[c], inv, -d[c]);
      const float* kc = ks + i * K + row0;
      if (i + 1 < n) {
        token_pass<R, NC, true, true>(y, kc, cc, kc + K, d);
        reduce_parts<CW, NC>(d);
        const float fac = fac_s[i + 1];
        if (fac != 1.0f) {  // rescale before token i + 1: its dot products scale alike
          scale_state<R, NC>(y, fac);
#pragma unroll
          for (int c = 0; c < NC; ++c) d[c] *= fac;
        }
      } else {
        token_pass<R, NC, true, false>(y, kc, cc, nullptr, d);
      }
    }
  }
  if (!live) return;
  const float s = s_end[0];
  if (is_h) {
    float* h = j.H + unit * (int64_t)K * V;
    if (j.layout == 0) {  // kv: H[k][v], NC consecutive columns per row
#pragma unroll
      for (int r = 0; r < R; ++r) {
        float* dst = h + (int64_t)(row0 + r) * V + gc;
        if constexpr (NC == 4)
          *reinterpret_cast<float4*>(dst) = make_float4(yat<R, NC>(y, 0, r) * s, yat<R, NC>(y, 1, r) * s,
                                                        yat<R, NC>(y, 2, r) * s, yat<R, NC>(y, 3, r) * s);
        else
          *reinterpret_cast<float2*>(dst) = make_float2(yat<R, NC>(y, 0, r) * s, yat<R, NC>(y, 1, r) * s);
      }
    } else {  // vk: H[v][k], R consecutive rows per column
#pragma unroll
      for (int c = 0; c < NC; ++c) {
        float* dst = h + (int64_t)(gc + c) * K + row0;
#pragma unroll
        for (int r = 0; r < R; r += 4)
          *reinterpret_cast<float4*>(dst + r) = make_float4(y[c][r / 2].x * s, y[c][r / 2].y * s,
                                                            y[c][r / 2 + 1].x * s, y[c][r / 2 + 1].y * s);
      }
    }
  } else {
    float* m = j.M + unit * (int64_t)K * K;
#pragma unroll
    for (int r = 0; r < R; ++r) {
      float* dst = m + (int64_t)(row0 + r) * K + mc;
      if constexpr (NC == 4)
        *reinterpret_cast<float4*>(dst) = make_float4(yat<R, NC>(y, 0, r) * s, yat<R, NC>(y, 1, r) * s,
                                                      yat<R, NC>(y, 2, r) * s, yat<R, NC>(y, 3, r) * s);
      else
        *reinterpret_cast<float2*>(dst) = make_float2(yat<R, NC>(y, 0, r) * s, yat<R, NC>(y, 1, r) * s);
    }
  }
}

template <int R, int G, int NC>
size_t smem_rg(const LocalJob& j) {
  // fp32 tile, per-token scalars, raw next tile (bf16 keys and values, fp32 scalars)
  return sizeof(float) * (size_t)(kTT * (j.K + j.V) + 3 * kTT + 4 + 2 * kTT) +
         sizeof(uint16_t) * (size_t)kTT * (j.K + j.V);
}

// CTAs of a launch, and how many fit on one SM at once.
template <int R, int G, int NC>
cudaError_t info_rg(const LocalJob& j, bool with_h, bool with_m, int64_t* ctas, int* per_sm) {
  const int cols = (with_h ? j.V : 0) + (with_m ? j.K : 0);
  const int per_cta = kLocalWarps * NC * (32 / G);
  *ctas = (int64_t)j.nchains * j.S * ((cols + per_cta - 1) / per_cta);
  const size_t smem = smem_rg<R, G, NC>(j);
  cudaError_t e = cudaFuncSetAttribute(local_pass_kernel<R, G, NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(per_sm, local_pass_kernel<R, G, NC>, kLocalThreads, smem);
}

template <int R, int G, int NC>
cudaError_t launch_rg(const LocalJob& j, cudaStream_t stream) {
  LocalParams p{};
  p.j = j;
  p.col_begin = j.H ? 0 : j.V;
  p.col_end = j.M ? j.V + j.K : j.V;
  p.cols_per_cta = kLocalWarps * NC * (32 / G);
  const int64_t units = (int64_t)j.nchains * j.S;
  const int xblocks = (p.col_end - p.col_begin + p.cols_per_cta - 1) / p.cols_per_cta;
  dim3 grid(xblocks, 1, 1);
  if (units <= 65535) {
    grid.y = (unsigned)units;
  } else {
    grid.y = 65535u;
    grid.z = (unsigned)((units + 65534) / 65535);
  }
  const size_t smem = smem_rg<R, G, NC>(j);
  cudaError_t e = cudaFuncSetAttribute(local_pass_kernel<R, G, NC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  return launch_kernel(local_pass_kernel<R, G, NC>, grid, kLocalThreads, smem, stream, j.pdl != 0, p);
}

}  // namespace

// Rows per lane R, lanes per column group G and columns per lane NC for a key
// dimension K (a multiple of 32 up to 256): four columns of 32 or fewer rows
// up to K = 128 (each key value read feeds four FMAs per use), two columns of
// at most 64 rows above.
cudaError_t local_grid_info(const LocalJob& j, bool with_h, bool with_m, int64_t* ctas, int* per_sm) {
  switch (j.K) {
    case 32: return info_rg<32, 1, 4>(j, with_h, with_m, ctas, per_sm);
    case 64: return info_rg<32, 2, 4>(j, with_h, with_m, ctas, per_sm);
    case 96: return info_rg<24, 4, 4>(j, with_h, with_m, ctas, per_sm);
    case 128: return info_rg<32, 4, 4>(j, with_h, with_m, ctas, per_sm);
    case 160: return info_rg<40, 4, 2>(j, with_h, with_m, ctas, per_sm);
    case 192: return info_rg<48, 4, 2>(j, with_h, with_m, ctas, per_sm);
    case 224: return info_rg<56, 4, 2>(j, with_h, with_m, ctas, per_sm);
    case 256: return info_rg<64, 4, 2>(j, with_h, with_m, ctas, per_sm);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_local_simt(const LocalJob& j, cudaStream_t stream) {
  switch (j.K) {
    case 32: return launch_rg<32, 1, 4>(j, stream);
    case 64: return launch_rg<32, 2, 4>(j, stream);
    case 96: return launch_rg<24, 4, 4>(j, stream);
    case 128: return launch_rg<32, 4, 4>(j, stream);
    case 160: return launch_rg<40, 4, 2>(j, stream);
    case 192: return launch_rg<48, 4, 2>(j, stream);
    case 224: return launch_rg<56, 4, 2>(j, stream);
    case 256: return launch_rg<64, 4, 2>(j, stream);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace qla
