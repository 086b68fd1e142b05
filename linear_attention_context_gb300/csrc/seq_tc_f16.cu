// Sequential state correction, tensor-core engine with fp16 operand pairs
// (sm_103a), K = 128.
//
// Computes the recurrence of Antarx Memos, "一次 TileLang Warp Specialization 数
// 值错误的定位与修复", section "理解三个缓冲区，才能判断哪里需要同步":
// X_{j+1} = A_j X_j + H_j in the kv view, A_j = M (forward) or M^T (reverse),
// out[seg] = the state entering seg.  Same producer/consumer shape as the
// 3xTF32 engine (seq_tc.cu): a TMA producer streams H and M tiles through
// shared-memory rings, splitters turn M into tensor-core operands in TMEM,
// three threads issue tcgen05.mma, and epilogue warpgroups drain the
// accumulators, add H and write the next state operand and out.
//
// What differs is the operand format.  The MMAs are kind::f16, twice the TF32
// rate and 16 k per instruction, on hi/lo pairs of power-of-two-scaled
// operands:
//     (s_A A)(s_X X) ~= A_hi X_hi + A_hi X_lo + A_lo X_hi,
//     hi = RN_f16(s x),  lo = RN_f16(s x - hi)   (s x - hi is exact in fp32),
// so a step takes 24 MMAs instead of 48 and the state operand is 16 KB
// instead of 32.  A pair carries 22 significant bits, as the TF32 pair does,
// and the dropped A_lo X_lo term is below 2^-22 of the product.
//
// Scales (powers of two, so scaling and unscaling are exact):
//   s_A   one per step: max|A_j| s_A in [2^14, 2^15), from a max pass over
//         the step's M tile by the splitters (off the critical path);
//   s_X   one per 8-column group of the state (an epilogue warpgroup's
//         columns), from a bound on the new state that is known before its
//         accumulators are ready:
//             max|X_{j+1}| <= K max|A_j| max|X_j| + max|H_j|,
//         bound * s_X in [2^14, 2^15).  So no reduction sits between the
//         accumulators and the next state operand.  Every scaled value stays
//         below 2^15 (fp16 holds up to 65504); the bound may exceed the true
//         maximum by up to a factor K, which costs nothing as long as values
//         stay in fp16's normal range, and below it a pair's absolute error is
//         at most 2^-25 / s_X: 2^-39 of the bound, well under the state's own
//         fp32 rounding.
// The epilogue drains sum(chains) * 2^-p_A * 2^-p_X + H (two exact scalings,
// so neither can leave the fp32 range on its own).
//
// Accumulation: the tensor core rounds its fp32 accumulator toward zero, so
// the 8 big A_hi X_hi MMAs of a step go to two chains (4 each, as in the TF32
// engine) and the two small terms to one chain each; the epilogue adds the
// chains with round-to-nearest adds.
//
// Operand layouts.  A (hi, lo) in TMEM: lane = row m, each 32-bit column two
// consecutive k (the lower half the even one); a step is 64 columns of hi and
// 64 of lo, in two groups of 64 k.  B = X (hi, lo) in shared memory, MN-major
// with the 64-byte swizzle: row k holds the state's 32 columns as fp16 (64
// bytes), so an epilogue thread, which holds row k of 8 columns, writes its
// hi and its lo with one 16-byte store each.
//
//  role      warps    does
//  producer  0 (1 th) TMA: H_j tile -> h slot j&1; M_j in four 32-column
//                     chunks -> m ring (two steps).
//  mma       1, 2, 3  (1 thread each) tcgen05.mma kind::f16: big terms,
//                     A_hi X_lo, A_lo X_hi.
//  splitter  4..11    two warpgroups, alternate steps: max pass over the
//                     step's four chunks (one scale per step), then split
//                     each chunk -> TMEM A slot of the step (two slots).
//  epilogue  12..27   four warpgroups of 8 columns: H_j, the chains = X_{j+1};
//                     its hi/lo -> B first (the next step waits on it), then
//                     out via per-warp TMA stores; then the scale of X_{j+2}.
//
//  storage        written by           read by             reusable after
//  m ring [s]     TMA (async)          splitter (generic)  splitter's last read: fence + m_empty arrive
//  h slot [j&1]   TMA (async)          epilogue (generic)  epilogue's last read: fence + h_empty arrive
//  A slot (TMEM)  splitter tcgen05.st  mma (async)         3 commits -> a_empty (per group of 64 k)
//  B hi/lo        epilogue st.shared   mma (async)         d_full (3 commits: all MMAs of the step done)
//                 + fence.proxy.async
//  chains (TMEM)  mma                  epilogue tcgen05.ld x_ready (epilogue's wait::ld done)
//  A scale [j%4]  splitter st.shared   epilogue            the splitter of step j+4 waits a_empty of
//                 + sc_full arrive                         step j+2, which follows the epilogue's
//                                                          last read (step j's drain)
//  out staging    epilogue st.shared   TMA store (async)   bulk wait_group.read
//                 + fence.proxy.async
//
// Warpgroup maxima are exchanged through shared memory and an mbarrier per
// warpgroup (bounded waits, unlike bar.sync), double-buffered by use.
//
// The slot-release fence (Antarx Memos, section "三个可用源码方案的具体差别")
// is selectable as in the TF32 engine.  In place (out == H): out[seg] is
// stored over H[seg] only after the TMA load of that H tile has completed.
// Every wait is bounded; on expiry the CTA drains its copies in flight, frees
// TMEM and returns with the device status word set.
#include <cuda.h>
#include <cuda_fp16.h>

#include "ptx.cuh"
#include "qla_internal.h"
#include "tma_map.h"

// Optional pipeline trace (compile with -DQLA_TRACE): clock64() stamps of the
// handoffs of CTA (0, 0), read back with qla_debug_trace16().  Slots are
// [role][step][event][thread]; roles 0 producer, 1 mma, 2 splitter, 3 epilogue.
#ifdef QLA_TRACE
__device__ long long g_qla_trace16[4 * 8 * 8 * 16];
#define TR16(role, step, ev, ch)                                                                            \
  do {                                                                                                      \
    if (tr && (step) < 8 && (ch) < 16) g_qla_trace16[(((role) * 8 + (step)) * 8 + (ev)) * 16 + (ch)] = clock64(); \
  } while (0)
#else
#define TR16(role, step, ev, ch) \
  do {                           \
  } while (0)
#endif

namespace qla {
namespace {

using namespace ptx;

namespace h16 {
constexpr int K = 128;
constexpr int VT = 32;                        // state columns per CTA
constexpr int NI = 3;                         // MMA-issuing threads
constexpr int NB = 2;                         // big-term chains
constexpr int NQ = NB + 2;                    // chains (+ A_hi X_lo, A_lo X_hi)
constexpr int NE = 4;                         // epilogue warpgroups ...
constexpr int EC = VT / NE;                   // ... of 8 columns
constexpr int NSG = 2;                        // splitter warpgroups (alternate steps)
constexpr int CPS = 4;                        // 32-wide k chunks of M per step
constexpr int NM = NSG * CPS;                 // m ring stages: one step per splitter warpgroup
constexpr int KS = K / 16;                    // MMA k-steps per step (16 k each)
constexpr int SPL_WARP0 = 1 + NI;
constexpr int EPI_WARP0 = SPL_WARP0 + 4 * NSG;
constexpr int WARPS = EPI_WARP0 + 4 * NE;     // 28
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t ACOL = NQ * VT;            // first column of the A slots
constexpr uint32_t AGRP = 64;                 // TMEM columns of one A group (64 k: hi 32, lo 32)
constexpr uint32_t ASTEP = 2 * AGRP;          // one step's A slot
constexpr uint32_t kChunkBytes = 128 * 32 * 4;
constexpr uint32_t TILE = K * VT * 4;         // fp32 state tile
constexpr uint32_t BTILE = K * VT * 2;        // fp16 operand tile
constexpr int NOUT = 2;                       // out staging buffers
constexpr uint32_t OFF_M = 0;
constexpr uint32_t OFF_H = OFF_M + NM * kChunkBytes;
constexpr uint32_t OFF_BHI = OFF_H + 2 * TILE;
constexpr uint32_t OFF_BLO = OFF_BHI + BTILE;
constexpr uint32_t OFF_OUT = OFF_BLO + BTILE;
constexpr uint32_t OFF_CTRL = OFF_OUT + NOUT * TILE;
constexpr uint32_t CTRL_BYTES = 1024;
constexpr uint32_t SMEM = OFF_CTRL + CTRL_BYTES + 1024;  // + alignment slack
static_assert(SMEM <= 232448, "shared memory budget");
static_assert(ACOL + NSG * ASTEP <= kTmemCols, "TMEM columns");
static_assert(OFF_BHI % 1024 == 0 && OFF_BLO % 1024 == 0, "swizzled operands need aligned atoms");
}  // namespace h16

struct H16Params {
  CUtensorMap map_h;    // H (load)
  CUtensorMap map_out;  // out (store)
  CUtensorMap map_m;    // M chunks (load)
  SeqJob job;
  unsigned int* status;
  uint64_t limit_ns;
  int has_h;
  int in_place;
  int release;          // 0 membar, 1 proxy, 2 delay, 3 none
  int stall_test;       // epilogue waits on a barrier nothing arrives on
};

struct H16Ctrl {
  uint64_t m_full[h16::NM], m_empty[h16::NM];
  uint64_t a_full[2 * h16::NSG], a_empty[2 * h16::NSG];  // [step slot][group of 64 k]
  uint64_t h_full[2], h_empty[2];
  uint64_t x_ready, d_full;
  uint64_t sc_full[4];              // splitter -> epilogue: A scale of step j, [j % 4]
  uint64_t sx[h16::NSG][2];         // splitter warpgroup max exchange [group][buffer]
  uint64_t ex[h16::NE][2];          // epilogue warpgroup max exchange [group][buffer]
  uint64_t never;
  uint64_t mma_done[h16::NI];
  float ascale[4][2];               // [j % 4]: max|A_j|, 2^-p_A
  alignas(16) uint32_t smax[h16::NSG][2][4];    // [group][buffer][warp]: max bits
  alignas(16) uint32_t emax[h16::NE][2][4][2];  // [group][buffer][warp][state, H]: max bits
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(H16Ctrl) <= h16::CTRL_BYTES, "control block");

__device__ __forceinline__ void release_fence16(int mode) {
  if (mode == 0) membar_cta();
  else if (mode == 1) fence_proxy_async_smem();
}

__device__ __forceinline__ bool warp_wait16(uint64_t* bar, uint32_t parity, const WaitCtl& c) {
  const bool ok = mbar_wait(bar, parity, c);
  return __all_sync(0xffffffffu, ok);
}

// Exponent p, clamped to [-100, 100], with v 2^p in [2^14, 2^15) for a
// finite v > 0 (v >= 0 here: a maximum of magnitudes or a bound).
__device__ __forceinline__ int scale_exp(float v) {
  const int e = (int)((__float_as_uint(v) >> 23) & 0xFFu) - 127;
  return max(-100, min(100, 14 - e));
}

// 2^p for p in [-126, 127].
__device__ __forceinline__ float exp2i(int p) { return __int_as_float((p + 127) << 23); }

// Two values at once: v = s x, hi = RN_f16(v), lo = RN_f16(v - hi); returns
// the packed pairs (x0 in the lower half).
__device__ __forceinline__ void split_f16x2(float x0, float x1, float s, uint32_t& hi, uint32_t& lo) {
  const float2 v = __fmul2_rn(make_float2(x0, x1), make_float2(s, s));
  const __half2 h = __floats2half2_rn(v.x, v.y);
  const float2 hf = __half22float2(h);
  const float2 r = __ffma2_rn(hf, make_float2(-1.f, -1.f), v);
  const __half2 l = __floats2half2_rn(r.x, r.y);
  hi = *reinterpret_cast<const uint32_t*>(&h);
  lo = *reinterpret_cast<const uint32_t*>(&l);
}

// The operands of one issuer's 8 MMAs of a step in A slot 0: D chain, A
// column, B descriptor low word (k-step ks reads B rows [16 ks, 16 ks + 16),
// 1024 bytes further per k-step).  Slot 1 is ASTEP columns further.
struct Ops16 {
  uint32_t d[h16::KS], a[h16::KS], b[h16::KS];
};

template <int ROLE>
__device__ __forceinline__ Ops16 ops16(uint32_t tmem, uint32_t bhi_lo, uint32_t blo_lo) {
  using namespace h16;
  Ops16 o;
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    o.d[ks] = tmem + (uint32_t)(ROLE == 0 ? ks % NB : ROLE == 1 ? NB : NB + 1) * VT;
    o.a[ks] = tmem + ACOL + (uint32_t)(ks / 4) * AGRP + (ROLE == 2 ? 32u : 0u) + (uint32_t)(ks % 4) * 8;
    o.b[ks] = (ROLE == 1 ? blo_lo : bhi_lo) + (uint32_t)((ks * 1024) >> 4);
  }
  return o;
}

template <int ROLE, int K0, int K1>
__device__ __forceinline__ void issue16(const Ops16& o, uint32_t aoff, uint32_t bhi) {
  constexpr uint32_t idesc = idesc_f16(128, h16::VT, true);
#pragma unroll
  for (int m = K0; m < K1; ++m) {
    if ((ROLE == 0 && m < h16::NB) || (ROLE != 0 && m == 0))
      mma_f16_ts_c<false>(o.d[m], o.a[m] + aoff, o.b[m], bhi, idesc);
    else
      mma_f16_ts_c<true>(o.d[m], o.a[m] + aoff, o.b[m], bhi, idesc);
  }
}

template <int ROLE>
__device__ __forceinline__ void mma_role16(H16Ctrl* ctl, uint8_t* smem, uint32_t tmem, int nsteps,
                                           const WaitCtl& wc, [[maybe_unused]] bool tr) {
  using namespace h16;
  const uint64_t dh = smem_desc_sw64(smem_u32(smem + OFF_BHI), 512, 512);
  const uint64_t dl = smem_desc_sw64(smem_u32(smem + OFF_BLO), 512, 512);
  const uint32_t bhi = (uint32_t)(dh >> 32);  // the same for both descriptors
  const Ops16 ops = ops16<ROLE>(tmem, (uint32_t)dh, (uint32_t)dl);
  bool ok = true;
  for (int step = 0; step < nsteps && ok; ++step) {
    if (!(ok = mbar_wait(&ctl->x_ready, step & 1, wc))) break;
    TR16(1, step, 0, ROLE);
    tc_fence_after();
    const int sl = step & 1;
    const uint32_t aph = (uint32_t)(step >> 1) & 1;
    const uint32_t aoff = (uint32_t)sl * ASTEP;
    // Group 1 is usually split before the step starts: test it without
    // blocking, so that no poll (which stalls until this thread's queued
    // MMAs have dispatched) sits between the step's MMAs unless it must.
    if (!(ok = mbar_wait(&ctl->a_full[2 * sl], aph, wc))) break;
    const bool g1_ready = mbar_test_wait(&ctl->a_full[2 * sl + 1], aph);
    TR16(1, step, 1, ROLE);
    tc_fence_after();
    issue16<ROLE, 0, KS / 2>(ops, aoff, bhi);
    mma_commit(&ctl->a_empty[2 * sl]);
    TR16(1, step, 2, ROLE);
    if (!g1_ready) {
      if (!(ok = mbar_wait(&ctl->a_full[2 * sl + 1], aph, wc))) break;
      tc_fence_after();
    }
    TR16(1, step, 3, ROLE);
    issue16<ROLE, KS / 2, KS>(ops, aoff, bhi);
    mma_commit(&ctl->a_empty[2 * sl + 1]);
    mma_commit(&ctl->d_full);
    TR16(1, step, 4, ROLE);
  }
  // All MMAs this thread issued must finish before TMEM is freed.
  mma_commit(&ctl->mma_done[ROLE]);
  mbar_wait_drain(&ctl->mma_done[ROLE], 0, 200000000ull);
}

__global__ void __launch_bounds__(32 * h16::WARPS, 1) seq_tc_f16_kernel(const __grid_constant__ H16Params p) {
  using namespace h16;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  H16Ctrl* ctl = reinterpret_cast<H16Ctrl*>(smem + OFF_CTRL);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const SeqJob& j = p.job;
  int u, tile;
  if (!unit_and_tile(j, u, tile)) return;
  const int chain = u / j.G;
  const int g = u - chain * j.G;
  int64_t cbase;  // the chain's first segment in the packed arrays
  int S;
  griddep_wait();  // (before the first global access: the offsets may be the previous kernel's output)
  if (!chain_span(j, chain, cbase, S)) return;  // invalid offsets: recorded, nothing touched
  const int s_lo = g * j.L;
  const int n = min(j.L, S - s_lo);
  const int nsteps = n - 1 + (j.fin ? 1 : 0);
  const int vbase = tile * VT;
  if (n <= 0) {  // a sequence without segments: its final state is its initial state
    if (j.fin) {
      float* F = j.fin + u * j.fin_unit_stride;
      const float* I = j.init_mode == kInitPointer ? j.init + u * j.init_unit_stride : nullptr;
      for (int e = threadIdx.x; e < K * VT; e += blockDim.x) {
        const int k = e / VT, v = vbase + e % VT;
        const int64_t idx = j.layout == 0 ? (int64_t)k * j.V + v : (int64_t)v * K + k;
        F[idx] = I ? I[idx] : (j.init_mode == kInitIdentity && k == v ? 1.f : 0.f);
      }
    }
    return;
  }
  const bool fwd = j.direction == 0;
  auto seg_of = [&](int step) { return fwd ? s_lo + step : s_lo + n - 1 - step; };
#ifdef QLA_TRACE
  const bool tr = blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && lane == 0 &&
                  (warp <= NI || warp == SPL_WARP0 || warp == SPL_WARP0 + 4 || warp == EPI_WARP0 || warp == WARPS - 1);
  const int trc = warp == WARPS - 1 ? 1 : 0;
  (void)trc;
#else
  constexpr bool tr = false;
#endif

  // Epilogue warps load the initial state before set-up, so its global-memory
  // latency overlaps barrier initialisation and the TMEM allocation.
  float y[EC];
  if (warp >= EPI_WARP0) {
    const int e = (warp - EPI_WARP0) >> 2;
    const int k = 32 * (warp & 3) + lane;
    const int c0 = e * EC;
    if (j.init_mode == kInitPointer) {
      const float* src = j.init + u * j.init_unit_stride;
      if (j.layout == 0) {
#pragma unroll
        for (int q = 0; q < EC / 4; ++q) {
          const float4 v = *reinterpret_cast<const float4*>(src + (int64_t)k * j.V + vbase + c0 + 4 * q);
          y[4 * q] = v.x; y[4 * q + 1] = v.y; y[4 * q + 2] = v.z; y[4 * q + 3] = v.w;
        }
      } else {
#pragma unroll
        for (int c = 0; c < EC; ++c) y[c] = src[(int64_t)(vbase + c0 + c) * K + k];
      }
    } else {
#pragma unroll
      for (int c = 0; c < EC; ++c) y[c] = (j.init_mode == kInitIdentity && k == vbase + c0 + c) ? 1.f : 0.f;
    }
  }

  if (threadIdx.x == 0) {
    prefetch_tensormap(&p.map_m);
    if (p.has_h) prefetch_tensormap(&p.map_h);
    if (j.out) prefetch_tensormap(&p.map_out);
    for (int i = 0; i < NM; ++i) {
      mbar_init(&ctl->m_full[i], 1);
      mbar_init(&ctl->m_empty[i], 4);
    }
    for (int i = 0; i < 2 * NSG; ++i) {
      mbar_init(&ctl->a_full[i], 4);   // the step's splitter warpgroup
      mbar_init(&ctl->a_empty[i], NI);  // one commit per issuing thread
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&ctl->h_full[i], 1);
      mbar_init(&ctl->h_empty[i], 4 * NE);
    }
    mbar_init(&ctl->x_ready, 4 * NE);
    mbar_init(&ctl->d_full, NI);
    for (int i = 0; i < 4; ++i) mbar_init(&ctl->sc_full[i], 1);
    for (int i = 0; i < NSG; ++i)
      for (int b = 0; b < 2; ++b) mbar_init(&ctl->sx[i][b], 4);
    for (int i = 0; i < NE; ++i)
      for (int b = 0; b < 2; ++b) mbar_init(&ctl->ex[i][b], 4);
    mbar_init(&ctl->never, 1);
    for (int i = 0; i < NI; ++i) mbar_init(&ctl->mma_done[i], 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(&ctl->tmem_base, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  WaitCtl wc{&ctl->abort, p.status, p.limit_ns};
  TR16(0, 0, 7, 0);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t mit = 0;
      int hissued = 0;
      bool ok = true;
      const int hrows = j.layout == 0 ? K : j.V;  // rows of one state in the 2-D view of H
      for (int step = 0; step < nsteps && ok; ++step) {
        const int seg = seg_of(step);
        const int64_t mrow0 = (cbase + seg) * K;
        if (p.has_h) {
          const int slot = step & 1;
          const int64_t hrow0 = (cbase + seg) * hrows;
          if (!(ok = mbar_wait(&ctl->h_empty[slot], ((step >> 1) & 1) ^ 1, wc))) break;
          mbar_arrive_expect_tx(&ctl->h_full[slot], TILE);
          uint8_t* dst = smem + OFF_H + slot * TILE;
          if (j.layout == 0)
            tma_load_2d(dst, &p.map_h, vbase, (int32_t)hrow0, &ctl->h_full[slot]);
          else
            tma_load_2d(dst, &p.map_h, 0, (int32_t)(hrow0 + vbase), &ctl->h_full[slot]);
          ++hissued;
          TR16(0, step, 0, 0);
        }
        for (int c = 0; c < CPS; ++c, ++mit) {
          const int stage = mit % NM;
          if (!(ok = mbar_wait(&ctl->m_empty[stage], ((mit / NM) & 1) ^ 1, wc))) break;
          mbar_arrive_expect_tx(&ctl->m_full[stage], kChunkBytes);
          uint8_t* dst = smem + OFF_M + stage * kChunkBytes;
          if (fwd)  // A = M: columns 32c.. of all 128 rows (128-byte swizzle, box 32 x 128)
            tma_load_2d(dst, &p.map_m, 32 * c, (int32_t)mrow0, &ctl->m_full[stage]);
          else      // A = M^T: M rows 32c.., all 128 columns (box 128 x 32)
            tma_load_2d(dst, &p.map_m, 0, (int32_t)(mrow0 + 32 * c), &ctl->m_full[stage]);
          TR16(0, step, 1, c);
        }
      }
      // Drain: every issued load must land before shared memory goes away.
      const uint64_t drain = 200000000ull;  // 200 ms
      for (int s = 0; s < NM; ++s) {
        const uint32_t uses = mit > (uint32_t)s ? (mit - 1 - s) / NM + 1 : 0;
        if (uses) mbar_wait_drain(&ctl->m_full[s], (uses - 1) & 1, drain);
      }
      for (int s = 0; s < 2; ++s) {
        const int uses = hissued > s ? (hissued - 1 - s) / 2 + 1 : 0;
        if (uses) mbar_wait_drain(&ctl->h_full[s], (uses - 1) & 1, drain);
      }
    }
    __syncwarp();
  } else if (warp <= NI) {
    // ------------------------------------------------------------ mma issuers
    if (lane == 0) {
      if (warp == 1) mma_role16<0>(ctl, smem, tmem, nsteps, wc, tr);
      else if (warp == 2) mma_role16<1>(ctl, smem, tmem, nsteps, wc, tr);
      else mma_role16<2>(ctl, smem, tmem, nsteps, wc, tr);
    }
    __syncwarp();
  } else if (warp < EPI_WARP0) {
    // ------------------------------------------------------------ A splitters
    const int sg = (warp - SPL_WARP0) >> 2;  // takes steps sg, sg + 2, ...: m stages 4 sg.., A slot sg
    const int wq = warp & 3;
    const int t = 32 * wq + lane;            // A row = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    bool ok = true;
    int xu = 0;                              // uses of this warpgroup's max exchange
    for (int step = sg; step < nsteps && ok; step += NSG, ++xu) {
      const uint32_t mph = (uint32_t)(step >> 1) & 1;
#pragma unroll 1
      for (int c = 0; c < CPS && ok; ++c) ok = warp_wait16(&ctl->m_full[CPS * sg + c], mph, wc);
      if (!ok) break;
      TR16(2, step, 0, sg);
      // Max pass over the whole tile (any partition of its elements will do).
      float am = 0.f;
#pragma unroll
      for (int c = 0; c < CPS; ++c) {
        const float4* ch = reinterpret_cast<const float4*>(smem + OFF_M + (CPS * sg + c) * kChunkBytes);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 v = ch[t + 128 * q];
          am = fmaxf(am, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
      }
      const int b = xu & 1;
      const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(am));
      if (lane == 0) ctl->smax[sg][b][wq] = wm;
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->sx[sg][b]);
      if (!(ok = warp_wait16(&ctl->sx[sg][b], (xu >> 1) & 1, wc))) break;
      const uint4 mv = *reinterpret_cast<const uint4*>(ctl->smax[sg][b]);
      const float amax = __uint_as_float(max(max(mv.x, mv.y), max(mv.z, mv.w)));
      TR16(2, step, 1, sg);
      const int pa = scale_exp(amax);
      const float sa = exp2i(pa);
      if (t == 0) {
        ctl->ascale[step & 3][0] = amax;
        ctl->ascale[step & 3][1] = exp2i(-pa);
        mbar_arrive(&ctl->sc_full[step & 3]);
      }
      // Split pass: each group of two chunks -> its A group, then a_full.
#pragma unroll 1
      for (int grp = 0; grp < 2 && ok; ++grp) {
        const int gi = 2 * sg + grp;
        if (!(ok = warp_wait16(&ctl->a_empty[gi], mph ^ 1, wc))) break;
        TR16(2, step, 2 + 2 * grp, sg);
        tc_fence_after();
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          const int stage = CPS * sg + 2 * grp + cc;
          const uint8_t* chunk = smem + OFF_M + stage * kChunkBytes;
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            float x[16];
            if (fwd) {  // row t of a [128][32] tile, 16-byte pieces swizzled by (t & 7)
              const uint8_t* row = chunk + t * 128;
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                const float4 v = *reinterpret_cast<const float4*>(row + (((4 * half + q) ^ (t & 7)) << 4));
                x[4 * q] = v.x; x[4 * q + 1] = v.y; x[4 * q + 2] = v.z; x[4 * q + 3] = v.w;
              }
            } else {    // column t of a [32][128] tile
              const float* col = reinterpret_cast<const float*>(chunk) + t + 16 * half * 128;
#pragma unroll
              for (int k = 0; k < 16; ++k) x[k] = col[k * 128];
            }
            if (half == 1 && p.release != 2) {  // the stage's last ordinary read is done: release it
              release_fence16(p.release);
              __syncwarp();
              if (lane == 0) mbar_arrive(&ctl->m_empty[stage]);
            }
            uint32_t hi[8], lo[8];
#pragma unroll
            for (int k = 0; k < 16; k += 2) split_f16x2(x[k], x[k + 1], sa, hi[k / 2], lo[k / 2]);
            const uint32_t a = tmem + lane_off + ACOL + (uint32_t)gi * AGRP + (uint32_t)(cc * 16 + half * 8);
            tmem_st8(a, hi);
            tmem_st8(a + 32, lo);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->a_full[gi]);
        TR16(2, step, 3 + 2 * grp, sg);
        if (p.release == 2) {
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&ctl->m_empty[CPS * sg + 2 * grp]);
            mbar_arrive(&ctl->m_empty[CPS * sg + 2 * grp + 1]);
          }
        }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int e = (warp - EPI_WARP0) >> 2;  // column group [EC e, EC e + EC)
    const int wq = warp & 3;
    const int t = 32 * wq + lane;           // state row = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const int V = j.V;
    const int c0 = e * EC;
    int out_count = 0;
    int xu = 0;  // uses of this warpgroup's max exchange
    bool ok = true;

    // out[seg] <- y through per-warp staging (32 rows x EC floats) and TMA stores
    auto store_out = [&](int seg) {
      const int b = out_count % NOUT;
      if (lane == 0) bulk_wait_read<NOUT - 1>();
      __syncwarp();
      uint8_t* stg = smem + OFF_OUT + b * TILE + (e * 4 + wq) * (32 * EC * 4);
      float* f = reinterpret_cast<float*>(stg);
      if (j.layout == 0) {  // [32 rows][8 floats], 32-byte swizzle: piece q of row r at q ^ ((r / 4) & 1)
#pragma unroll
        for (int q = 0; q < EC / 4; ++q)
          *reinterpret_cast<float4*>(f + lane * EC + 4 * (q ^ ((lane >> 2) & 1))) =
              make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
      } else {              // [8 rows][32 floats]: column `lane`
#pragma unroll
        for (int c = 0; c < EC; ++c) f[c * 32 + lane] = y[c];
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        if (j.layout == 0)
          tma_store_2d(&p.map_out, stg, vbase + c0, (int32_t)((cbase + seg) * K + 32 * wq));
        else
          tma_store_2d(&p.map_out, stg, 32 * wq, (int32_t)((cbase + seg) * V + vbase + c0));
        bulk_commit();
      }
      ++out_count;
    };

    // Row t of the B operands: 64 bytes at t * 64; this warpgroup's 16-byte
    // piece e sits at piece e ^ ((t / 2) & 3).
    const uint32_t baddr = smem_u32(smem + OFF_BHI) + (uint32_t)t * 64 + (((uint32_t)e ^ (((uint32_t)t >> 1) & 3)) << 4);
    auto write_b = [&](float s) {
      uint32_t hv[4], lv[4];
#pragma unroll
      for (int c = 0; c < EC; c += 2) split_f16x2(y[c], y[c + 1], s, hv[c / 2], lv[c / 2]);
      sts128<0>(baddr, hv[0], hv[1], hv[2], hv[3]);
      sts128<BTILE>(baddr, lv[0], lv[1], lv[2], lv[3]);
      fence_proxy_async_smem();  // generic writes -> read by tcgen05.mma (async proxy)
    };

    // Warpgroup maxima of two magnitudes (as fp32 bits; both >= 0).
    auto exchange = [&](float a, float b, float& ma, float& mb) -> bool {
      const uint32_t ra = __reduce_max_sync(0xffffffffu, __float_as_uint(a));
      const uint32_t rb = __reduce_max_sync(0xffffffffu, __float_as_uint(b));
      const int bf = xu & 1;
      if (lane == 0) {
        ctl->emax[e][bf][wq][0] = ra;
        ctl->emax[e][bf][wq][1] = rb;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->ex[e][bf]);
      if (!warp_wait16(&ctl->ex[e][bf], (xu >> 1) & 1, wc)) return false;
      const uint4 p0 = *reinterpret_cast<const uint4*>(&ctl->emax[e][bf][0][0]);
      const uint4 p1 = *reinterpret_cast<const uint4*>(&ctl->emax[e][bf][2][0]);
      ma = __uint_as_float(max(max(p0.x, p0.z), max(p1.x, p1.z)));
      mb = __uint_as_float(max(max(p0.y, p0.w), max(p1.y, p1.w)));
      ++xu;
      return true;
    };
    auto absmax = [](const float (&v)[EC]) {
      float m = 0.f;
#pragma unroll
      for (int c = 0; c < EC; ++c) m = fmaxf(m, fabsf(v[c]));
      return m;
    };

    // X_0: scale from its exact maximum, then the B operand (the first
    // step's MMAs wait on it) and out[first segment].
    float xmax, unused;
    ok = exchange(absmax(y), 0.f, xmax, unused);
    int px = scale_exp(xmax);
    if (ok && nsteps > 0) {
      write_b(exp2i(px));
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->x_ready);
    }
    if (ok && j.out) {
      if (p.in_place && p.has_h && nsteps > 0) ok = warp_wait16(&ctl->h_full[0], 0, wc);
      if (ok) store_out(seg_of(0));
    }
    for (int step = 0; step < nsteps && ok; ++step) {
      // Everything the drain needs that does not depend on the MMAs: H_j,
      // the step's A scale and the scale of X_{j+1}.
      const int slot = step & 1;
      float h[EC];
      if (p.has_h) {
        if (!(ok = warp_wait16(&ctl->h_full[slot], (step >> 1) & 1, wc))) break;
        const uint8_t* ht = smem + OFF_H + slot * TILE;
        if (j.layout == 0) {  // [128 rows][32 floats], 128-byte swizzle: piece q of row k at q ^ (k & 7)
          const uint8_t* row = ht + t * (VT * 4);
#pragma unroll
          for (int q = 0; q < EC / 4; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(row + (((c0 / 4 + q) ^ (t & 7)) << 4));
            h[4 * q] = v.x; h[4 * q + 1] = v.y; h[4 * q + 2] = v.z; h[4 * q + 3] = v.w;
          }
        } else {              // [32 rows][128 floats]
          const float* f = reinterpret_cast<const float*>(ht) + t;
#pragma unroll
          for (int c = 0; c < EC; ++c) h[c] = f[(c0 + c) * K];
        }
        if (p.release != 2) {  // the h slot's last ordinary read is done: release it
          release_fence16(p.release);
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->h_empty[slot]);
        }
      } else {
#pragma unroll
        for (int c = 0; c < EC; ++c) h[c] = 0.f;
      }
      TR16(3, step, 0, trc);
      if (!(ok = warp_wait16(&ctl->sc_full[step & 3], (step >> 2) & 1, wc))) break;
      TR16(3, step, 1, trc);
      const float amax = ctl->ascale[step & 3][0];
      const float inv_a = ctl->ascale[step & 3][1];
      float hmax;
      if (!(ok = exchange(absmax(y), absmax(h), xmax, hmax))) break;
      TR16(3, step, 2, trc);
      const int pn = scale_exp(fmaf((float)K * amax, xmax, hmax));  // scale of X_{j+1}
      const float inv_x = exp2i(-px);

      uint64_t* dbar = (p.stall_test && step == 0) ? &ctl->never : &ctl->d_full;
      if (!(ok = warp_wait16(dbar, step & 1, wc))) break;
      TR16(3, step, 3, trc);
      tc_fence_after();
      {
        float b0[EC], b1[EC], s0[EC], s1[EC];
        const uint32_t base = tmem + lane_off + (uint32_t)c0;
        tmem_ld8(base, b0);
        tmem_ld8(base + VT, b1);
        tmem_ld8(base + 2 * VT, s0);
        tmem_ld8(base + 3 * VT, s1);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < EC; c += 2) {
          const float2 bb = __fadd2_rn(make_float2(b0[c], b0[c + 1]), make_float2(b1[c], b1[c + 1]));
          const float2 ss = __fadd2_rn(make_float2(s0[c], s0[c + 1]), make_float2(s1[c], s1[c + 1]));
          const float2 sum = __fadd2_rn(bb, ss);
          const float2 ua = __fmul2_rn(sum, make_float2(inv_a, inv_a));
          const float2 r = __ffma2_rn(ua, make_float2(inv_x, inv_x), make_float2(h[c], h[c + 1]));
          y[c] = r.x;
          y[c + 1] = r.y;
        }
      }
      TR16(3, step, 4, trc);
      if (step + 1 < nsteps) {  // X_{j+1} -> B operand: the critical path to the next step
        write_b(exp2i(pn));
        px = pn;
        tc_fence_before();  // the chains have been read (wait::ld above)
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->x_ready);
        TR16(3, step, 5, trc);
      } else if (j.fin) {
        float* F = j.fin + u * j.fin_unit_stride;
        if (j.layout == 0) {
#pragma unroll
          for (int q = 0; q < EC / 4; ++q)
            *reinterpret_cast<float4*>(F + (int64_t)t * V + vbase + c0 + 4 * q) =
                make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
        } else {
#pragma unroll
          for (int c = 0; c < EC; ++c) F[(int64_t)(vbase + c0 + c) * K + t] = y[c];
        }
      }
      if (step + 1 < n && j.out) {
        if (p.in_place && p.has_h && step + 1 < nsteps)
          if (!(ok = warp_wait16(&ctl->h_full[(step + 1) & 1], ((step + 1) >> 1) & 1, wc))) break;
        store_out(seg_of(step + 1));
        TR16(3, step, 6, trc);
      }
      if (p.has_h && p.release == 2) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->h_empty[slot]);
      }
    }
    // Shared memory may go once the stores have read it; the grid completes
    // only after its global writes are performed.
    if (lane == 0) bulk_wait_read<0>();
    __syncwarp();
  }

  griddep_launch_dependents();
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

#ifdef QLA_TRACE
extern "C" __attribute__((visibility("default"))) int qla_debug_trace16(long long* out, int n) {
  const int total = 4 * 8 * 8 * 16;
  if (n > total) n = total;
  return cudaMemcpyFromSymbol(out, g_qla_trace16, sizeof(long long) * n) == cudaSuccess ? n : -1;
}
#endif

bool tc_f16_supports(int K, int V) { return K == 128 && V % h16::VT == 0 && V >= h16::VT; }

cudaError_t launch_seq_tc_f16(const SeqJob& j, int release, unsigned int* status, uint64_t limit_ns, int stall_test,
                              cudaStream_t stream) {
  using namespace h16;
  if (!tc_f16_supports(j.K, j.V) || !tma_job_supported(j)) return cudaErrorInvalidValue;
  H16Params p;
  memset(&p, 0, sizeof p);
  p.job = j;
  p.status = status;
  p.limit_ns = limit_ns;
  p.has_h = j.H != nullptr;
  p.in_place = j.out != nullptr && (const void*)j.out == (const void*)j.H;
  p.release = release;
  p.stall_test = stall_test;
  if (!make_job_maps(j, VT, EC, &p.map_h, &p.map_out, &p.map_m)) return cudaErrorInvalidValue;
  cudaError_t e = cudaFuncSetAttribute(seq_tc_f16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid = job_grid(j, j.V / VT);
  e = launch_kernel(seq_tc_f16_kernel, grid, 32 * WARPS, SMEM, stream, j.pdl != 0, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace qla
