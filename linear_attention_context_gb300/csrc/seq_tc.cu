// Sequential state correction, warp-specialised tensor-core engine (sm_103a).
//
// Computes the recurrence of Antarx Memos, "一次 TileLang Warp Specialization 数
// 值错误的定位与修复", section "理解三个缓冲区，才能判断哪里需要同步":
// X_{j+1} = A_j X_j + H_j in the kv view, A_j = M (forward) or M^T (reverse),
// out[seg] = the state entering seg.  The page's kernel streams h and m tiles
// into two-slot shared buffers with a TMA producer and lets consumers do the
// GEMM; its bug was a slot released before its last ordinary read.  This
// engine keeps that producer/consumer shape and moves the contraction onto
// tcgen05 with fp32 accuracy from three TF32 products:
//     A X ~= A_hi X_hi + A_hi X_lo + A_lo X_hi,
// The tensor core reads an fp32 operand as TF32 by cutting its 13 low mantissa
// bits toward zero (measured).  Both operands split as hi = RN_tf32(x) and
// lo = x - hi (exact in fp32), and the MMA reads lo cut toward zero.  With hi
// rounded to nearest, lo's sign is that of x times an even coin (x rounded
// down or up), so the cut of lo (below 2^-23 relative to x) and the dropped
// A_lo X_lo term (below 2^-22) carry no bias.  (With hi = trunc(x) instead,
// lo keeps x's sign and a cut lo shrank every state coherently, by about
// 2^-20 per step: measured.)
//
// Accumulation: the tensor core also rounds its fp32 accumulator toward zero,
// so a long chain of MMAs into one accumulator shrinks the result coherently
// (measured about -6e-7 per step with 48 MMAs per output).  The big A_hi X_hi
// terms are therefore spread over NB chains by k-step (no chain sees more than
// 4 big MMAs per step); the two small terms, 2^-11 of the result, take one
// chain each.  The epilogue adds the chains in pairs with round-to-nearest
// fp32 adds.
//
// Issue rate: one thread issues a tcgen05.mma about every 45 cycles, while
// an M=128, N=32, K=8 tf32 MMA keeps the tensor pipe busy for about 17, so
// three threads issue: one the big terms, one A_hi X_lo, one A_lo X_hi, each
// into its own accumulators (no two threads ever accumulate into the same
// TMEM columns).  A barrier poll from an issuing thread waits until that
// thread's queued MMAs have been dispatched (~110 cycles measured), so the
// issuers poll once per pair of chunks, not per chunk.
//
// One CTA owns a VT-column tile of one unit (chain, group) for all of the
// unit's segments.  Roles, storage, handoff and lifetime (the table the
// mlc.ai page "调试 Warp-Specialized Kernels", section "先写清楚数据如何交接",
// asks for):
//
//  role      warps    does
//  producer  0 (1 th) TMA: H_j tile -> h slot j&1; A_j in 32-column chunks
//                     -> m ring (NM stages).  Needs no state: runs ahead.
//  mma       1, 2, 3  (1 thread each) tcgen05.mma kind::tf32, A from TMEM,
//                     B (= X_j hi/lo, K-major, 128-byte swizzle) from shared
//                     memory, D in the accumulator chains (TMEM).
//  splitter  4..11    two warpgroups, alternate chunks: m chunk (ordinary
//                     shared loads) -> hi/lo -> TMEM A ring (NA slots).
//  epilogue  12..      NE warpgroups (four of 8 columns at K = 128, two of 16
//                     at K = 256): H_j (ordinary shared loads, then the h-slot
//                     release) + the chains (tcgen05.ld) = X_{j+1}; its hi/lo
//                     -> B operand first (the next step waits on it), then out
//                     via per-warp TMA stores.  (Stores straight from
//                     registers measured slower: 19.0 against 18.5 us.)
//
//  storage        written by           read by             reusable after
//  m ring [s]     TMA (async)          splitter (generic)  splitter's last read: fence + m_empty arrive
//  h slot [j&1]   TMA (async)          epilogue (generic)  epilogue's last read: fence + h_empty arrive
//  A ring (TMEM)  splitter tcgen05.st  mma (async)         3 commits -> a_empty (per group of 2 chunks)
//  B hi/lo        epilogue st.shared   mma (async)         d_full (3 commits: all MMAs of the step done)
//                 + fence.proxy.async
//  chains (TMEM)  mma                  epilogue tcgen05.ld x_ready (epilogue's wait::ld done)
//  out staging    epilogue st.shared   TMA store (async)   bulk wait_group.read
//                 + fence.proxy.async
//
// Chunks go kc-major: chunk c = kc * HALVES + h is A[128h.., 32kc..], so the
// two row blocks of K = 256 interleave.  Barriers: m_full/h_full count 1 +
// transaction bytes; m_empty count 4 (the splitter warpgroup's warps); a_full
// count 8 (a group of two A slots gets one chunk from each splitter warpgroup);
// h_empty, x_ready count 4 NE (the epilogue warps); a_empty, d_full count 3 (one
// tcgen05.commit per issuing thread).  Producers wait their empty barriers
// with the parity of (use / slots) ^ 1, consumers their full barriers with
// (use / slots), so the first producer wait passes at once.
//
// The slot-release fence (the page's section "三个可用源码方案的具体差别") is
// selectable: membar.cta, fence.proxy.async.shared::cta, none, or a release
// delayed to the end of the slot's use.  It sits between the last ordinary
// shared load of a slot and the arrive on its empty barrier, and every asm
// here carries a "memory" clobber so the compiler keeps that order.
//
// In place (out == H): out[seg] is stored over H[seg] only after the TMA load
// of that tile of H[seg] has completed (its full barrier has been observed).
//
// Every wait is bounded (see ptx.cuh); on expiry the CTA drains its copies in
// flight, frees TMEM and returns with the device status word set.
#include <cuda.h>

#include "ptx.cuh"
#include "qla_internal.h"
#include "tma_map.h"

// Optional pipeline trace (compile with -DQLA_TRACE): clock64() stamps of
// every handoff of CTA (0, 0), read back with qla_debug_trace().  Slots are
// [role][step][event][chunk]; roles 0 producer, 1 mma, 2 splitter, 3 epilogue.
#ifdef QLA_TRACE
__device__ long long g_qla_trace[4 * 8 * 8 * 16];
// Wall-clock (%globaltimer) entry and exit of every CTA of the last 64 calls:
// [call % 64][CTA slot][entry, exit]; CTAs of consecutive calls are told apart
// by the order of an atomic counter (the calls are stream-ordered).
__device__ unsigned long long g_qla_gt[64 * 256 * 2];
__device__ unsigned int g_qla_gt_count;
#define QLA_TR(role, step, ev, ch)                                                                        \
  do {                                                                                                    \
    if (tr && (step) < 8 && (ch) < 16) g_qla_trace[(((role) * 8 + (step)) * 8 + (ev)) * 16 + (ch)] = clock64(); \
  } while (0)
#else
#define QLA_TR(role, step, ev, ch) \
  do {                             \
  } while (0)
#endif

namespace qla {
namespace {

using namespace ptx;

constexpr int kCtaCols = 32;                    // state columns per CTA (TILES x VT)
constexpr uint32_t kChunkBytes = 128 * 32 * 4;  // one A chunk: 128 rows x 32 columns fp32
constexpr uint32_t kTmemCols = 512;

// TILES column tiles of VT columns share one CTA, one M stream and one A
// split; with two, the issuers run all of tile 0's MMAs of a step before
// tile 1's, so tile 0's epilogue overlaps tile 1's MMAs.  (Two tiles, as
// 2 x 32 or 2 x 16 columns, measured slower than one 32-column tile and are
// not launched; the configuration stays generic.)
template <int K, int TILES, int VT>
struct Cfg {
  static constexpr int HALVES = K / 128;          // 128-row MMA blocks of the output
  static constexpr int KCH = K / 32;              // 32-wide k chunks per block
  static constexpr int CPS = HALVES * KCH;        // chunks per step
  static constexpr int NI = 3;                    // MMA-issuing warps (one thread each)
  static constexpr int NB = K == 128 ? 4 : 2;     // big-term chains per row block
  static constexpr int NQ = NB + 2;               // chains per row block (+ A_hi X_lo, A_lo X_hi)
  static constexpr uint32_t ACOL = TILES * HALVES * NQ * VT;  // first column of the A ring
  static constexpr int NA = (int)((kTmemCols - ACOL) / 128) * 2;  // A ring slots (hi, lo: 64 columns each) ...
  static constexpr int NAG = NA / 2;              // ... in groups of two chunks, one barrier pair per group
  static constexpr int NM = (TILES == 2 && VT == 32) ? 4 : (K == 128 ? 6 : 4);  // m ring stages
  static constexpr int NOUT = K == 128 ? 2 : 1;   // out staging buffers per tile
  static constexpr int NSG = 2;                   // splitter warpgroups (take chunks round-robin)
  static constexpr int NE = (TILES == 1 && K == 128) ? 4 : 2;  // epilogue warpgroups per tile ...
  static constexpr int EC = VT / NE;              // ... each owning EC state columns
  static constexpr int SPL_WARP0 = 1 + NI;        // first splitter warp (after producer + issuers)
  static constexpr int EPI_WARP0 = SPL_WARP0 + 4 * NSG;  // first epilogue warp
  static constexpr int WARPS = EPI_WARP0 + 4 * NE * TILES;
  static constexpr uint32_t TILE = (uint32_t)K * VT * 4;  // one state tile (bytes)
  static constexpr uint32_t OFF_M = 0;
  static constexpr uint32_t OFF_H = OFF_M + NM * kChunkBytes;       // [TILES][2 slots]
  static constexpr uint32_t OFF_BHI = OFF_H + TILES * 2 * TILE;     // [TILES] (hi), then [TILES] (lo)
  static constexpr uint32_t OFF_BLO = OFF_BHI + TILES * TILE;
  static constexpr uint32_t OFF_OUT = OFF_BLO + TILES * TILE;       // [TILES][NOUT]
  static constexpr uint32_t OFF_CTRL = OFF_OUT + TILES * NOUT * TILE;
  static constexpr uint32_t CTRL_BYTES = 512;
  static constexpr uint32_t SMEM = OFF_CTRL + CTRL_BYTES + 1024;  // + alignment slack
  static_assert(SMEM <= 232448, "shared memory budget");
  static_assert(ACOL + NA * 64 <= kTmemCols, "TMEM columns");
  static_assert(CPS % 2 == 0 && NAG >= 1 && NAG <= 4, "chunks per step, A groups");
  static_assert(TILES == 1 || K == 128, "two tiles only for K = 128");
  static_assert(TILES * VT == kCtaCols && EC % 8 == 0, "tile widths");
  // A splitter group may wait on a ring slot only for a use whose previous
  // use was its own: otherwise, while another group's fill of the previous
  // use is still in flight, the phase two uses back (same parity) would
  // satisfy its parity wait.  So each ring depth is a multiple of NSG.
  static_assert(NM % NSG == 0 && NA % NSG == 0, "ring depths must be multiples of the splitter groups");
};

struct TcParams {
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

struct Ctrl {
  uint64_t m_full[8], m_empty[8];
  uint64_t a_full[4], a_empty[4];
  uint64_t h_full[2][2], h_empty[2][2];  // [tile][slot]
  uint64_t x_ready[2], d_full[2];        // [tile]
  uint64_t never;
  uint64_t mma_done[3];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(Ctrl) <= 512, "control block");

__device__ __forceinline__ void release_fence(int mode) {
  if (mode == 0) membar_cta();
  else if (mode == 1) fence_proxy_async_smem();
}

// Warp-uniform bounded wait: every lane polls, the warp agrees on the outcome.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const WaitCtl& c) {
  const bool ok = mbar_wait(bar, parity, c);
  return __all_sync(0xffffffffu, ok);
}

// Nearest TF32 value (ties away from zero) as fp32 bits: add half of the
// 13-bit tail, then clear the tail; a carry correctly bumps the exponent.
// (cvt.rna.tf32.f32 gives bit-identical results on GB300 but made the kernel
// slower: 21.5 against 19.1 us per call.)
__device__ __forceinline__ uint32_t tf32_rn_bits(float x) { return (__float_as_uint(x) + 0x1000u) & 0xFFFFE000u; }

// Two values at once: hi = RN_tf32(x), lo = x - hi exactly (one packed fma).
__device__ __forceinline__ void split_tf32x2(float x0, float x1, uint32_t& hi0, uint32_t& hi1, uint32_t& lo0,
                                             uint32_t& lo1) {
  hi0 = tf32_rn_bits(x0);
  hi1 = tf32_rn_bits(x1);
  const float2 d = __ffma2_rn(make_float2(__uint_as_float(hi0), __uint_as_float(hi1)), make_float2(-1.f, -1.f),
                              make_float2(x0, x1));
  lo0 = __float_as_uint(d.x);
  lo1 = __float_as_uint(d.y);
}

// The MMAs one issuing thread owes chunk c (k-block kc = c / HALVES, row
// block h = c % HALVES) of tile `tl`: role 0 the four A_hi X_hi k-steps, role
// 1 the A_hi X_lo ones, role 2 the A_lo X_hi ones.  With c, tl and the role
// compile-time constants every chain index and accumulate flag folds.
template <int K, int TILES, int VT, int ROLE>
__device__ __forceinline__ void mma_chunk(const int tl, const int c, uint32_t tmem, uint32_t a_hi, uint64_t dh0,
                                          uint64_t dl0) {
  using C = Cfg<K, TILES, VT>;
  constexpr uint32_t idesc = idesc_tf32(128, VT);
  const int kc = c / C::HALVES, h = c % C::HALVES;
  const int q0 = (tl * C::HALVES + h) * C::NQ;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const int ks = kc * 4 + s;  // k-step within the row block: B rows [8 ks, 8 ks + 8)
    // B rows of k-step ks: k-block kc, 32 bytes per 8 tf32 inside the swizzled row
    const uint64_t off = (uint64_t)(((uint32_t)kc * (VT * 128) + (uint32_t)s * 32) >> 4);
    if (ROLE == 0)
      mma_tf32_ts(tmem + (q0 + ks % C::NB) * VT, a_hi + s * 8, dh0 + off, idesc, ks >= C::NB);
    else if (ROLE == 1)
      mma_tf32_ts(tmem + (q0 + C::NB) * VT, a_hi + s * 8, dl0 + off, idesc, ks > 0);
    else
      mma_tf32_ts(tmem + (q0 + C::NB + 1) * VT, a_hi + 32 + s * 8, dh0 + off, idesc, ks > 0);
  }
}

// The operands of one issuer's 16 MMAs of a step (K = 128, one tile), the
// same every step: D chain, A slot column, B descriptor low word.  Computed
// once, so a step's issue is the MMA instructions alone.
template <int VT, int ROLE>
struct MmaOps {
  uint32_t d[16], a[16], b[16];
};

template <int K, int TILES, int VT, int ROLE>
__device__ __forceinline__ MmaOps<VT, ROLE> mma_ops(uint32_t tmem, uint64_t dh0, uint64_t dl0) {
  using C = Cfg<K, TILES, VT>;
  MmaOps<VT, ROLE> o;
#pragma unroll
  for (int m = 0; m < 16; ++m) {
    const int c = m / 4, s = m % 4, ks = m;
    const uint32_t off = ((uint32_t)c * (VT * 128) + (uint32_t)s * 32) >> 4;
    o.d[m] = tmem + (uint32_t)(ROLE == 0 ? ks % C::NB : ROLE == 1 ? C::NB : C::NB + 1) * VT;
    o.a[m] = tmem + C::ACOL + (uint32_t)c * 64 + (ROLE == 2 ? 32u : 0u) + (uint32_t)s * 8;
    o.b[m] = (uint32_t)(ROLE == 1 ? dl0 : dh0) + off;
  }
  return o;
}

// Chunks C0..C1 of a step from precomputed operands.
template <int K, int TILES, int VT, int ROLE, int C0, int C1>
__device__ __forceinline__ void mma_issue(const MmaOps<VT, ROLE>& o, uint32_t bhi) {
  using C = Cfg<K, TILES, VT>;
  constexpr uint32_t idesc = idesc_tf32(128, VT);
#pragma unroll
  for (int m = 4 * C0; m < 4 * C1 + 4; ++m) {
    if ((ROLE == 0 && m < C::NB) || (ROLE != 0 && m == 0))
      mma_tf32_ts_c<false>(o.d[m], o.a[m], o.b[m], bhi, idesc);
    else
      mma_tf32_ts_c<true>(o.d[m], o.a[m], o.b[m], bhi, idesc);
  }
}

template <int K, int TILES, int VT, int ROLE>
__device__ __forceinline__ void mma_role(Ctrl* ctl, uint8_t* smem, uint32_t tmem, int nsteps, const WaitCtl& wc
#ifdef QLA_TRACE
                                         ,
                                         bool tr
#endif
) {
  using C = Cfg<K, TILES, VT>;
  // Descriptors of the k-block 0 rows of each tile's B hi / lo; every other
  // k-step adds a compile-time byte offset (>> 4) to the start-address field.
  uint64_t dh0[TILES], dl0[TILES];
#pragma unroll
  for (int tl = 0; tl < TILES; ++tl) {
    dh0[tl] = smem_desc_sw128(smem_u32(smem + C::OFF_BHI + tl * C::TILE), 1024);
    dl0[tl] = smem_desc_sw128(smem_u32(smem + C::OFF_BLO + tl * C::TILE), 1024);
  }
  int grp0 = 0;
  uint32_t phase0 = 0;
  bool ok = true;
  [[maybe_unused]] MmaOps<VT, ROLE> ops;
  [[maybe_unused]] uint32_t bhi = (uint32_t)(dh0[0] >> 32);  // the same for the hi and lo descriptors
  if constexpr (TILES == 1 && C::CPS == 4 && C::NAG == 2) ops = mma_ops<K, TILES, VT, ROLE>(tmem, dh0[0], dl0[0]);
  for (int step = 0; step < nsteps && ok; ++step) {
#pragma unroll
    for (int tl = 0; tl < TILES && ok; ++tl) {
      if (!(ok = mbar_wait(&ctl->x_ready[tl], step & 1, wc))) break;
      if (tl == 0) QLA_TR(1, step, 0, ROLE);
      tc_fence_after();
      if constexpr (TILES == 1 && C::CPS == 4 && C::NAG == 2) {
        // The A ring holds exactly one step (two pairs).  Pair 1 is usually
        // split before the step starts: test it without blocking, so that
        // no poll (which would stall until this thread's queued MMAs have
        // dispatched) sits between the step's MMAs unless it must.
        if (!(ok = mbar_wait(&ctl->a_full[0], phase0, wc))) break;
        const bool pair1_ready = mbar_test_wait(&ctl->a_full[1], phase0);
        QLA_TR(1, step, 1, 4 * ROLE);
        tc_fence_after();
        mma_issue<K, TILES, VT, ROLE, 0, 1>(ops, bhi);
        mma_commit(&ctl->a_empty[0]);
        QLA_TR(1, step, 3, 4 * ROLE);
        if (!pair1_ready) {
          if (!(ok = mbar_wait(&ctl->a_full[1], phase0, wc))) break;
          tc_fence_after();
        }
        QLA_TR(1, step, 1, 2 + 4 * ROLE);
        mma_issue<K, TILES, VT, ROLE, 2, 3>(ops, bhi);
        mma_commit(&ctl->a_empty[1]);
        mma_commit(&ctl->d_full[0]);
        QLA_TR(1, step, 3, 2 + 4 * ROLE);
        phase0 ^= 1;
        continue;
      }
      int grp = grp0;
      uint32_t phase = phase0;
      // One wait and one commit per pair of chunks: a barrier poll from this
      // thread stalls until its queued MMAs have been dispatched.  The A
      // pairs are waited for by tile 0 and released after the last tile.
#pragma unroll
      for (int c = 0; c < C::CPS; c += 2) {
        if (tl == 0) {
          if (!(ok = mbar_wait(&ctl->a_full[grp], phase, wc))) break;
          QLA_TR(1, step, 1, c + 4 * ROLE);
          tc_fence_after();
        }
        mma_chunk<K, TILES, VT, ROLE>(tl, c, tmem, tmem + C::ACOL + (2 * grp) * 64, dh0[tl], dl0[tl]);
        if (tl == 0) QLA_TR(1, step, 2, c + 4 * ROLE);
        mma_chunk<K, TILES, VT, ROLE>(tl, c + 1, tmem, tmem + C::ACOL + (2 * grp + 1) * 64, dh0[tl], dl0[tl]);
        if (tl == 0) QLA_TR(1, step, 2, c + 1 + 4 * ROLE);
        if (tl == TILES - 1) mma_commit(&ctl->a_empty[grp]);
        if (tl == 0) QLA_TR(1, step, 3, c + 4 * ROLE);
        if (++grp == C::NAG) {
          grp = 0;
          phase ^= 1;
        }
      }
      if (ok) mma_commit(&ctl->d_full[tl]);
      if (tl == TILES - 1) {
        grp0 = grp;
        phase0 = phase;
      }
    }
  }
  // All MMAs this thread issued must finish before TMEM is freed.
  mma_commit(&ctl->mma_done[ROLE]);
  mbar_wait_drain(&ctl->mma_done[ROLE], 0, 200000000ull);
}

template <int K, int TILES, int VT>
__global__ void __launch_bounds__(32 * Cfg<K, TILES, VT>::WARPS, 1) seq_tc_kernel(const __grid_constant__ TcParams p) {
  using C = Cfg<K, TILES, VT>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  Ctrl* ctl = reinterpret_cast<Ctrl*>(smem + C::OFF_CTRL);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const SeqJob& j = p.job;
#ifdef QLA_TRACE
  __shared__ unsigned int gt_slot;
  if (threadIdx.x == 0) {
    const unsigned long long now = globaltimer();
    const unsigned int idx = atomicAdd(&g_qla_gt_count, 1u);
    const unsigned int nb = gridDim.x * gridDim.y;
    gt_slot = ((idx / nb) % 64) * 256 + (blockIdx.y * gridDim.x + blockIdx.x) % 256;
    g_qla_gt[gt_slot * 2] = now;
  }
#endif
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
  const int vbase = tile * (TILES * VT);
  if (n <= 0) {  // a sequence without segments: its final state is its initial state
    if (j.fin) {
      float* F = j.fin + u * j.fin_unit_stride;
      const float* I = j.init_mode == kInitPointer ? j.init + u * j.init_unit_stride : nullptr;
      for (int e = threadIdx.x; e < K * TILES * VT; e += blockDim.x) {
        const int k = e / (TILES * VT), v = vbase + e % (TILES * VT);
        const int64_t idx = j.layout == 0 ? (int64_t)k * j.V + v : (int64_t)v * K + k;
        F[idx] = I ? I[idx] : (j.init_mode == kInitIdentity && k == v ? 1.f : 0.f);
      }
    }
    return;
  }
  const bool fwd = j.direction == 0;
  auto seg_of = [&](int step) { return fwd ? s_lo + step : s_lo + n - 1 - step; };
#ifdef QLA_TRACE
  const bool tr = blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 &&
                  ((threadIdx.x & 31) == 0 &&
                   (warp <= C::NI || warp == C::SPL_WARP0 || warp == C::SPL_WARP0 + 4 || warp == C::EPI_WARP0 ||
                    warp == C::WARPS - 1));
  const int trc = warp == C::WARPS - 1 ? 1 : 0;  // second traced epilogue warp
  (void)trc;
#endif

  // Epilogue warps load the initial state before set-up, so its global-memory
  // latency overlaps barrier initialisation and the TMEM allocation.
  constexpr int EC = C::EC;
  float y[C::HALVES][EC];
  if (warp >= C::EPI_WARP0) {
    const int e = ((warp - C::EPI_WARP0) >> 2) % C::NE;
    const int t = 32 * (warp & 3) + lane;
    const int v0 = vbase + ((warp - C::EPI_WARP0) / (4 * C::NE)) * VT;
    const int c0 = e * EC;
    const int V = j.V;
#pragma unroll
    for (int h = 0; h < C::HALVES; ++h) {
      const int k = t + 128 * h;
      if (j.init_mode == kInitPointer) {
        const float* src = j.init + u * j.init_unit_stride;
        if (j.layout == 0) {
#pragma unroll
          for (int q = 0; q < EC / 4; ++q) {
            const float4 v = *reinterpret_cast<const float4*>(src + (int64_t)k * V + v0 + c0 + 4 * q);
            y[h][4 * q] = v.x; y[h][4 * q + 1] = v.y; y[h][4 * q + 2] = v.z; y[h][4 * q + 3] = v.w;
          }
        } else {
#pragma unroll
          for (int c = 0; c < EC; ++c) y[h][c] = src[(int64_t)(v0 + c0 + c) * K + k];
        }
      } else {
#pragma unroll
        for (int c = 0; c < EC; ++c) y[h][c] = (j.init_mode == kInitIdentity && k == v0 + c0 + c) ? 1.f : 0.f;
      }
    }
  }

  if (threadIdx.x == 0) {
    // The first TMA of a map fetches its descriptor: start that before set-up.
    prefetch_tensormap(&p.map_m);
    if (p.has_h) prefetch_tensormap(&p.map_h);
    if (j.out) prefetch_tensormap(&p.map_out);
    for (int i = 0; i < C::NM; ++i) {
      mbar_init(&ctl->m_full[i], 1);
      mbar_init(&ctl->m_empty[i], 4);
    }
    for (int i = 0; i < C::NAG; ++i) {
      mbar_init(&ctl->a_full[i], 8);   // two splitter warpgroups fill one chunk each of the group
      mbar_init(&ctl->a_empty[i], C::NI);  // one commit per issuing thread
    }
    for (int tl = 0; tl < TILES; ++tl) {
      for (int i = 0; i < 2; ++i) {
        mbar_init(&ctl->h_full[tl][i], 1);
        mbar_init(&ctl->h_empty[tl][i], 4 * C::NE);  // the tile's epilogue warps
      }
      mbar_init(&ctl->x_ready[tl], 4 * C::NE);
      mbar_init(&ctl->d_full[tl], C::NI);
    }
    mbar_init(&ctl->never, 1);
    for (int i = 0; i < C::NI; ++i) mbar_init(&ctl->mma_done[i], 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  // The first step's loads need no TMEM and no other thread: the producer
  // thread issues them before the set-up barrier, so their DRAM latency runs
  // under the TMEM allocation and the barrier.  These are the first uses of
  // their slots (no empty wait); the producer loop continues after them.
  int pre_m = 0;   // M chunks of step 0 already issued (ring stages 0 ..)
  bool pre_h = false;
  if (threadIdx.x == 0 && nsteps > 0) {
    const int64_t mrow0 = (cbase + seg_of(0)) * K;
    pre_m = C::CPS < C::NM ? C::CPS : C::NM;
    for (int c = 0; c < pre_m; ++c) {
      mbar_arrive_expect_tx(&ctl->m_full[c], kChunkBytes);
      const int kc = c / C::HALVES, h = c % C::HALVES;
      uint8_t* dst = smem + C::OFF_M + c * kChunkBytes;
      if (fwd)
        tma_load_2d(dst, &p.map_m, 32 * kc, (int32_t)(mrow0 + 128 * h), &ctl->m_full[c]);
      else
        tma_load_2d(dst, &p.map_m, 128 * h, (int32_t)(mrow0 + 32 * kc), &ctl->m_full[c]);
    }
    if (p.has_h) {
      const int64_t hrow0 = (cbase + seg_of(0)) * (j.layout == 0 ? K : j.V);
      for (int tl = 0; tl < TILES; ++tl) {
        mbar_arrive_expect_tx(&ctl->h_full[tl][0], C::TILE);
        uint8_t* dst = smem + C::OFF_H + (tl * 2) * C::TILE;
        const int v0 = vbase + tl * VT;
        if (j.layout == 0)
          tma_load_2d(dst, &p.map_h, v0, (int32_t)hrow0, &ctl->h_full[tl][0]);
        else
          tma_load_2d(dst, &p.map_h, 0, (int32_t)(hrow0 + v0), &ctl->h_full[tl][0]);
      }
      pre_h = true;
    }
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
  QLA_TR(0, 0, 7, 0);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      uint32_t mit = (uint32_t)pre_m;
      int hissued[TILES] = {};
      if (pre_h)
        for (int tl = 0; tl < TILES; ++tl) hissued[tl] = 1;
      bool ok = true;
      const int hrows = j.layout == 0 ? K : j.V;  // rows of one state in the 2-D view of H
      for (int step = 0; step < nsteps && ok; ++step) {
        const int seg = seg_of(step);
        const int64_t mrow0 = (cbase + seg) * K;
        auto load_h = [&]() {
          if (!p.has_h) return;
          const int slot = step & 1;
          const int64_t hrow0 = (cbase + seg) * hrows;
          for (int tl = 0; tl < TILES && ok; ++tl) {
            if (!(ok = mbar_wait(&ctl->h_empty[tl][slot], ((step >> 1) & 1) ^ 1, wc))) break;
            mbar_arrive_expect_tx(&ctl->h_full[tl][slot], C::TILE);
            uint8_t* dst = smem + C::OFF_H + (tl * 2 + slot) * C::TILE;
            const int v0 = vbase + tl * VT;
            if (j.layout == 0)
              tma_load_2d(dst, &p.map_h, v0, (int32_t)hrow0, &ctl->h_full[tl][slot]);
            else
              tma_load_2d(dst, &p.map_h, 0, (int32_t)(hrow0 + v0), &ctl->h_full[tl][slot]);
            ++hissued[tl];
          }
          QLA_TR(0, step, 0, 0);
        };
        auto load_m = [&]() {
          for (int c = step == 0 ? pre_m : 0; c < C::CPS && ok; ++c, ++mit) {
            const int stage = mit % C::NM;
            if (!(ok = mbar_wait(&ctl->m_empty[stage], ((mit / C::NM) & 1) ^ 1, wc))) break;
            QLA_TR(0, step, 1, c);
            mbar_arrive_expect_tx(&ctl->m_full[stage], kChunkBytes);
            const int kc = c / C::HALVES, h = c % C::HALVES;
            uint8_t* dst = smem + C::OFF_M + stage * kChunkBytes;
            if (fwd)  // A = M: rows 128h.., columns 32kc..  (128-byte swizzle, box 32 x 128)
              tma_load_2d(dst, &p.map_m, 32 * kc, (int32_t)(mrow0 + 128 * h), &ctl->m_full[stage]);
            else      // A = M^T: M rows 32kc.., columns 128h..  (box 128 x 32)
              tma_load_2d(dst, &p.map_m, 128 * h, (int32_t)(mrow0 + 32 * kc), &ctl->m_full[stage]);
          }
        };
        // The first step needs its M chunks before its H tile (the split and
        // the MMAs come before the drain); later steps' M chunks wait for ring
        // slots, so their H tile goes first.
        if (step == 0) {
          load_m();
          if (ok && !pre_h) load_h();
        } else {
          load_h();
          if (ok) load_m();
        }
      }
      // Drain: every issued load must land before shared memory goes away.
      const uint64_t drain = 200000000ull;  // 200 ms
      for (int s = 0; s < C::NM; ++s) {
        const uint32_t uses = mit > (uint32_t)s ? (mit - 1 - s) / C::NM + 1 : 0;
        if (uses) mbar_wait_drain(&ctl->m_full[s], (uses - 1) & 1, drain);
      }
      for (int tl = 0; tl < TILES; ++tl)
        for (int s = 0; s < 2; ++s) {
          const int uses = hissued[tl] > s ? (hissued[tl] - 1 - s) / 2 + 1 : 0;
          if (uses) mbar_wait_drain(&ctl->h_full[tl][s], (uses - 1) & 1, drain);
        }
    }
    __syncwarp();
  } else if (warp <= C::NI) {
    // ------------------------------------------------------------ mma issuers
    if (lane == 0) {
#ifdef QLA_TRACE
      if (warp == 1) mma_role<K, TILES, VT, 0>(ctl, smem, tmem, nsteps, wc, tr);
      else if (warp == 2) mma_role<K, TILES, VT, 1>(ctl, smem, tmem, nsteps, wc, tr);
      else mma_role<K, TILES, VT, 2>(ctl, smem, tmem, nsteps, wc, tr);
#else
      if (warp == 1) mma_role<K, TILES, VT, 0>(ctl, smem, tmem, nsteps, wc);
      else if (warp == 2) mma_role<K, TILES, VT, 1>(ctl, smem, tmem, nsteps, wc);
      else mma_role<K, TILES, VT, 2>(ctl, smem, tmem, nsteps, wc);
#endif
    }
    __syncwarp();
  } else if (warp < C::EPI_WARP0) {
    // ------------------------------------------------------------ A splitters
    const int grp = (warp - C::SPL_WARP0) >> 2;      // takes chunks grp, grp + NSG, grp + 2 NSG, ...
    const int t = 32 * (warp & 3) + lane;            // A row within the 128-row block = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;
    const int total = nsteps * C::CPS;
    int stage = grp;
    uint32_t mphase = 0;
    bool ok = true;
    for (int mit = grp; mit < total && ok; mit += C::NSG) {
      const int step = mit / C::CPS, c = mit % C::CPS;
      (void)step;
      (void)c;
      if (!(ok = warp_wait(&ctl->m_full[stage], mphase, wc))) break;
      QLA_TR(2, step, 0, c);
      const uint8_t* chunk = smem + C::OFF_M + stage * kChunkBytes;
      const int aslot = mit % C::NA, agrp = aslot >> 1;
      const uint32_t aphase = (uint32_t)(mit / C::NA) & 1;
      const uint32_t a = tmem + lane_off + C::ACOL + aslot * 64;
      // Two 16-column halves: read (ordinary shared loads), then split and
      // store to TMEM.  The slot is released after the second half's read.
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
        if (half == 1 && p.release != 2) {  // the slot's last ordinary read is done: release it
          release_fence(p.release);
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->m_empty[stage]);
        }
        if (half == 0) {
          if (!(ok = warp_wait(&ctl->a_empty[agrp], aphase ^ 1, wc))) break;
          QLA_TR(2, step, 1, c);
          tc_fence_after();
        }
        uint32_t hi[16], lo[16];
#pragma unroll
        for (int k = 0; k < 16; k += 2) split_tf32x2(x[k], x[k + 1], hi[k], hi[k + 1], lo[k], lo[k + 1]);
        tmem_st16(a + 16 * half, hi);
        tmem_st16(a + 32 + 16 * half, lo);
      }
      if (!ok) break;
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&ctl->a_full[agrp]);
      QLA_TR(2, step, 2, c);
      if (p.release == 2) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->m_empty[stage]);
      }
      if ((stage += C::NSG) >= C::NM) {
        stage -= C::NM;
        mphase ^= 1;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int ew = warp - C::EPI_WARP0;
    const int tl = ew / (4 * C::NE);                 // tile
    const int e = (ew >> 2) % C::NE;                 // column group of the tile: [EC e, EC e + EC)
    const int wq = warp & 3;
    const int t = 32 * wq + lane;                    // output row within a 128-row block = TMEM lane
    const uint32_t lane_off = (uint32_t)(32 * wq) << 16;
    const int V = j.V;
    const int c0 = e * EC;
    const int v0 = vbase + tl * VT;
    uint8_t* bhi = smem + C::OFF_BHI + tl * C::TILE;
    uint64_t* x_ready = &ctl->x_ready[tl];
    uint64_t* d_full = &ctl->d_full[tl];
    int out_count = 0;
    bool ok = true;
#ifdef QLA_TRACE
    int step_tr = 0;
#endif

    // out[seg] <- y through per-warp staging (32 x EC floats per row block) and TMA stores
    auto store_out = [&](int seg) {
      const int b = out_count % C::NOUT;
      if (lane == 0) bulk_wait_read<C::NOUT - 1>();
      __syncwarp();
      uint8_t* stg_base = smem + C::OFF_OUT + (tl * C::NOUT + b) * C::TILE;
#pragma unroll
      for (int h = 0; h < C::HALVES; ++h) {
        float* stg = reinterpret_cast<float*>(stg_base + ((h * C::NE + e) * 4 + wq) * (32 * EC * 4));
        if (j.layout == 0) {  // [32 rows][EC floats], (4 EC)-byte swizzle: 16-byte piece q of row r at
                              // q ^ ((r EC / 32) % (EC / 4))
#pragma unroll
          for (int q = 0; q < EC / 4; ++q)
            *reinterpret_cast<float4*>(stg + lane * EC + 4 * (q ^ ((lane * EC / 32) & (EC / 4 - 1)))) =
                make_float4(y[h][4 * q], y[h][4 * q + 1], y[h][4 * q + 2], y[h][4 * q + 3]);
        } else {              // [EC rows][32 floats]: column `lane`
#pragma unroll
          for (int c = 0; c < EC; ++c) stg[c * 32 + lane] = y[h][c];
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          const uint8_t* stg = stg_base + ((h * C::NE + e) * 4 + wq) * (32 * EC * 4);
          if (j.layout == 0)
            tma_store_2d(&p.map_out, stg, v0 + c0,
                         (int32_t)((cbase + seg) * K + 128 * h + 32 * wq));
          else
            tma_store_2d(&p.map_out, stg, 128 * h + 32 * wq, (int32_t)((cbase + seg) * V + v0 + c0));
        }
        bulk_commit();
      }
      ++out_count;
    };

    // X -> B operand (hi and lo), K-major, 128-byte swizzle: element (n, k) of
    // B^T sits in k-block k/32, row n, 16-byte piece ((k%32)/4) ^ (n%8).  The
    // shared addresses of this thread's elements (row k = t, its EC columns)
    // are fixed: computed once; row k + 128 is 4 k-blocks further, B_lo one
    // tile-set further.
    uint32_t baddr[EC];
    {
      const uint32_t kb = (uint32_t)(t >> 5) * (VT * 128) + (uint32_t)(t & 3) * 4 + (uint32_t)(c0 >> 3) * 1024;
      const uint32_t piece = (uint32_t)((t & 31) >> 2);
#pragma unroll
      for (int c = 0; c < EC; ++c)
        baddr[c] = smem_u32(bhi) + kb + (uint32_t)(c & 7) * 128 + ((piece ^ (uint32_t)(c & 7)) << 4) +
                   (uint32_t)(c >> 3) * 1024;
    }
    auto write_b = [&]() {
      constexpr uint32_t kLo = C::OFF_BLO - C::OFF_BHI;
      constexpr uint32_t kHalf = 4 * VT * 128;  // row k + 128
#pragma unroll
      for (int h = 0; h < C::HALVES; ++h) {
#pragma unroll
        for (int c = 0; c < EC; c += 2) {
          uint32_t h0, h1, l0, l1;
          split_tf32x2(y[h][c], y[h][c + 1], h0, h1, l0, l1);
          if (h == 0) {
            sts32<0>(baddr[c], h0);
            sts32<kLo>(baddr[c], l0);
            sts32<0>(baddr[c + 1], h1);
            sts32<kLo>(baddr[c + 1], l1);
          } else {
            sts32<kHalf>(baddr[c], h0);
            sts32<kLo + kHalf>(baddr[c], l0);
            sts32<kHalf>(baddr[c + 1], h1);
            sts32<kLo + kHalf>(baddr[c + 1], l1);
          }
        }
      }
      QLA_TR(3, step_tr, 7, trc);
      fence_proxy_async_smem();  // generic writes -> read by tcgen05.mma (async proxy)
    };

    // acc += the accumulator chains of one 128-row block (this warpgroup's EC
    // columns), in pairs, round-to-nearest: big chains first, then the small.
    // (Loading all chains before a single wait measured slower.)
    auto drain_add = [&](int h, float (&acc)[EC]) {
      float a[EC], b[EC];
      const uint32_t base = tmem + lane_off + (uint32_t)((tl * C::HALVES + h) * C::NQ * VT + c0);
      static_assert(C::NQ % 2 == 0, "chains are drained in pairs");
#pragma unroll
      for (int q = 0; q < C::NQ; q += 2) {
        tmem_ld<EC>(base + q * VT, a);
        tmem_ld<EC>(base + (q + 1) * VT, b);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < EC; c += 2) {  // acc += a + b, two columns per packed add
          const float2 sab = __fadd2_rn(make_float2(a[c], a[c + 1]), make_float2(b[c], b[c + 1]));
          const float2 r = __fadd2_rn(make_float2(acc[c], acc[c + 1]), sab);
          acc[c] = r.x;
          acc[c + 1] = r.y;
        }
      }
    };

    if (nsteps > 0) {  // X_0 -> B operand first: the first step's MMAs wait on it
      write_b();
      __syncwarp();
      if (lane == 0) mbar_arrive(x_ready);
    }
    if (j.out) {
      if (p.in_place && p.has_h && nsteps > 0) ok = warp_wait(&ctl->h_full[tl][0], 0, wc);
      if (ok) store_out(seg_of(0));
    }
    for (int step = 0; step < nsteps && ok; ++step) {
#ifdef QLA_TRACE
      step_tr = step + 1;
#endif
      // H_j into the accumulator registers first: it does not depend on the MMAs
      const int slot = step & 1;
      if (p.has_h) {
        if (!(ok = warp_wait(&ctl->h_full[tl][slot], (step >> 1) & 1, wc))) break;
        QLA_TR(3, step, 2, trc);
        const uint8_t* ht = smem + C::OFF_H + (tl * 2 + slot) * C::TILE;
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          const int k = t + 128 * h;
          if (j.layout == 0) {  // [K rows][VT floats], (4 VT)-byte swizzle: 16-byte piece p of row k
                                // at p ^ ((k VT / 32) % (VT / 4)); this warp's pieces are c0/4 ..
            const uint8_t* row = ht + k * (VT * 4);
#pragma unroll
            for (int q = 0; q < EC / 4; ++q) {
              const float4 v = *reinterpret_cast<const float4*>(row + (((c0 / 4 + q) ^ ((k * VT / 32) & (VT / 4 - 1))) << 4));
              y[h][4 * q] = v.x; y[h][4 * q + 1] = v.y; y[h][4 * q + 2] = v.z; y[h][4 * q + 3] = v.w;
            }
          } else {              // [VT rows][K floats]
            const float* f = reinterpret_cast<const float*>(ht) + k;
#pragma unroll
            for (int c = 0; c < EC; ++c) y[h][c] = f[(c0 + c) * K];
          }
        }
        if (p.release != 2) {  // the h slot's last ordinary read is done: release it
          release_fence(p.release);
          __syncwarp();
          if (lane == 0) mbar_arrive(&ctl->h_empty[tl][slot]);
        }
      } else {
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h)
#pragma unroll
          for (int c = 0; c < EC; ++c) y[h][c] = 0.f;
      }
      uint64_t* dbar = (p.stall_test && step == 0) ? &ctl->never : d_full;
      if (!(ok = warp_wait(dbar, step & 1, wc))) break;
      QLA_TR(3, step, 1, trc);
      tc_fence_after();
#pragma unroll
      for (int h = 0; h < C::HALVES; ++h) drain_add(h, y[h]);
      QLA_TR(3, step, 5, trc);
      if (step + 1 < nsteps) {  // X_{j+1} -> B operand: the critical path to the next step
        write_b();
        QLA_TR(3, step, 6, trc);
        tc_fence_before();  // the chains have been read (wait::ld in drain_add)
        __syncwarp();
        if (lane == 0) mbar_arrive(x_ready);
        QLA_TR(3, step, 4, trc);
      } else if (j.fin) {
        float* F = j.fin + u * j.fin_unit_stride;
#pragma unroll
        for (int h = 0; h < C::HALVES; ++h) {
          const int k = t + 128 * h;
          if (j.layout == 0) {
#pragma unroll
            for (int q = 0; q < EC / 4; ++q)
              *reinterpret_cast<float4*>(F + (int64_t)k * V + v0 + c0 + 4 * q) =
                  make_float4(y[h][4 * q], y[h][4 * q + 1], y[h][4 * q + 2], y[h][4 * q + 3]);
          } else {
#pragma unroll
            for (int c = 0; c < EC; ++c) F[(int64_t)(v0 + c0 + c) * K + k] = y[h][c];
          }
        }
      }
      if (step + 1 < n && j.out) {
        if (p.in_place && p.has_h && step + 1 < nsteps)
          if (!(ok = warp_wait(&ctl->h_full[tl][(step + 1) & 1], ((step + 1) >> 1) & 1, wc))) break;
        store_out(seg_of(step + 1));
        QLA_TR(3, step, 3, trc);
      }
      if (p.has_h && p.release == 2) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&ctl->h_empty[tl][slot]);
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
#ifdef QLA_TRACE
  __syncthreads();
  if (threadIdx.x == 0) g_qla_gt[gt_slot * 2 + 1] = globaltimer();
#endif
}

// ---------------------------------------------------------------- host side

template <int K, int TILES, int VT>
cudaError_t launch_k(const SeqJob& j, int release, unsigned int* status, uint64_t limit_ns, int stall_test,
                     cudaStream_t stream) {
  using C = Cfg<K, TILES, VT>;
  TcParams p;
  memset(&p, 0, sizeof p);
  p.job = j;
  p.status = status;
  p.limit_ns = limit_ns;
  p.has_h = j.H != nullptr;
  p.in_place = j.out != nullptr && (const void*)j.out == (const void*)j.H;
  p.release = release;
  p.stall_test = stall_test;
  if (!make_job_maps(j, VT, C::EC, &p.map_h, &p.map_out, &p.map_m)) return cudaErrorInvalidValue;
  auto kern = seq_tc_kernel<K, TILES, VT>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (e != cudaSuccess) return e;
  const dim3 grid = job_grid(j, j.V / (TILES * VT));
  e = launch_kernel(kern, grid, 32 * C::WARPS, C::SMEM, stream, j.pdl != 0, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

#ifdef QLA_TRACE
extern "C" __attribute__((visibility("default"))) int qla_debug_walltimes(unsigned long long* out, int n) {
  const int total = 64 * 256 * 2;
  if (n > total) n = total;
  return cudaMemcpyFromSymbol(out, g_qla_gt, sizeof(unsigned long long) * n) == cudaSuccess ? n : -1;
}

extern "C" __attribute__((visibility("default"))) int qla_debug_trace(long long* out, int n) {
  const int total = 4 * 8 * 8 * 16;
  if (n > total) n = total;
  return cudaMemcpyFromSymbol(out, g_qla_trace, sizeof(long long) * n) == cudaSuccess ? n : -1;
}
#endif

bool tc_supports(int K, int V) { return (K == 128 || K == 256) && V % kCtaCols == 0 && V >= kCtaCols; }

cudaError_t launch_seq_tc(const SeqJob& job, int release, unsigned int* status, uint64_t limit_ns, int stall_test,
                          cudaStream_t stream) {
  if (!tc_supports(job.K, job.V) || !tma_job_supported(job)) return cudaErrorInvalidValue;
  // One column tile per CTA.  (Two tiles per CTA, with tile 0's epilogue
  // overlapping tile 1's MMAs, measured slower on the 32-head K=V=128 S=8
  // workload: 27.6 us against 19.9 us per call.)
  if (job.K == 256) return launch_k<256, 1, 32>(job, release, status, limit_ns, stall_test, stream);
  // (Two independent 16-column halves per CTA, one's epilogue overlapping the
  // other's MMAs, measured slower: 23.9 against 18.5 us; the A splitters could
  // not keep up.)
  return launch_k<128, 1, 32>(job, release, status, limit_ns, stall_test, stream);
}

}  // namespace qla
