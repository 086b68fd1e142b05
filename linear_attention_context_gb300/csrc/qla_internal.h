// Internal interfaces between the host API (api.cpp) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace qla {

// One launch of the sequential recurrence over a set of independent units.
//
// A unit is (chain, group): chain c in [0, nchains) selects H, M (and out)
// through the chain strides; group g in [0, G) covers the segments
// [g*L, min(g*L + L, S)).  Inside a unit the segments are visited ascending
// (forward) or descending (reverse); the unit writes out[seg] for each of its
// segments (the state entering that segment, in visiting order) and, when
// `fin` is set, the state after its last segment.  The plain call is G = 1,
// L = S; the scan variant uses the other forms.
struct SeqJob {
  const float* H;       // local states, [nchains][S][state]; nullptr = zero local states
  const float* M;       // propagation matrices, [nchains][S][K][K]
  const float* init;    // initial state per unit (init_mode 1)
  float* out;           // [nchains][S][state] or nullptr
  float* fin;           // final state per unit or nullptr
  int64_t h_chain_stride;    // elements between chains of H and out
  int64_t m_chain_stride;    // elements between chains of M
  int64_t init_unit_stride;  // elements between units' initial states
  int64_t fin_unit_stride;   // elements between units' final states
  int nchains, S, L, G;
  int K, V, layout, direction;
  int init_mode;  // 0 zeros, 1 pointer, 2 identity (K == V)
  // Variable length (cu_seg != nullptr): H, out are [heads][T][state],
  // M [heads][T][K][K]; chain c = n * heads + h covers head h's segments
  // cu_seg[n] .. cu_seg[n+1] - 1 (device memory, N + 1 offsets).
  const int* cu_seg;
  int heads, T;
  int64_t nstates;        // states in H / out / M (nchains * S, or heads * T)
  unsigned int* status;   // device status word (bit 1: invalid offsets)
  int pdl;                // launch as a programmatic dependent of the stream's previous kernel
};

enum InitMode { kInitZero = 0, kInitPointer = 1, kInitIdentity = 2 };

// Device status word bits.
constexpr unsigned int kStatusTimeout = 1u;     // a bounded wait gave up
constexpr unsigned int kStatusBadOffsets = 2u;  // variable-length offsets outside [0, T], decreasing, or
                                                // a sequence longer than the scan's bound

#ifdef __CUDACC__
// Programmatic dependent launch (xuesongtap, "PTX 内存一致性", section on PDL):
// a kernel launched with programmatic stream serialization may start while the
// stream's previous kernel is still running, once that kernel's CTAs have all
// issued launch_dependents or exited.  The trigger says nothing about data:
// griddepcontrol.wait returns only after the prerequisite grids have completed
// and their memory operations are visible, so every kernel here executes it
// before its first global-memory access (it returns at once when the launch
// has no programmatic prerequisite).  The "memory" clobbers keep the compiler
// from moving loads, non-coherent ones included, above the wait.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The segments of chain `chain`: index of its first segment in the packed
// arrays and its segment count.  Returns false, after recording the event in
// the status word, when its variable-length offsets are invalid or its
// sequence is longer than the launch's L * G segments (the chain is then
// skipped: nothing is read or written for it).
__device__ __forceinline__ bool chain_span(const SeqJob& j, int chain, int64_t& base, int& S) {
  if (!j.cu_seg) {
    base = (int64_t)chain * j.S;
    S = j.S;
    return true;
  }
  const int n = chain / j.heads, h = chain - n * j.heads;
  const int s0 = j.cu_seg[n], s1 = j.cu_seg[n + 1];
  // (the groups of a scan phase cover L * G segments per chain)
  if (s0 < 0 || s1 < s0 || s1 > j.T || (int64_t)(s1 - s0) > (int64_t)j.L * j.G) {
    if (j.status && threadIdx.x == 0) atomicOr(j.status, kStatusBadOffsets);
    return false;
  }
  base = (int64_t)h * j.T + s0;
  S = s1 - s0;
  return true;
}

// Grid: x = column tile, units along y and then z (job_grid), so a unit's
// tiles are adjacent in launch order and the unit count is not held to the
// 65535 limit of one grid dimension.  Returns false for the padding CTAs of
// the last z slab, which have no unit.
__device__ __forceinline__ bool unit_and_tile(const SeqJob& j, int& u, int& tile) {
  tile = (int)blockIdx.x;
  if (blockIdx.z == 0) {  // every unit of a grid with at most 65535 of them
    u = (int)blockIdx.y;
    return true;
  }
  const unsigned uu = blockIdx.z * gridDim.y + blockIdx.y;  // below 65535^2: no wrap
  u = (int)uu;
  return uu < (unsigned)(j.nchains * j.G);
}
#endif

// The grid of a job with `ntiles` column tiles per unit: (ntiles, units) while
// the units fit one dimension, else (ntiles, 65535, slabs).  x = 0 when the
// units exceed 2^31 - 1.
inline dim3 job_grid(const SeqJob& j, int ntiles) {
  const int64_t units = (int64_t)j.nchains * j.G;
  if (units < 1 || units > 0x7fffffff || ntiles < 1) return dim3(0, 1, 1);
  if (units <= 65535) return dim3((unsigned)ntiles, (unsigned)units, 1);
  return dim3((unsigned)ntiles, 65535u, (unsigned)((units + 65534) / 65535));
}

// Launches `kern` with the optional programmatic-serialization attribute.
template <class P>
cudaError_t launch_kernel(void (*kern)(P), dim3 grid, unsigned threads, size_t smem, cudaStream_t stream, bool pdl,
                          const P& params) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, params);
}

// seq_simt.cu: plain FFMA kernel, any K, V that are multiples of 32 up to 256.
cudaError_t launch_seq_simt(const SeqJob& job, cudaStream_t stream);

// seq_tc.cu: warp-specialised TMA/mbarrier pipeline with a tcgen05 3xTF32
// propagate.  K in {128, 256}, V a multiple of 32.  `release` selects the
// slot-release fence (QLA_RELEASE_*); `status` is the device status word a
// timed-out wait sets; `limit_ns` bounds every wait; `stall_test` makes the
// epilogue wait on a barrier nothing arrives on.
bool tc_supports(int K, int V);
cudaError_t launch_seq_tc(const SeqJob& job, int release, unsigned int* status, uint64_t limit_ns,
                          int stall_test, cudaStream_t stream);

// One launch of the per-segment local pass (local_simt.cu): for every chain
// and segment of L = T / S tokens, H = the segment's gated-delta-rule state
// from zero and M = the product of its token transitions.
struct LocalJob {
  const uint16_t* k;  // [nchains][T][K] bf16 bit patterns
  const uint16_t* v;  // [nchains][T][V] bf16 bit patterns
  const float* beta;  // [nchains][T]
  const float* g;     // [nchains][T] log-space decays
  float* H;           // [nchains][S][K][V] (kv) or [..][V][K] (vk), or nullptr
  float* M;           // [nchains][S][K][K], or nullptr
  int nchains, T, S, L, K, V, layout;
  int pdl;            // launch as a programmatic dependent of the stream's previous kernel
};
cudaError_t launch_local_simt(const LocalJob& job, cudaStream_t stream);
// The CTA count of a launch computing the H columns (with_h) and/or the M
// columns (with_m) of `job`'s units, and how many of its CTAs fit on one SM.
cudaError_t local_grid_info(const LocalJob& job, bool with_h, bool with_m, int64_t* ctas, int* per_sm);

// Bound on every device-side wait of the pipelined engines.
constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s

}  // namespace qla
