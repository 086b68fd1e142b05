// Host side of the C ABI declared in include/qla.h: argument checks, the
// per-device architecture check, variant/engine selection, the scan
// orchestration and the device status word.  No compute happens here: every
// step of the recurrence runs in the kernels of the other files.
#include <cuda_runtime.h>
#include <stdint.h>

#include <algorithm>
#include <atomic>
#include <cstdarg>
#include <cstdlib>
#include <cmath>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>

#include "qla.h"
#include "qla_internal.h"

namespace qla {

// Set by a kernel whose bounded wait gave up; read and cleared by
// qla_device_status().  Kernels receive its device address as a parameter.
__device__ unsigned int g_device_status;

namespace {

thread_local std::string t_last_error;

int fail(int status, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int status, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  t_last_error = buf;
  return status;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(QLA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool probed = false;
  bool is_sm103 = false;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  unsigned int* status_word = nullptr;
  // Side stream and fork/join events for the scan's two independent first
  // phases (null: the phases run one after the other on the caller's stream).
  cudaStream_t side = nullptr;
  cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
  std::mutex* side_mutex = nullptr;
};

std::mutex g_dev_mutex;
DeviceInfo g_dev[kMaxDevices];

// Probes the current device once: compute capability, SM count, status word.
int current_device(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(QLA_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_dev_mutex);
  DeviceInfo& d = g_dev[dev];
  if (!d.probed) {
    if ((e = cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(major)");
    if ((e = cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(minor)");
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return cuda_fail(e, "cudaDeviceGetAttribute(sm count)");
    d.is_sm103 = (d.cc_major == 10 && d.cc_minor == 3);
    if (d.is_sm103) {
      void* p = nullptr;
      if ((e = cudaGetSymbolAddress(&p, g_device_status)) != cudaSuccess)
        return cuda_fail(e, "cudaGetSymbolAddress(status word)");
      d.status_word = static_cast<unsigned int*>(p);
      // Created here, at the first call on the device, so that no scan call
      // (which may run inside a CUDA graph capture) has to create them.
      if (cudaStreamCreateWithFlags(&d.side, cudaStreamNonBlocking) != cudaSuccess ||
          cudaEventCreateWithFlags(&d.ev_fork, cudaEventDisableTiming) != cudaSuccess ||
          cudaEventCreateWithFlags(&d.ev_join, cudaEventDisableTiming) != cudaSuccess) {
        d.side = nullptr;
        cudaGetLastError();
      } else {
        d.side_mutex = new std::mutex;
      }
    }
    d.probed = true;
  }
  if (!d.is_sm103)
    return fail(QLA_ERR_ARCH, "device %d is sm_%d%d; this library is built for sm_103 (GB300) only", dev,
                d.cc_major, d.cc_minor);
  *out = &d;
  return QLA_OK;
}

struct Range {
  uintptr_t lo, hi;
  const char* name;
};

bool overlap(const Range& a, const Range& b) { return a.lo < b.hi && b.lo < a.hi; }

struct Shape {
  int B, heads, S, K, V, layout, direction;
  int64_t chains() const { return (int64_t)B * heads; }
  int64_t state() const { return (int64_t)K * V; }
};

int check_args(const float* H, const float* M, const float* h_init, const float* out, const float* fin,
               const Shape& s) {
  if (s.B < 1 || s.heads < 1 || s.S < 1 || s.K < 1 || s.V < 1)
    return fail(QLA_ERR_INVALID_ARG, "B, heads, S, K, V must be >= 1 (got %d, %d, %d, %d, %d)", s.B, s.heads, s.S,
                s.K, s.V);
  if (s.layout != QLA_LAYOUT_KV && s.layout != QLA_LAYOUT_VK)
    return fail(QLA_ERR_INVALID_ARG, "layout must be QLA_LAYOUT_KV or QLA_LAYOUT_VK (got %d)", s.layout);
  if (s.direction != QLA_FORWARD && s.direction != QLA_REVERSE)
    return fail(QLA_ERR_INVALID_ARG, "direction must be QLA_FORWARD or QLA_REVERSE (got %d)", s.direction);
  if (!H || !M) return fail(QLA_ERR_INVALID_ARG, "H and M must not be NULL");
  if (!out && !fin) return fail(QLA_ERR_INVALID_ARG, "out and final_state are both NULL: nothing to compute");
  if (s.K % 32 || s.K > 256 || s.V % 32 || s.V > 256)
    return fail(QLA_ERR_UNSUPPORTED, "K and V must be multiples of 32 in [32, 256] (got K=%d, V=%d)", s.K, s.V);
  const double elems = (double)s.chains() * s.S * s.K * std::max(s.K, s.V);
  if (elems >= 4.6e18) return fail(QLA_ERR_INVALID_ARG, "problem too large for 64-bit indexing");
  // one CTA per (chain, group, 32-column tile): a scan's G groups per chain are at most S
  if (s.chains() * s.S * ((s.V + 31) / 32) > 0x7fffffff)
    return fail(QLA_ERR_UNSUPPORTED, "B*heads*S*(V/32) must be below 2^31");
  const void* ptrs[] = {H, M, h_init, out, fin};
  const char* names[] = {"H", "M", "h_init", "out", "final_state"};
  for (int i = 0; i < 5; ++i)
    if (ptrs[i] && (reinterpret_cast<uintptr_t>(ptrs[i]) & 15))
      return fail(QLA_ERR_ALIGNMENT, "%s is not 16-byte aligned", names[i]);
  const uintptr_t sb = (uintptr_t)(s.chains() * s.S * s.state() * 4);
  Range r[5];
  int n = 0;
  r[n++] = {(uintptr_t)H, (uintptr_t)H + sb, "H"};
  r[n++] = {(uintptr_t)M, (uintptr_t)M + (uintptr_t)(s.chains() * s.S * s.K * s.K * 4), "M"};
  if (h_init) r[n++] = {(uintptr_t)h_init, (uintptr_t)h_init + (uintptr_t)(s.chains() * s.state() * 4), "h_init"};
  if (fin) r[n++] = {(uintptr_t)fin, (uintptr_t)fin + (uintptr_t)(s.chains() * s.state() * 4), "final_state"};
  if (out && out != H) r[n++] = {(uintptr_t)out, (uintptr_t)out + sb, "out"};
  for (int a = 0; a < n; ++a)
    for (int b = a + 1; b < n; ++b)
      if (overlap(r[a], r[b]))
        return fail(QLA_ERR_ALIAS, "%s and %s overlap (only out == H is allowed)", r[a].name, r[b].name);
  return QLA_OK;
}

// Host-side checks of a variable-length call (the offsets themselves live in
// device memory and are checked by the kernels).
int check_varlen_args(const float* H, const float* M, const float* h_init, const float* out, const float* fin,
                      const int* cu_seg, int N, int T, int heads, int K, int V, int layout, int direction) {
  if (N < 1 || T < 0 || heads < 1 || K < 1 || V < 1)
    return fail(QLA_ERR_INVALID_ARG, "N, heads, K, V must be >= 1 and T >= 0 (got %d, %d, %d, %d, %d)", N, heads, K,
                V, T);
  if (layout != QLA_LAYOUT_KV && layout != QLA_LAYOUT_VK)
    return fail(QLA_ERR_INVALID_ARG, "layout must be QLA_LAYOUT_KV or QLA_LAYOUT_VK (got %d)", layout);
  if (direction != QLA_FORWARD && direction != QLA_REVERSE)
    return fail(QLA_ERR_INVALID_ARG, "direction must be QLA_FORWARD or QLA_REVERSE (got %d)", direction);
  if (!H || !M || !cu_seg) return fail(QLA_ERR_INVALID_ARG, "H, M and cu_seg must not be NULL");
  if (!out && !fin) return fail(QLA_ERR_INVALID_ARG, "out and final_state are both NULL: nothing to compute");
  if (K % 32 || K > 256 || V % 32 || V > 256)
    return fail(QLA_ERR_UNSUPPORTED, "K and V must be multiples of 32 in [32, 256] (got K=%d, V=%d)", K, V);
  if ((int64_t)N * heads * (V / 32) > 0x7fffffff) return fail(QLA_ERR_UNSUPPORTED, "N*heads*(V/32) must be below 2^31");
  if ((int64_t)heads * T >= (int64_t)1 << 31) return fail(QLA_ERR_UNSUPPORTED, "heads*T must be below 2^31");
  const void* ptrs[] = {H, M, h_init, out, fin};
  const char* names[] = {"H", "M", "h_init", "out", "final_state"};
  for (int i = 0; i < 5; ++i)
    if (ptrs[i] && (reinterpret_cast<uintptr_t>(ptrs[i]) & 15))
      return fail(QLA_ERR_ALIGNMENT, "%s is not 16-byte aligned", names[i]);
  if (reinterpret_cast<uintptr_t>(cu_seg) & 3) return fail(QLA_ERR_ALIGNMENT, "cu_seg is not 4-byte aligned");
  const uintptr_t state = (uintptr_t)K * V * 4;
  const uintptr_t sb = (uintptr_t)heads * T * state;
  Range r[6];
  int n = 0;
  r[n++] = {(uintptr_t)H, (uintptr_t)H + sb, "H"};
  r[n++] = {(uintptr_t)M, (uintptr_t)M + (uintptr_t)heads * T * K * K * 4, "M"};
  r[n++] = {(uintptr_t)cu_seg, (uintptr_t)cu_seg + (uintptr_t)(N + 1) * 4, "cu_seg"};
  if (h_init) r[n++] = {(uintptr_t)h_init, (uintptr_t)h_init + (uintptr_t)N * heads * state, "h_init"};
  if (fin) r[n++] = {(uintptr_t)fin, (uintptr_t)fin + (uintptr_t)N * heads * state, "final_state"};
  if (out && out != H) r[n++] = {(uintptr_t)out, (uintptr_t)out + sb, "out"};
  for (int a = 0; a < n; ++a)
    for (int b = a + 1; b < n; ++b)
      if (overlap(r[a], r[b]))
        return fail(QLA_ERR_ALIAS, "%s and %s overlap (only out == H is allowed)", r[a].name, r[b].name);
  return QLA_OK;
}

// Cost models of the two variants on one-CTA-per-SM launches (each unit and
// 32-column tile is one CTA of the tensor-core kernel).  A phase that has more
// CTAs than SMs runs in waves, each costing its steps again.  The scan's model,
// in us, for G groups of L segments:
//     4.74 + 1.96 L w1 + 2.01 G w2 + 1.24 L w3,
// w = waves of phase 1 (products and offsets together, G (K + V) / 32 CTAs per
// chain), phase 2 (V / 32 per chain) and phase 3 (G V / 32 per chain).  The
// sequential kernel's is
//     4.7 + 1.62 (S - 1) w.
// Both are least-squares fits to calls timed on GB300 at K = V = 128: the scan
// at 1, 2 and 4 heads, S = 32 .. 128 and every G from 4 to 32; the sequential
// kernel over S = 2 .. 128.  Within 10 % of the measured time at 1 to 32 heads.
double waves_of(int64_t ctas, int sms) { return (double)((ctas + sms - 1) / sms); }

double scan_model_us(int S, int G, int64_t chains, int K, int V, int sms) {
  const int L = (S + G - 1) / G;
  const int Gr = (S + L - 1) / L;
  return 4.74 + 1.96 * L * waves_of(chains * Gr * ((K + V) / 32), sms) + 2.01 * Gr * waves_of(chains * (V / 32), sms) +
         1.24 * L * waves_of(chains * Gr * (V / 32), sms);
}

double seq_model_us(int S, int64_t chains, int V, int sms) {
  return 4.7 + 1.62 * (S - 1) * waves_of(chains * ((V + 31) / 32), sms);
}

// Scan group count for S segments of `chains` chains.  The critical path is
// about 2L + G steps with G*L >= S, smallest near G = sqrt(2S); with more
// chains the phases with G units per chain run in several waves, so fewer
// groups can be faster.  Among the group counts up to sqrt(2S) (never more
// scratch than that choice), the one the scan's model rates fastest; it picks
// the fastest measured G at each of the points it was fitted on.  Without the
// SM count (sms <= 0), the step-count balance alone.
int auto_groups(int S, int64_t chains, int K, int V, int sms) {
  const int G0 = std::max(1, (int)std::lround(std::sqrt(2.0 * S)));
  if (sms <= 0 || chains <= 0) {
    const int L = (S + G0 - 1) / G0;
    return (S + L - 1) / L;
  }
  int best = 1;
  double best_cost = 0.0;
  for (int G = 1; G <= std::min(G0, S); ++G) {
    const int L = (S + G - 1) / G;
    if ((S + L - 1) / L != G) continue;  // the same (L, Gr) as a smaller G
    const double cost = scan_model_us(S, G, chains, K, V, sms);
    if (G == 1 || cost < best_cost) {
      best = G;
      best_cost = cost;
    }
  }
  return best;
}

bool known_engine(int engine) {
  return engine == QLA_ENGINE_AUTO || engine == QLA_ENGINE_SIMT || engine == QLA_ENGINE_TC;
}

// Longest chain the automatic choice gives to the tensor-core engine.  The
// tensor core accumulates in fp32 rounding toward zero; with norm-preserving
// M the states shrink coherently by about 4.4e-8 per step at K = 128 (four
// accumulations per chain and step) and 1.4e-7 at K = 256 (sixteen), so the
// worst per-state relative L2 error reaches 1e-5 near 200 and 64 steps
// (measured on GB300: 8.0e-6 at S = 160, K = 128; 7.8e-6 at S = 48, K = 256).
// Longer chains go to the FFMA engine, which rounds to nearest (3.3e-6 at
// S = 512).  The scan regroups the same products and drifts the same way, so
// the limit applies to the whole chain there too.
int tc_auto_max_segments(int K) { return K <= 128 ? 160 : 48; }

int resolve_engine(const Shape& s, int engine) {
  if (engine == QLA_ENGINE_AUTO)
    return (tc_supports(s.K, s.V) && s.S <= tc_auto_max_segments(s.K)) ? QLA_ENGINE_TC : QLA_ENGINE_SIMT;
  return engine;
}

// The engine a scan phase runs on: phase 1a's V' = K may differ from V.
int engine_for(const SeqJob& j, int engine) {
  if (engine == QLA_ENGINE_TC && !tc_supports(j.K, j.V)) return QLA_ENGINE_SIMT;
  return engine;
}

// The scan trades a sequential chain of S-1 steps for about 2L + G steps in
// three launches whose parallel phases hold tiles * G CTAs.  Measured on
// GB300 (K = V = 128, tensor-core engine): it wins for S >= 32 with up to
// 16 column tiles (1.25x - 2.9x) and loses for S <= 8 or 128 tiles.
// Process-wide override of the automatic variant choice (qla_set_variant);
// -1 until first read, then initialised from the QLA_VARIANT environment
// variable ("auto", "seq", "scan" or 0, 1, 2; anything else means auto).
std::atomic<int> g_variant_override{-1};

int parse_variant_env(const char* v) {
  if (!v) return QLA_VARIANT_AUTO;
  if (!strcmp(v, "seq") || !strcmp(v, "1")) return QLA_VARIANT_SEQ;
  if (!strcmp(v, "scan") || !strcmp(v, "2")) return QLA_VARIANT_SCAN;
  return QLA_VARIANT_AUTO;
}

int variant_override() {
  int v = g_variant_override.load(std::memory_order_relaxed);
  if (v < 0) {
    int expected = -1;
    g_variant_override.compare_exchange_strong(expected, parse_variant_env(std::getenv("QLA_VARIANT")));
    v = g_variant_override.load(std::memory_order_relaxed);
  }
  return v;
}

// Process-wide choice of programmatic dependent launch for the sequential
// variant's launch (-1: not read yet; initial value from QLA_PDL).
std::atomic<int> g_dependent_launch{-1};

int dependent_launch() {
  int v = g_dependent_launch.load(std::memory_order_relaxed);
  if (v < 0) {
    const char* e = std::getenv("QLA_PDL");
    int expected = -1;
    g_dependent_launch.compare_exchange_strong(expected, (e && (!strcmp(e, "1") || !strcmp(e, "on"))) ? 1 : 0);
    v = g_dependent_launch.load(std::memory_order_relaxed);
  }
  return v;
}

// The sequential variant's single launch, as a programmatic dependent of the
// stream's previous kernel when the process-wide switch is on.
SeqJob dependent(SeqJob j) {
  j.pdl = dependent_launch();
  return j;
}

// Automatic variant: the scan where its model (with its automatic group
// count) is below 0.95 of the sequential kernel's, else the sequential kernel.
// The margin covers the scan's extra launches where the two are close.
int resolve_variant(const Shape& s, int variant, const DeviceInfo* d) {
  if (variant != QLA_VARIANT_AUTO) return variant;
  const int forced = variant_override();
  if (forced != QLA_VARIANT_AUTO) return forced;
  if (s.S < 2 || d->sm_count < 1) return QLA_VARIANT_SEQ;
  const int64_t chains = s.chains();
  const int G = auto_groups(s.S, chains, s.K, s.V, d->sm_count);
  const double scan = scan_model_us(s.S, G, chains, s.K, s.V, d->sm_count);
  return scan < 0.95 * seq_model_us(s.S, chains, s.V, d->sm_count) ? QLA_VARIANT_SCAN : QLA_VARIANT_SEQ;
}

int launch_seq(const SeqJob& job, int engine, int release, const DeviceInfo* d, cudaStream_t stream) {
  SeqJob j = job;
  j.status = d->status_word;
  cudaError_t e;
  switch (engine) {
    case QLA_ENGINE_SIMT:
      e = launch_seq_simt(j, stream);
      break;
    case QLA_ENGINE_TC:
      if (!tc_supports(j.K, j.V))
        return fail(QLA_ERR_UNSUPPORTED, "the tensor-core engine takes K in {128, 256} (got K=%d, V=%d)", j.K, j.V);
      e = launch_seq_tc(j, release, d->status_word, kWaitLimitNs, 0, stream);
      break;
    default:
      return fail(QLA_ERR_UNSUPPORTED, "engine %d is not compiled into this library", engine);
  }
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return QLA_OK;
}

SeqJob plain_job(const float* H, const float* M, const float* h_init, float* out, float* fin, const Shape& s) {
  SeqJob j{};
  j.H = H;
  j.M = M;
  j.init = h_init;
  j.out = out;
  j.fin = fin;
  j.h_chain_stride = (int64_t)s.S * s.state();
  j.m_chain_stride = (int64_t)s.S * s.K * s.K;
  j.init_unit_stride = s.state();
  j.fin_unit_stride = s.state();
  j.nchains = (int)s.chains();
  j.S = s.S;
  j.L = s.S;
  j.G = 1;
  j.K = s.K;
  j.V = s.V;
  j.layout = s.layout;
  j.direction = s.direction;
  j.init_mode = h_init ? kInitPointer : kInitZero;
  return j;
}

size_t scan_bytes(const Shape& s, int G) {
  // A_agg [chains][G][K][K], b_agg and carries [chains][G][state]
  return (size_t)s.chains() * G * ((size_t)s.K * s.K + 2 * (size_t)s.state()) * sizeof(float);
}

// Runs `on_main` on `stream` and `on_side` on the device's side stream
// concurrently: the side stream waits for everything issued to `stream`
// before the call, and `stream` waits for the side stream's work before
// anything issued after the call (event fork and join, which CUDA graph
// capture follows).  The side stream and its events are shared by the
// device's callers, so the fork, the side launch and the join are issued
// under a lock.  Without a side stream both run on `stream`.  (When the two
// launches' CTAs exceed the SMs, running them concurrently measured neither
// faster nor slower than one after the other.)
template <class MainFn, class SideFn>
int fork_join(const DeviceInfo* d, cudaStream_t stream, MainFn&& on_main, SideFn&& on_side) {
  if (!d->side) {
    const int st = on_side(stream);
    return st != QLA_OK ? st : on_main(stream);
  }
  std::lock_guard<std::mutex> lock(*d->side_mutex);
  cudaError_t e = cudaEventRecord(d->ev_fork, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaEventRecord(fork)");
  if ((e = cudaStreamWaitEvent(d->side, d->ev_fork, 0)) != cudaSuccess) return cuda_fail(e, "cudaStreamWaitEvent(fork)");
  const int st_side = on_side(d->side);
  // join even after a failed side launch, so that a capturing stream is not left forked
  const cudaError_t e_rec = cudaEventRecord(d->ev_join, d->side);
  const int st_main = st_side == QLA_OK ? on_main(stream) : st_side;
  const cudaError_t e_wait = e_rec == cudaSuccess ? cudaStreamWaitEvent(stream, d->ev_join, 0) : e_rec;
  if (st_main != QLA_OK) return st_main;
  if (e_wait != cudaSuccess) return cuda_fail(e_wait, "event join");
  return QLA_OK;
}

// The scan variant.  For groups g of L consecutive segments (by index):
//  1a. A_g = M_{last} ... M_{first} over the group's segments (forward products
//      from the identity, kv view, V' = K); in reverse this is the transpose of
//      the group's reverse aggregate.
//  1b. b_g = the group's recurrence from a zero state, in the caller's layout
//      and direction (its final state).
//  2.  The same recurrence over the G aggregates, (M', H') = (A_g, b_g), from
//      h_init: its exclusive outputs are the states entering each group.
//  3.  Every group re-run from its entering state, writing out.
// `base` is the job of the whole call (fixed length, or variable length with
// offsets: then phases 1a, 1b and 3 locate each (chain, group) through them,
// and a group past its sequence's end is empty, with the identity and zero
// as aggregates, which phase 2 steps through unchanged in either direction).
// `ws` holds A_agg [chains][Gr][K][K], then b_agg and carries
// [chains][Gr][state] (scan_bytes).
int scan_phases(const SeqJob& base, const Shape& s, int L, int Gr, float* ws, int engine, int release,
                const DeviceInfo* d, cudaStream_t stream) {
  const int64_t chains = base.nchains;
  float* Aagg = ws;
  float* bagg = Aagg + (size_t)chains * Gr * s.K * s.K;
  float* carry = bagg + (size_t)chains * Gr * s.state();
  // 1a and 1b are independent: they run concurrently.
  SeqJob j1a = base;
  j1a.H = nullptr;
  j1a.init = nullptr;
  j1a.init_mode = kInitIdentity;
  j1a.out = nullptr;
  j1a.fin = Aagg;
  j1a.fin_unit_stride = (int64_t)s.K * s.K;
  j1a.L = L;
  j1a.G = Gr;
  j1a.V = s.K;
  j1a.layout = QLA_LAYOUT_KV;
  j1a.direction = QLA_FORWARD;
  SeqJob j1b = base;
  j1b.init = nullptr;
  j1b.init_mode = kInitZero;
  j1b.out = nullptr;
  j1b.fin = bagg;
  j1b.fin_unit_stride = s.state();
  j1b.L = L;
  j1b.G = Gr;
  int st = fork_join(
      d, stream, [&](cudaStream_t cs) { return launch_seq(j1a, engine_for(j1a, engine), release, d, cs); },
      [&](cudaStream_t cs) { return launch_seq(j1b, engine_for(j1b, engine), release, d, cs); });
  if (st != QLA_OK) return st;
  {  // 2: carries across the group aggregates (fixed length Gr per chain)
    SeqJob j = base;
    j.cu_seg = nullptr;
    j.H = bagg;
    j.M = Aagg;
    j.h_chain_stride = (int64_t)Gr * s.state();
    j.m_chain_stride = (int64_t)Gr * s.K * s.K;
    j.out = carry;
    j.S = Gr;
    j.L = Gr;
    j.G = 1;
    j.nstates = chains * Gr;
    if ((st = launch_seq(j, engine_for(j, engine), release, d, stream)) != QLA_OK) return st;
  }
  if (base.out) {  // 3: re-run each group from its entering state
    SeqJob j = base;
    j.init = carry;
    j.init_mode = kInitPointer;
    j.init_unit_stride = s.state();
    j.fin = nullptr;
    j.L = L;
    j.G = Gr;
    if ((st = launch_seq(j, engine_for(j, engine), release, d, stream)) != QLA_OK) return st;
  }
  return QLA_OK;
}

// Group length L and the number of groups actually formed for S segments of
// `chains` chains and a requested group count (0: automatic, for a device
// with `sms` SMs).
void scan_groups_for(int S, int group, int64_t chains, int K, int V, int sms, int* L, int* Gr) {
  const int G = group > 0 ? std::min(group, S) : auto_groups(S, chains, K, V, sms);
  *L = (S + G - 1) / G;
  *Gr = (S + *L - 1) / *L;
}

// The scan with its workspace from the stream-ordered allocator.
int run_scan_alloc(const SeqJob& base, const Shape& s, int engine, int release, int group, const DeviceInfo* d,
                   cudaStream_t stream) {
  int L, Gr;
  scan_groups_for(s.S, group, base.nchains, s.K, s.V, d->sm_count, &L, &Gr);
  const size_t bytes = (size_t)base.nchains * Gr * ((size_t)s.K * s.K + 2 * (size_t)s.state()) * sizeof(float);
  float* ws = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&ws), bytes, stream);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMallocAsync(scan workspace)");
  const int st = scan_phases(base, s, L, Gr, ws, engine, release, d, stream);
  e = cudaFreeAsync(ws, stream);
  if (st == QLA_OK && e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(scan workspace)");
  return st;
}

int run_scan(const float* H, const float* M, const float* h_init, float* out, float* fin, const Shape& s,
             int engine, int release, int group, const DeviceInfo* d, cudaStream_t stream) {
  return run_scan_alloc(plain_job(H, M, h_init, out, fin, s), s, engine, release, group, d, stream);
}

// ---------------------------------------------------------------- local pass split
//
// A local pass's CTAs all run the same number of tokens, so when they exceed
// what the SMs hold at once the last partial wave costs a whole segment's
// time on a few SMs.  Splitting each segment into F sub-segments makes the
// units F times shorter (more, shorter waves); the F sub-segments' maps are
// then composed per segment by the correction kernels: M_seg = the product of
// the sub-segment M's (from the identity) and H_seg = their recurrence from
// zero, exactly the scan's first phase with groups of F.

// Relative cost of one composition step per wave of its CTAs, in tokens of a
// local-pass wave (both measured on GB300 at K = V = 128: a correction step
// ~1.6 us, a local-pass token per wave ~0.5 us; rounded up for set-up).
constexpr double kComposeStepTokens = 4.0;

int local_auto_split(const LocalJob& j, const DeviceInfo* d, int* F) {
  *F = 1;
  if (d->sm_count < 1) return QLA_OK;
  double best = 0.0;
  for (int f = 1; f <= 16; f *= 2) {
    if (j.L % f || j.L / f < 64 || (int64_t)j.nchains * j.S * f > 0x7fffffff) break;
    LocalJob t = j;
    t.S = j.S * f;
    t.L = j.L / f;
    // the split always computes the sub-segments' M (H only if H is wanted)
    int64_t ctas = 0;
    int per_sm = 0;
    const cudaError_t e = local_grid_info(t, t.H != nullptr, f > 1 || t.M != nullptr, &ctas, &per_sm);
    if (e != cudaSuccess) return cuda_fail(e, "occupancy query");
    if (per_sm < 1) per_sm = 1;
    const int64_t slots = (int64_t)per_sm * d->sm_count;
    const double waves = (double)((ctas + slots - 1) / slots);
    double cost = waves * t.L;
    if (f > 1) {  // composition: f steps over (H, M) column tiles, one CTA per SM
      const int64_t ccta = j.nchains * (int64_t)j.S * ((j.V + j.K + 31) / 32);
      cost += f * kComposeStepTokens * (double)((ccta + d->sm_count - 1) / d->sm_count);
    }
    if (f == 1 || cost < best) {
      best = cost;
      *F = f;
    }
  }
  return QLA_OK;
}

// `no_scratch` (optional) is set when the sub-segments' scratch could not be
// allocated; nothing was launched then.
int local_pass_split(const LocalJob& j, int F, const DeviceInfo* d, cudaStream_t stream, bool* no_scratch) {
  const int64_t units = (int64_t)j.nchains * j.S * F;  // sub-segments
  const size_t hbytes = (size_t)units * j.K * j.V * sizeof(float);
  const size_t mbytes = (size_t)units * j.K * j.K * sizeof(float);
  const bool need_h = j.H != nullptr;
  float* ws = nullptr;
  cudaError_t e = cudaMallocAsync(reinterpret_cast<void**>(&ws), (need_h ? hbytes : 0) + mbytes, stream);
  if (e != cudaSuccess) {
    if (no_scratch) *no_scratch = true;
    return cuda_fail(e, "cudaMallocAsync(local pass sub-segments)");
  }
  float* Ms = ws;
  float* Hs = need_h ? ws + (size_t)units * j.K * j.K : nullptr;
  LocalJob t = j;
  t.S = j.S * F;
  t.L = j.L / F;
  t.H = Hs;
  t.M = Ms;
  int st = QLA_OK;
  e = launch_local_simt(t, stream);
  if (e != cudaSuccess) st = cuda_fail(e, "kernel launch");
  if (st == QLA_OK) {
    // segment s of chain c = group s of F sub-segments: 1a the product of the
    // M's from the identity, 1b the recurrence over (H, M) from zero
    SeqJob base{};
    base.M = Ms;
    base.m_chain_stride = (int64_t)t.S * j.K * j.K;
    base.h_chain_stride = (int64_t)t.S * j.K * j.V;
    base.nchains = j.nchains;
    base.S = t.S;
    base.L = F;
    base.G = j.S;
    base.K = j.K;
    base.direction = QLA_FORWARD;
    SeqJob ja = base;
    ja.H = nullptr;
    ja.init_mode = kInitIdentity;
    ja.fin = j.M;
    ja.fin_unit_stride = (int64_t)j.K * j.K;
    ja.V = j.K;
    ja.layout = QLA_LAYOUT_KV;
    SeqJob jb = base;
    jb.H = Hs;
    jb.init_mode = kInitZero;
    jb.fin = j.H;
    jb.fin_unit_stride = (int64_t)j.K * j.V;
    jb.V = j.V;
    jb.layout = j.layout;
    auto run = [&](const SeqJob& jj, cudaStream_t s) {
      return launch_seq(jj, engine_for(jj, QLA_ENGINE_TC), QLA_RELEASE_MEMBAR, d, s);
    };
    if (j.M && j.H)
      st = fork_join(d, stream, [&](cudaStream_t s) { return run(ja, s); }, [&](cudaStream_t s) { return run(jb, s); });
    else if (j.M)
      st = run(ja, stream);
    else
      st = run(jb, stream);
  }
  e = cudaFreeAsync(ws, stream);
  if (st == QLA_OK && e != cudaSuccess) return cuda_fail(e, "cudaFreeAsync(local pass sub-segments)");
  return st;
}

// ---------------------------------------------------------------- allocation-free scan
//
// Scratch of qla_cp_correct_scan_static(): a fixed array of this file, one
// per device that loads the library.  Host code must not use the symbol as
// an address; it looks up each device's address once, with that device
// current, and passes the result to the kernels.
static __device__ __align__(256) float g_scan_static[QLA_SCAN_STATIC_BYTES / sizeof(float)];

std::mutex g_static_mutex;
float* g_static_ptr[kMaxDevices];

int scan_static_pointer(float** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(QLA_ERR_CUDA, "device ordinal %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_static_mutex);
  if (!g_static_ptr[dev]) {
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, g_scan_static)) != cudaSuccess)
      return cuda_fail(e, "cudaGetSymbolAddress(scan scratch)");
    g_static_ptr[dev] = static_cast<float*>(p);
  }
  *out = g_static_ptr[dev];
  return QLA_OK;
}

// The scan phases on a caller-provided workspace (`group` groups requested,
// 0 = automatic, as for the workspace size).
int run_scan_in(const float* H, const float* M, const float* h_init, float* out, float* fin, const Shape& s,
                int engine, int release, int group, float* ws, const DeviceInfo* d, cudaStream_t stream) {
  int L, Gr;
  scan_groups_for(s.S, group, (int64_t)s.B * s.heads, s.K, s.V, d->sm_count, &L, &Gr);
  return scan_phases(plain_job(H, M, h_init, out, fin, s), s, L, Gr, ws, engine, release, d, stream);
}

// The scan variant for variable-length calls: every chain gets the groups
// that the caller's bound s.S on any sequence's length needs (scan_phases).
int run_scan_varlen(const SeqJob& vj, const Shape& s, int engine, int group, const DeviceInfo* d,
                    cudaStream_t stream) {
  return run_scan_alloc(vj, s, engine, QLA_RELEASE_MEMBAR, group, d, stream);
}

}  // namespace
}  // namespace qla

using namespace qla;

// Test producer for programmatic dependent launch: every CTA lets its
// dependents start at once, then holds its copy back for `delay_ns`, so a
// dependent that touched the copied bytes before its griddepcontrol.wait
// would see their previous contents.  The delay is a bounded sleep on the
// global timer.
__global__ void dependent_producer_kernel(const float4* __restrict__ src, float4* __restrict__ dst, size_t n,
                                          uint64_t delay_ns) {
  griddep_launch_dependents();
  uint64_t t0, t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  do {
    __nanosleep(1000);
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  } while (t - t0 < delay_ns);
  for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x)
    dst[i] = src[i];
}

extern "C" {

int qla_version(void) { return 100; }

int qla_cp_correct_scan_static(const float* H, const float* M, const float* h_init, float* out, float* final_state,
                               int B, int heads, int S, int K, int V, int layout, int direction, int engine,
                               int release, int scan_group, void* stream) {
  t_last_error.clear();
  Shape s{B, heads, S, K, V, layout, direction};
  int st = check_args(H, M, h_init, out, final_state, s);
  if (st != QLA_OK) return st;
  if (!known_engine(engine)) return fail(QLA_ERR_INVALID_ARG, "unknown engine %d", engine);
  if (release < QLA_RELEASE_MEMBAR || release > QLA_RELEASE_NONE)
    return fail(QLA_ERR_INVALID_ARG, "unknown release mode %d", release);
  if (scan_group < 0) return fail(QLA_ERR_INVALID_ARG, "scan_group must be >= 0");
  DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != QLA_OK) return st;
  int L, Gr;
  scan_groups_for(S, scan_group, (int64_t)B * heads, K, V, d->sm_count, &L, &Gr);
  const size_t need = scan_bytes(s, Gr);
  if (need > QLA_SCAN_STATIC_BYTES)
    return fail(QLA_ERR_UNSUPPORTED,
                "this shape needs %zu bytes of scan scratch; the allocation-free scan holds %u bytes "
                "(use qla_cp_correct_ex with QLA_VARIANT_SCAN instead)",
                need, (unsigned)QLA_SCAN_STATIC_BYTES);
  float* ws = nullptr;
  if ((st = scan_static_pointer(&ws)) != QLA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  const int eng = resolve_engine(s, engine);
  if (S == 1) return launch_seq(dependent(plain_job(H, M, h_init, out, final_state, s)), eng, release, d, cs);
  return run_scan_in(H, M, h_init, out, final_state, s, eng, release, scan_group, ws, d, cs);
}

const char* qla_status_string(int status) {
  switch (status) {
    case QLA_OK: return "QLA_OK";
    case QLA_ERR_INVALID_ARG: return "QLA_ERR_INVALID_ARG: invalid argument";
    case QLA_ERR_UNSUPPORTED: return "QLA_ERR_UNSUPPORTED: unsupported shape or option";
    case QLA_ERR_ALIGNMENT: return "QLA_ERR_ALIGNMENT: pointer not 16-byte aligned";
    case QLA_ERR_ALIAS: return "QLA_ERR_ALIAS: overlapping buffers";
    case QLA_ERR_CUDA: return "QLA_ERR_CUDA: CUDA runtime error";
    case QLA_ERR_ARCH: return "QLA_ERR_ARCH: device is not sm_103";
    case QLA_ERR_TIMEOUT: return "QLA_ERR_TIMEOUT: a bounded device wait gave up";
    default: return "unknown status";
  }
}

const char* qla_last_error(void) { return t_last_error.c_str(); }

size_t qla_scan_workspace_bytes(int B, int heads, int S, int K, int V, int scan_group) {
  if (B < 1 || heads < 1 || S < 1 || K < 1 || V < 1) return 0;
  Shape s{B, heads, S, K, V, 0, 0};
  // the automatic group count depends on the current device's SM count;
  // without a usable device, the step-count rule (never fewer groups, so
  // never less scratch)
  int sms = 0;
  DeviceInfo* d = nullptr;
  if (current_device(&d) == QLA_OK) sms = d->sm_count;
  t_last_error.clear();
  int L, Gr;
  scan_groups_for(S, scan_group, (int64_t)B * heads, K, V, sms, &L, &Gr);
  return scan_bytes(s, Gr);
}

int qla_set_variant(int variant) {
  t_last_error.clear();
  if (variant != QLA_VARIANT_AUTO && variant != QLA_VARIANT_SEQ && variant != QLA_VARIANT_SCAN)
    return fail(QLA_ERR_INVALID_ARG, "unknown variant %d", variant);
  g_variant_override.store(variant, std::memory_order_relaxed);
  return QLA_OK;
}

int qla_set_dependent_launch(int enable) {
  t_last_error.clear();
  if (enable != 0 && enable != 1) return fail(QLA_ERR_INVALID_ARG, "enable must be 0 or 1 (got %d)", enable);
  g_dependent_launch.store(enable, std::memory_order_relaxed);
  return QLA_OK;
}

int qla_resolve(int B, int heads, int S, int K, int V, int layout, int* variant, int* engine) {
  t_last_error.clear();
  DeviceInfo* d = nullptr;
  int st = current_device(&d);
  if (st != QLA_OK) return st;
  Shape s{B, heads, S, K, V, layout, 0};
  if (variant) *variant = resolve_variant(s, QLA_VARIANT_AUTO, d);
  if (engine) *engine = resolve_engine(s, QLA_ENGINE_AUTO);
  return QLA_OK;
}

int qla_cp_correct_ex(const float* H, const float* M, const float* h_init, float* out, float* final_state, int B,
                      int heads, int S, int K, int V, int layout, int direction, int variant, int engine,
                      int release, int scan_group, void* stream) {
  t_last_error.clear();
  Shape s{B, heads, S, K, V, layout, direction};
  int st = check_args(H, M, h_init, out, final_state, s);
  if (st != QLA_OK) return st;
  if (variant < QLA_VARIANT_AUTO || variant > QLA_VARIANT_SCAN)
    return fail(QLA_ERR_INVALID_ARG, "unknown variant %d", variant);
  if (!known_engine(engine)) return fail(QLA_ERR_INVALID_ARG, "unknown engine %d", engine);
  if (release < QLA_RELEASE_MEMBAR || release > QLA_RELEASE_NONE)
    return fail(QLA_ERR_INVALID_ARG, "unknown release mode %d", release);
  if (scan_group < 0) return fail(QLA_ERR_INVALID_ARG, "scan_group must be >= 0");
  DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != QLA_OK) return st;
  const int v = resolve_variant(s, variant, d);
  const int eng = resolve_engine(s, engine);
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  if (v == QLA_VARIANT_SCAN && S > 1)
    return run_scan(H, M, h_init, out, final_state, s, eng, release, scan_group, d, cs);
  return launch_seq(dependent(plain_job(H, M, h_init, out, final_state, s)), eng, release, d, cs);
}

int qla_cp_correct(const float* H, const float* M, const float* h_init, float* out, int B, int heads, int S, int K,
                   int V, int layout, int direction, void* stream) {
  return qla_cp_correct_ex(H, M, h_init, out, nullptr, B, heads, S, K, V, layout, direction, QLA_VARIANT_AUTO,
                           QLA_ENGINE_AUTO, QLA_RELEASE_MEMBAR, 0, stream);
}

int qla_cp_correct_varlen(const float* H, const float* M, const float* h_init, float* out, float* final_state,
                          const int* cu_seg, int N, int T, int heads, int K, int V, int layout, int direction,
                          int engine, void* stream) {
  return qla_cp_correct_varlen_ex(H, M, h_init, out, final_state, cu_seg, N, T, heads, K, V, layout, direction,
                                  QLA_VARIANT_SEQ, engine, 0, 0, stream);
}

int qla_cp_correct_varlen_ex(const float* H, const float* M, const float* h_init, float* out, float* final_state,
                             const int* cu_seg, int N, int T, int heads, int K, int V, int layout, int direction,
                             int variant, int engine, int max_segments, int scan_group, void* stream) {
  t_last_error.clear();
  int st = check_varlen_args(H, M, h_init, out, final_state, cu_seg, N, T, heads, K, V, layout, direction);
  if (st != QLA_OK) return st;
  if (!known_engine(engine)) return fail(QLA_ERR_INVALID_ARG, "unknown engine %d", engine);
  if (variant != QLA_VARIANT_AUTO && variant != QLA_VARIANT_SEQ && variant != QLA_VARIANT_SCAN)
    return fail(QLA_ERR_INVALID_ARG, "unknown variant %d", variant);
  if (max_segments < 0 || max_segments > T)
    return fail(QLA_ERR_INVALID_ARG, "max_segments must be in [0, T] (got %d, T=%d)", max_segments, T);
  if (scan_group < 0) return fail(QLA_ERR_INVALID_ARG, "scan_group must be >= 0 (got %d)", scan_group);
  DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != QLA_OK) return st;
  const int Smax = max_segments > 0 ? max_segments : T;
  Shape s{N, heads, std::max(1, Smax), K, V, layout, direction};
  const int eng = resolve_engine(s, engine);
  const int var = variant == QLA_VARIANT_AUTO ? resolve_variant(s, QLA_VARIANT_AUTO, d) : variant;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  SeqJob j{};
  j.H = H;
  j.M = M;
  j.init = h_init;
  j.out = out;
  j.fin = final_state;
  j.init_unit_stride = (int64_t)K * V;
  j.fin_unit_stride = (int64_t)K * V;
  j.nchains = N * heads;
  j.S = 0;
  j.L = 1 << 30;
  j.G = 1;
  j.K = K;
  j.V = V;
  j.layout = layout;
  j.direction = direction;
  j.init_mode = h_init ? kInitPointer : kInitZero;
  j.cu_seg = cu_seg;
  j.heads = heads;
  j.T = T;
  j.nstates = (int64_t)heads * T;
  if (var == QLA_VARIANT_SEQ || Smax < 2) return launch_seq(dependent(j), eng, QLA_RELEASE_MEMBAR, d, cs);
  int L, Gr;
  scan_groups_for(s.S, scan_group, (int64_t)N * heads, K, V, d->sm_count, &L, &Gr);
  if ((int64_t)N * heads * Gr * (V / 32) > 0x7fffffff)
    return fail(QLA_ERR_UNSUPPORTED, "N*heads*G*(V/32) must be below 2^31 for the scan variant");
  return run_scan_varlen(j, s, eng, scan_group, d, cs);
}

int qla_local_pass(const void* k, const void* v, const float* beta, const float* g, float* H, float* M, int B,
                   int heads, int T, int S, int K, int V, int layout, void* stream) {
  return qla_local_pass_ex(k, v, beta, g, H, M, B, heads, T, S, K, V, layout, 0, stream);
}

int qla_local_pass_ex(const void* k, const void* v, const float* beta, const float* g, float* H, float* M, int B,
                      int heads, int T, int S, int K, int V, int layout, int split, void* stream) {
  t_last_error.clear();
  if (B < 1 || heads < 1 || S < 1 || T < 1 || K < 1 || V < 1)
    return fail(QLA_ERR_INVALID_ARG, "B, heads, T, S, K, V must be >= 1 (got %d, %d, %d, %d, %d, %d)", B, heads, T,
                S, K, V);
  if (T % S) return fail(QLA_ERR_INVALID_ARG, "T (%d) must be a multiple of S (%d)", T, S);
  if (layout != QLA_LAYOUT_KV && layout != QLA_LAYOUT_VK)
    return fail(QLA_ERR_INVALID_ARG, "layout must be QLA_LAYOUT_KV or QLA_LAYOUT_VK (got %d)", layout);
  if (!k || !v || !beta || !g) return fail(QLA_ERR_INVALID_ARG, "k, v, beta and g must not be NULL");
  if (!H && !M) return fail(QLA_ERR_INVALID_ARG, "H and M are both NULL: nothing to compute");
  if (K % 32 || K > 256 || V % 32 || V > 256)
    return fail(QLA_ERR_UNSUPPORTED, "K and V must be multiples of 32 in [32, 256] (got K=%d, V=%d)", K, V);
  const int L = T / S;
  if (split < 0 || (split > 0 && L % split))
    return fail(QLA_ERR_INVALID_ARG, "split must be 0 (automatic) or divide the segment length %d (got %d)", L, split);
  const int64_t chains = (int64_t)B * heads;
  if (chains * S * (split > 0 ? split : 1) > 0x7fffffff)
    return fail(QLA_ERR_UNSUPPORTED, "B*heads*S*split must be below 2^31");
  if ((double)chains * T * std::max(K, V) >= 4.6e18) return fail(QLA_ERR_INVALID_ARG, "problem too large");
  const void* p16[] = {k, v, H, M};
  const char* n16[] = {"k", "v", "H", "M"};
  for (int i = 0; i < 4; ++i)
    if (p16[i] && (reinterpret_cast<uintptr_t>(p16[i]) & 15))
      return fail(QLA_ERR_ALIGNMENT, "%s is not 16-byte aligned", n16[i]);
  if ((reinterpret_cast<uintptr_t>(beta) | reinterpret_cast<uintptr_t>(g)) & 3)
    return fail(QLA_ERR_ALIGNMENT, "beta and g must be 4-byte aligned");
  Range r[6];
  int n = 0;
  r[n++] = {(uintptr_t)k, (uintptr_t)k + (uintptr_t)(chains * T * K * 2), "k"};
  r[n++] = {(uintptr_t)v, (uintptr_t)v + (uintptr_t)(chains * T * V * 2), "v"};
  r[n++] = {(uintptr_t)beta, (uintptr_t)beta + (uintptr_t)(chains * T * 4), "beta"};
  r[n++] = {(uintptr_t)g, (uintptr_t)g + (uintptr_t)(chains * T * 4), "g"};
  if (H) r[n++] = {(uintptr_t)H, (uintptr_t)H + (uintptr_t)(chains * S * K * V * 4), "H"};
  if (M) r[n++] = {(uintptr_t)M, (uintptr_t)M + (uintptr_t)(chains * S * K * K * 4), "M"};
  for (int a = 4; a < n; ++a)  // outputs against everything before them
    for (int b = 0; b < a; ++b)
      if (overlap(r[a], r[b])) return fail(QLA_ERR_ALIAS, "%s and %s overlap", r[a].name, r[b].name);
  DeviceInfo* d = nullptr;
  int st = current_device(&d);
  if (st != QLA_OK) return st;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  LocalJob j{};
  j.k = static_cast<const uint16_t*>(k);
  j.v = static_cast<const uint16_t*>(v);
  j.beta = beta;
  j.g = g;
  j.H = H;
  j.M = M;
  j.nchains = (int)chains;
  j.T = T;
  j.S = S;
  j.L = L;
  j.K = K;
  j.V = V;
  j.layout = layout;
  j.pdl = dependent_launch();
  int F = split;
  if (F == 0 && (st = local_auto_split(j, d, &F)) != QLA_OK) return st;
  if (F > 1) {
    bool no_scratch = false;
    st = local_pass_split(j, F, d, cs, &no_scratch);
    // an automatic split that finds no memory for its scratch runs unsplit
    if (!(split == 0 && no_scratch)) return st;
    cudaGetLastError();
    t_last_error.clear();
  }
  const cudaError_t e = launch_local_simt(j, cs);
  return e == cudaSuccess ? QLA_OK : cuda_fail(e, "kernel launch");
}

int qla_device_status(int* flags) {
  t_last_error.clear();
  DeviceInfo* d = nullptr;
  int st = current_device(&d);
  if (st != QLA_OK) return st;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  unsigned int w = 0;
  if ((e = cudaMemcpy(&w, d->status_word, sizeof w, cudaMemcpyDeviceToHost)) != cudaSuccess)
    return cuda_fail(e, "read status word");
  const unsigned int zero = 0;
  if ((e = cudaMemcpy(d->status_word, &zero, sizeof zero, cudaMemcpyHostToDevice)) != cudaSuccess)
    return cuda_fail(e, "clear status word");
  if (flags) *flags = (int)w;
  if (w & kStatusTimeout) return QLA_ERR_TIMEOUT;
  return w ? QLA_ERR_INVALID_ARG : QLA_OK;
}

int qla_selftest_stalled_wait(const float* H, const float* M, float* out, int S, int wait_limit_us, int engine,
                              void* stream) {
  t_last_error.clear();
  Shape s{1, 1, S, 128, 128, QLA_LAYOUT_KV, QLA_FORWARD};
  int st = check_args(H, M, nullptr, out, nullptr, s);
  if (st != QLA_OK) return st;
  if (S < 2) return fail(QLA_ERR_INVALID_ARG, "the stalled-wait self-test needs S >= 2");
  if (wait_limit_us < 1 || wait_limit_us > 10000000)
    return fail(QLA_ERR_INVALID_ARG, "wait_limit_us must be in [1, 10^7]");
  if (engine != QLA_ENGINE_TC)
    return fail(QLA_ERR_INVALID_ARG, "the stalled-wait self-test takes the pipelined engine (got %d)", engine);
  DeviceInfo* d = nullptr;
  if ((st = current_device(&d)) != QLA_OK) return st;
  const uint64_t limit = (uint64_t)wait_limit_us * 1000ull;
  cudaStream_t cs = static_cast<cudaStream_t>(stream);
  SeqJob j = plain_job(H, M, nullptr, out, nullptr, s);
  j.status = d->status_word;
  cudaError_t e = launch_seq_tc(j, QLA_RELEASE_MEMBAR, d->status_word, limit, 1, cs);
  if (e != cudaSuccess) return cuda_fail(e, "kernel launch");
  return QLA_OK;
}

int qla_selftest_dependent_producer(const void* src, void* dst, size_t bytes, int delay_us, void* stream) {
  t_last_error.clear();
  if (!src || !dst) return fail(QLA_ERR_INVALID_ARG, "src and dst must not be NULL");
  if (bytes % 16) return fail(QLA_ERR_INVALID_ARG, "bytes must be a multiple of 16 (got %zu)", bytes);
  if ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst)) & 15)
    return fail(QLA_ERR_ALIGNMENT, "src and dst must be 16-byte aligned");
  const uintptr_t a = reinterpret_cast<uintptr_t>(src), b = reinterpret_cast<uintptr_t>(dst);
  if (bytes && a < b + bytes && b < a + bytes) return fail(QLA_ERR_ALIAS, "src and dst overlap");
  if (delay_us < 0 || delay_us > 100000) return fail(QLA_ERR_INVALID_ARG, "delay_us must be in [0, 100000]");
  DeviceInfo* d = nullptr;
  int st = current_device(&d);
  if (st != QLA_OK) return st;
  if (bytes == 0 && delay_us == 0) return QLA_OK;
  // A few CTAs only, so that the dependent grid finds free SMs and starts
  // while the producer is still sleeping.
  dependent_producer_kernel<<<std::min(16, d->sm_count), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const float4*>(src), static_cast<float4*>(dst), bytes / 16, (uint64_t)delay_us * 1000ull);
  const cudaError_t e = cudaGetLastError();
  return e == cudaSuccess ? QLA_OK : cuda_fail(e, "kernel launch");
}

}  // extern "C"
