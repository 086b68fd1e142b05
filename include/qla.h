/*
 * qla.h -- C ABI of the GB300 (sm_103a) context-parallel state-correction pass.
 *
 * The operation.  Antarx Memos, "一次 TileLang Warp Specialization 数值错误的定位
 * 与修复：从双缓冲竞争到 membar", section "从版本升级后的数值偏差开始": a long
 * sequence is split into S segments; each segment yields a local state H_i
 * ("ht") and a K x K propagation matrix M_i ("mt"); one kernel corrects the
 * segment-initial states on the forward pass and the segment-terminal states
 * on the reverse pass, with the state stored K x V ("kv") or V x K ("vk").
 * Section "理解三个缓冲区，才能判断哪里需要同步" gives the recurrence (its
 * formula was lost in text extraction; the reading below follows the buffer
 * roles the same section lists):
 *
 *     X_0 = h_init,   X_{i+1} = propagate(M_i, X_i) + H_i
 *
 *                    forward          reverse
 *     kv (K x V)     M_i X            M_i^T X
 *     vk (V x K)     X M_i^T          X M_i
 *
 * Outputs are exclusive, one state per segment, in H's shape:
 *     forward  out[i] = X_i                                   i = 0..S-1
 *     reverse  out[S-1] = h_init,
 *              out[i] = propagate_rev(M_{i+1}, out[i+1]) + H_{i+1}
 * so the forward pass never reads H_{S-1}, M_{S-1} and the reverse pass never
 * reads H_0, M_0 -- unless the final state is requested (qla_cp_correct_ex),
 * which is the state after the last segment: X_S going forward,
 * propagate_rev(M_0, out[0]) + H_0 in reverse.
 *
 * Memory (all fp32, contiguous, row-major, DEVICE pointers owned by the caller):
 *     H      [B][heads][S][K][V]  (kv)   or  [B][heads][S][V][K]  (vk)
 *     M      [B][heads][S][K][K]         (independent of the layout)
 *     h_init [B][heads][K][V]     (kv)   or  [B][heads][V][K]     (vk);  NULL = zeros
 *     out    same shape as H
 *
 * Calls are asynchronous and stream-ordered on `stream` (a cudaStream_t; NULL
 * is the legacy default stream).  A status other than QLA_OK from the argument
 * checks means nothing was launched; a launch failure inside the scan variant
 * may leave its earlier phases enqueued (their results are then unused
 * scratch).  Device-side faults surface at the caller's next synchronisation,
 * as with any CUDA launch.
 *
 * Aliasing: out == H (exactly the same pointer) is supported and computes the
 * same result as separate buffers: each tile's H_i is read before out[i] is
 * written over it.  Any other overlap among H, M, h_init, out and final_state
 * returns QLA_ERR_ALIAS.  H, M and h_init are never written.
 *
 * Limits: B, heads, S >= 1; K and V multiples of 32 in [32, 256]; every pointer
 * 16-byte aligned; B*heads*S*(V/32) < 2^31 (one CTA per chain and 32-column
 * tile, per scan group in the scan variant) and B*heads*S*K*max(K,V) < 2^62
 * (QLA_ERR_UNSUPPORTED or QLA_ERR_INVALID_ARG otherwise).  The device must be
 * sm_103 (GB300): checked once per device, QLA_ERR_ARCH otherwise.
 */
#ifndef QLA_H_
#define QLA_H_

#include <stddef.h>

/* Exported symbols; everything else in the library has hidden visibility. */
#if defined(__GNUC__)
#define QLA_API __attribute__((visibility("default")))
#else
#define QLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

enum { QLA_LAYOUT_KV = 0, QLA_LAYOUT_VK = 1 };
enum { QLA_FORWARD = 0, QLA_REVERSE = 1 };

enum {
  QLA_OK = 0,
  QLA_ERR_INVALID_ARG = -1, /* null pointer, non-positive size, unknown enum */
  QLA_ERR_UNSUPPORTED = -2, /* K or V outside the supported set, engine not built for the shape */
  QLA_ERR_ALIGNMENT = -3,   /* a pointer not 16-byte aligned */
  QLA_ERR_ALIAS = -4,       /* overlapping buffers other than out == H */
  QLA_ERR_CUDA = -5,        /* a CUDA runtime call failed; qla_last_error() has its text */
  QLA_ERR_ARCH = -6,        /* the current device is not sm_103 */
  QLA_ERR_TIMEOUT = -7      /* a bounded device-side wait gave up (see qla_device_status) */
};

/* Which algorithm computes the recurrence. */
enum {
  QLA_VARIANT_AUTO = 0, /* the library chooses from the shape */
  QLA_VARIANT_SEQ = 1,  /* one sequential pass per (chain, column tile) */
  QLA_VARIANT_SCAN = 2  /* group aggregates -> carry pass -> per-group re-run (small B*heads) */
};

/* Which kernel engine runs the sequential pass. */
enum {
  QLA_ENGINE_AUTO = 0,    /* 3xTF32 engine where the shape and chain length allow, else SIMT */
  QLA_ENGINE_SIMT = 1,    /* plain FFMA kernel, no TMA: any supported K, V */
  /* (value 2 is not used: it is rejected with QLA_ERR_INVALID_ARG) */
  QLA_ENGINE_TC = 3       /* warp-specialised TMA/mbarrier pipeline, tcgen05 3xTF32 propagate */
};
/* Accuracy on long chains and the automatic engine choice.  The tensor core
 * accumulates in fp32 rounding toward zero, so with norm-preserving M (no
 * decay) the tensor-core engine shrinks the state coherently, about 4.4e-8
 * of its norm per step at K = 128 and 1.4e-7 at K = 256: the worst per-state
 * relative L2 error passes 1e-5 near 200 steps (K = 128) and 64 steps
 * (K = 256).  QLA_ENGINE_AUTO therefore takes the 3xTF32 engine only for
 * chains of at most 160 segments (K = 128) or 48 segments (K = 256) and the
 * FFMA engine, which rounds to nearest (about 3e-6 at 512 steps), for longer
 * ones, in both variants; with variable lengths the bound is max_segments (T
 * for the sequential variant).  An engine asked for explicitly is used as
 * asked, whatever the chain length. */

/* How a consumer releases a double-buffer slot it has read with ordinary
 * shared-memory loads, before the TMA producer may overwrite it (section
 * "三个可用源码方案的具体差别" of the page above). */
enum {
  QLA_RELEASE_MEMBAR = 0, /* membar.cta, then mbarrier arrive (the page's adopted fix) */
  QLA_RELEASE_PROXY = 1,  /* fence.proxy.async.shared::cta, then arrive */
  QLA_RELEASE_DELAY = 2,  /* arrive only at the end of the step (longer slot lifetime) */
  QLA_RELEASE_NONE = 3    /* mbarrier arrive alone (its default .release semantics) */
};

/*
 * The state correction with the library's default choices.
 * Arguments as described at the top of this file.  Returns QLA_OK or a
 * negative QLA_ERR_* code; nothing is launched unless QLA_OK.
 */
QLA_API int qla_cp_correct(const float* H, const float* M, const float* h_init, float* out, int B,
                   int heads, int S, int K, int V, int layout, int direction, void* stream);

/*
 * As qla_cp_correct, with explicit choices:
 *   final_state  NULL, or a [B][heads][state] buffer that receives the state
 *                after the last segment (reads H and M of the last segment
 *                visited as well).  out may be NULL when final_state is not.
 *   variant      QLA_VARIANT_*;  engine QLA_ENGINE_*;  release QLA_RELEASE_*
 *                (ignored by engines without a TMA producer).
 *   scan_group   number of scan groups G (QLA_VARIANT_SCAN), 0 = automatic;
 *                each group covers ceil(S / G) consecutive segments.  The
 *                automatic G is at most round(sqrt(2 S)) and fewer where the
 *                phases' CTAs (one per chain, group and 32-column tile) would
 *                run in several waves on the device's SMs.
 * QLA_VARIANT_AUTO takes the scan where a cost model of both variants (fitted
 * to GB300 timings at K = V = 128; qla_resolve reports the choice) rates it
 * below 0.95 of the sequential kernel: long chains with few heads.
 * The scan variant needs qla_scan_workspace_bytes() of device scratch, which
 * it takes from the stream-ordered allocator (cudaMallocAsync on `stream`) and
 * returns on the same stream.
 */
QLA_API int qla_cp_correct_ex(const float* H, const float* M, const float* h_init, float* out,
                      float* final_state, int B, int heads, int S, int K, int V, int layout,
                      int direction, int variant, int engine, int release, int scan_group,
                      void* stream);

/*
 * Variable-length form.  Antarx Memos, "一次 TileLang Warp Specialization 数值
 * 错误的定位与修复", sections "验证分别回答了什么问题" and "性能结果", list
 * variable-length inputs among the configurations the full operator is
 * checked and timed on, without fixing a layout; here the offsets follow the
 * cu_seqlens convention of varlen attention kernels.  N sequences share the
 * segment axis: sequence n owns segments cu_seg[n] .. cu_seg[n+1] - 1, so it
 * has cu_seg[n+1] - cu_seg[n] >= 0 segments, and each (sequence, head) chain
 * is the fixed-length recurrence over its own segments.
 *   H, out       [heads][T][state]: head h's segments of all sequences, packed;
 *                out may equal H (in place) or be NULL when final_state is not.
 *   M            [heads][T][K][K].
 *   h_init       [N][heads][state] or NULL (zero initial states).
 *   final_state  [N][heads][state] or NULL; a sequence without segments gets
 *                its initial state.
 *   cu_seg       DEVICE pointer to N + 1 int32 offsets, cu_seg[0] = 0,
 *                non-decreasing, cu_seg[N] = T (4-byte aligned).
 * Sequential variant; engine QLA_ENGINE_*.  The host checks everything but
 * the offsets' values; a kernel that finds a chain's offsets outside [0, T]
 * or decreasing skips that chain (reads and writes nothing for it) and sets
 * bit 1 (value 2) of the device status word (qla_device_status).
 * Requires N*heads*(V/32) < 2^31 (times the scan's group count for the scan
 * variant) and heads*T < 2^31.
 */
QLA_API int qla_cp_correct_varlen(const float* H, const float* M, const float* h_init, float* out,
                          float* final_state, const int* cu_seg, int N, int T, int heads, int K,
                          int V, int layout, int direction, int engine, void* stream);

/*
 * qla_cp_correct_varlen with a variant choice.  The scan variant needs the
 * groups' size on the host without reading the device offsets, so the caller
 * passes `max_segments`, an upper bound on every sequence's segment count
 * (1 .. T; 0 means T; the sequential variant uses it only for the automatic
 * engine choice).  Every chain is cut
 * into G groups of L consecutive segments, G = scan_group (0: automatic from
 * max_segments) and L = ceil(max_segments / G); groups past a sequence's end
 * are empty (their aggregates are the identity and zero).  A sequence longer
 * than max_segments is treated like invalid offsets: bit 1 of the device
 * status word is set and that chain's outputs are left unspecified.
 * variant QLA_VARIANT_AUTO decides as for fixed lengths with S = max_segments
 * and N * heads chains (qla_resolve).  The scan
 * allocates its workspace with cudaMallocAsync on `stream`
 * (N * heads * G * (K*K + 2*K*V) * 4 bytes) and frees it the same way.
 */
QLA_API int qla_cp_correct_varlen_ex(const float* H, const float* M, const float* h_init, float* out,
                          float* final_state, const int* cu_seg, int N, int T, int heads, int K,
                          int V, int layout, int direction, int variant, int engine,
                          int max_segments, int scan_group, void* stream);

/* Bytes of device scratch the scan variant uses for this shape and group
 * size (0 = automatic, for the current device; without a usable device, for
 * G = round(sqrt(2 S)), which is never less); 0 when the scan does not apply. */
QLA_API size_t qla_scan_workspace_bytes(int B, int heads, int S, int K, int V, int scan_group);

/* Process-wide override of the automatic variant choice: QLA_VARIANT_SEQ or
 * QLA_VARIANT_SCAN make every call that asks for QLA_VARIANT_AUTO (and
 * qla_cp_correct, which always does) use that variant; QLA_VARIANT_AUTO
 * restores the shape-based rule.  Its initial value comes from the
 * environment variable QLA_VARIANT ("auto", "seq", "scan" or 0, 1, 2; unset or
 * anything else: auto), read at the first call that needs it.  Returns
 * QLA_ERR_INVALID_ARG for other values.  The choice never changes results
 * beyond the parity bar (the variants compute the same recurrence). */
QLA_API int qla_set_variant(int variant);

/* Process-wide switch (0 off, 1 on) for programmatic dependent launch
 * (xuesongtap, "PTX 内存一致性", section on PDL and griddepcontrol): when on,
 * the sequential variant's kernel is launched with programmatic stream
 * serialization, so it may become resident while the stream's previous kernel
 * is still running, once that kernel has triggered (griddepcontrol.
 * launch_dependents) in all its CTAs.  Every kernel of this library executes
 * griddepcontrol.wait before its first global-memory access (H, M, h_init,
 * the offsets, out, final_state), so data the previous kernel writes is
 * read only after that kernel has completed and its writes are visible: the
 * trigger never stands for data readiness.  The kernels trigger their own
 * dependents after their last step.  The scan variant's launches follow an
 * allocation or an event and are never dependent launches.  Initial value from
 * the environment variable QLA_PDL ("1" or "on": on; anything else: off), read
 * at the first call that needs it.  Returns QLA_ERR_INVALID_ARG for other
 * values. */
QLA_API int qla_set_dependent_launch(int enable);

/* The variant and engine QLA_*_AUTO resolve to for this shape on the current
 * device (written to *variant and *engine; either may be NULL). */
QLA_API int qla_resolve(int B, int heads, int S, int K, int V, int layout, int* variant, int* engine);

/* Static text for a status code. */
QLA_API const char* qla_status_string(int status);

/* Detail of the last failure on the calling host thread ("" if none). */
QLA_API const char* qla_last_error(void);

/*
 * Reads and clears the device-side status word of the current device.  Bit 0
 * (value 1): one of a kernel's bounded waits gave up (the kernel then drained
 * its copies in flight and returned early, leaving its outputs incomplete).
 * Bit 1 (value 2): a variable-length call met invalid offsets and skipped
 * those chains.  Synchronises the device.  *flags receives the word (0 = no
 * event); returns QLA_ERR_TIMEOUT if bit 0 was set, else QLA_ERR_INVALID_ARG
 * if the word was non-zero, QLA_OK otherwise, QLA_ERR_CUDA on error.
 */
QLA_API int qla_device_status(int* flags);

/*
 * Self-test of the bounded waits: launches the warp-specialised pipeline
 * (engine QLA_ENGINE_TC; any other value is QLA_ERR_INVALID_ARG) on a tiny
 * problem in a mode where one consumer waits
 * on a barrier that nothing arrives on.  The wait gives up after
 * `wait_limit_us` microseconds, the kernel records QLA_ERR_TIMEOUT in the
 * device status word, drains and returns.  The buffers are as for
 * qla_cp_correct with K = V = 128; returns the launch status.  Used by the
 * tests to show that a stalled pipeline ends on its own.
 */
QLA_API int qla_selftest_stalled_wait(const float* H, const float* M, float* out, int S,
                              int wait_limit_us, int engine, void* stream);

/*
 * Test producer for the dependent launch: copies `bytes` (a multiple of 16)
 * from src to dst (device pointers, 16-byte aligned, not overlapping) on
 * `stream` with a few CTAs that trigger their dependents at once and then
 * sleep `delay_us` (0 .. 100000) microseconds before copying.  A correction
 * launched right after it with the dependent launch switched on starts
 * during the sleep, so it reads the copied bytes correctly only through its
 * griddepcontrol.wait.  Returns the launch status.
 */
QLA_API int qla_selftest_dependent_producer(const void* src, void* dst, size_t bytes, int delay_us,
                                            void* stream);

/*
 * The scan variant without any allocation (this entry point has no
 * counterpart on the pages; it exists for callers of this library).
 *
 * Some callers cannot call cudaMalloc or cudaMallocAsync: code that runs with
 * a fixed device-memory budget handed out at start-up (an inference server's
 * arena, an embedded or real-time host loop) must not grow the process's
 * device footprint per call, and cudaMalloc can synchronise the device, which
 * a latency-bound caller cannot afford.  This entry point runs the same scan
 * as qla_cp_correct_ex(..., QLA_VARIANT_SCAN, ...) but keeps its scratch in a
 * fixed device array inside the library (QLA_SCAN_STATIC_BYTES, allocated when
 * the library is loaded and held by every GPU that loads it until the process
 * exits), so it allocates nothing: no cudaMalloc, cudaMallocAsync, cudaFree or
 * allocating library routine.  The caller still passes H, M, h_init, out and
 * final_state as for qla_cp_correct_ex.
 *
 * - Scratch needed is qla_scan_workspace_bytes(B, heads, S, K, V, scan_group);
 *   a shape that needs more than QLA_SCAN_STATIC_BYTES returns
 *   QLA_ERR_UNSUPPORTED (qla_last_error() gives both sizes) and launches
 *   nothing.
 * - The first call on a device looks up that device's address of the array
 *   (once per device, with that device current); make that first call before
 *   any stream capture on the device.
 * - Every call on a device shares the one array and it keeps the last call's
 *   contents.  Nothing in it needs to start at zero: each scan phase writes
 *   every scratch element it later reads.  Calls whose work overlaps on the
 *   GPU (two streams, or two host threads without ordering) race on the
 *   array; order them on one stream.
 */
#define QLA_SCAN_STATIC_BYTES (8u << 20)
QLA_API int qla_cp_correct_scan_static(const float* H, const float* M, const float* h_init, float* out,
                                       float* final_state, int B, int heads, int S, int K, int V, int layout,
                                       int direction, int engine, int release, int scan_group, void* stream);

/*
 * The per-segment local pass that produces H and M for the correction.
 * Antarx Memos, "一次 TileLang Warp Specialization 数值错误的定位与修复", section
 * "从版本升级后的数值偏差开始", names each segment's local state ("ht") and
 * propagation matrix ("mt") but not how they are computed; this library reads
 * them as the gated delta rule (Yang, Kautz, Hatamizadeh, "Gated Delta
 * Networks", ICLR 2025), token by token in the kv view:
 *
 *     X_t = a_t (I - b_t k_t k_t^T) X_{t-1} + b_t k_t v_t^T,   a_t = exp(g_t),
 *
 * and for segment i (tokens i*L .. i*L + L - 1, L = T / S):
 *     H_i = that recurrence's state after the segment, from X = 0,
 *     M_i = A_last ... A_first,   A_t = a_t (I - b_t k_t k_t^T),
 * so that the state after the segment is M_i X_enter + H_i, the forward
 * recurrence qla_cp_correct composes (the reverse pass needs the segments'
 * local gradients, which this pass does not compute).
 *
 * Memory (DEVICE pointers owned by the caller, contiguous, row-major):
 *     k     [B][heads][T][K]  bf16 (16-bit patterns), 16-byte aligned
 *     v     [B][heads][T][V]  bf16, 16-byte aligned
 *     beta  [B][heads][T]     fp32 write strengths, 4-byte aligned
 *     g     [B][heads][T]     fp32 log-space decays, 4-byte aligned
 *     H     [B][heads][S][K][V] (kv) or [B][heads][S][V][K] (vk), fp32, or NULL
 *     M     [B][heads][S][K][K] fp32, or NULL (not both NULL); 16-byte aligned
 * exactly the H and M arguments of qla_cp_correct.  T must be a multiple of S;
 * K and V multiples of 32 in [32, 256].  H and M may not overlap each other or
 * the inputs (QLA_ERR_ALIAS).  Decays are applied as a running scale kept in
 * fp64 (no fp32 compounding); a single token whose g_t is below about -80
 * empties the state (exp underflows), as in exact arithmetic to fp32 range.
 * Asynchronous on `stream`.  With the dependent-launch switch on
 * (qla_set_dependent_launch) the kernel is itself a programmatic dependent,
 * and it lets the next kernel on the stream launch at once: a correction
 * enqueued right after it starts its set-up early and reads H and M only
 * after this kernel has completed.
 */
QLA_API int qla_local_pass(const void* k, const void* v, const float* beta, const float* g, float* H, float* M,
                           int B, int heads, int T, int S, int K, int V, int layout, void* stream);

/*
 * qla_local_pass with the sub-segment split chosen by the caller.  All of a
 * pass's CTAs run the same number of tokens, so when they exceed what the SMs
 * hold at once, the last partial wave costs a whole segment's time on a few
 * SMs.  With split = F > 1 each segment is run as F sub-segments of L / F
 * tokens (shorter units, more waves), and the F sub-segments' maps are then
 * composed per segment by the correction kernels: M_i = the product of the
 * sub-segment M's, H_i = their recurrence from zero (the same affine
 * composition the correction applies across segments).  The results equal
 * split = 1 up to rounding.  The sub-segments' H and M take
 * B*heads*S*F*(K*K + K*V)*4 bytes of device scratch from the stream-ordered
 * allocator (cudaMallocAsync on `stream`, returned the same way).
 *   split  0: automatic (the F in {1, 2, 4, 8, 16} that minimises the
 *          estimated time, from the launch's occupancy on this device;
 *          when its scratch cannot be allocated, the pass runs unsplit);
 *          otherwise F, which must divide L = T / S (an allocation failure
 *          is then returned as QLA_ERR_CUDA, with nothing launched).
 * qla_local_pass is split = 0.
 */
QLA_API int qla_local_pass_ex(const void* k, const void* v, const float* beta, const float* g, float* H, float* M,
                              int B, int heads, int T, int S, int K, int V, int layout, int split, void* stream);

/* ABI version of this header (major * 100 + minor). */
QLA_API int qla_version(void);

#ifdef __cplusplus
}
#endif

#endif /* QLA_H_ */
