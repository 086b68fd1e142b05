// Host helpers shared by the TMA engines: 2-D fp32 tensor maps and the
// per-job maps and checks of the tensor-core launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <mutex>

#include "qla_internal.h"
#include "tma_map.h"

namespace qla {

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
              int swizzle) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 4};
  cuuint32_t box[2] = {box_cols, box_rows};
  cuuint32_t estr[2] = {1, 1};
  const CUtensorMapSwizzle sw = swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                : swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                : swizzle == 32 ? CU_TENSOR_MAP_SWIZZLE_32B
                                                : CU_TENSOR_MAP_SWIZZLE_NONE;
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

bool tma_job_supported(const SeqJob& j) {
  if (job_grid(j, j.V / 32).x == 0) return false;  // one CTA per 32-column tile of each unit
  // Tensor-map row coordinates are 32-bit: every state's rows must be addressable.
  const int64_t states = j.cu_seg ? j.nstates : (int64_t)j.nchains * j.S;
  if (states * (int64_t)(j.K > j.V ? j.K : j.V) > 0x7fffffff) return false;
  // The tensor maps view H/out and M as 2-D arrays of all chains' states, so
  // chains must be packed back to back (H and out are absent in scan phase
  // 1a; variable-length jobs locate every chain and group through the
  // offsets).
  if (!j.cu_seg) {
    if ((j.H || j.out) && j.h_chain_stride != (int64_t)j.S * j.K * j.V) return false;
    if (j.m_chain_stride != (int64_t)j.S * j.K * j.K) return false;
  }
  return true;
}

bool make_job_maps(const SeqJob& j, int VT, int EC, CUtensorMap* map_h, CUtensorMap* map_out, CUtensorMap* map_m) {
  const int K = j.K;
  const uint64_t states = j.cu_seg ? (uint64_t)j.nstates : (uint64_t)j.nchains * j.S;
  const bool kv = j.layout == 0;
  const uint64_t rows = states * (kv ? (uint64_t)K : (uint64_t)j.V);
  const uint64_t cols = kv ? (uint64_t)j.V : (uint64_t)K;
  // H: kv box VT columns x K rows ((4 VT)-byte swizzle); vk box K columns x VT rows
  if (j.H && !make_map(map_h, j.H, rows, cols, kv ? VT : K, kv ? K : VT, kv ? 4 * VT : 0)) return false;
  // out: per-warp stores of [32 rows][EC columns] (kv, (4 EC)-byte swizzle) or [EC rows][32 columns] (vk)
  if (j.out && !make_map(map_out, j.out, rows, cols, kv ? EC : 32, kv ? 32 : EC, kv ? 4 * EC : 0)) return false;
  // M chunks: forward [128 rows][32 columns] (128-byte swizzle), reverse [32 rows][128 columns]
  const bool fwd = j.direction == 0;
  return make_map(map_m, j.M, states * K, K, fwd ? 32 : 128, fwd ? 128 : 32, fwd ? 128 : 0);
}

}  // namespace qla
