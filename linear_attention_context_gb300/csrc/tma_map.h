// Host helpers shared by the TMA engines: 2-D fp32 tensor maps (tma_map.cu).
#pragma once

#include <cuda.h>
#include <stdint.h>

#include "qla_internal.h"

namespace qla {

// 2-D fp32 tensor map: `rows` x `cols` row-major at `base`, box box_cols x
// box_rows, swizzle 0 (none), 32, 64 or 128 (bytes).  False when the driver
// entry point is missing or rejects the map.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
              int swizzle);

// Whether a tensor-core launch can take the job: its units fit the grid (at
// most 2^31 - 1, see job_grid), every state row has a 32-bit
// tensor-map coordinate, and chains are packed back to back (the maps view
// all chains' states as one 2-D array) unless the job locates them through
// variable-length offsets.
bool tma_job_supported(const SeqJob& j);

// The three maps of a tensor-core launch with VT-column CTA tiles and
// per-warp out stores of EC columns: H (skipped when null), out (skipped when
// null) and M.  False when a map cannot be encoded.
bool make_job_maps(const SeqJob& j, int VT, int EC, CUtensorMap* map_h, CUtensorMap* map_out, CUtensorMap* map_m);

}  // namespace qla
