// Host helper shared by the TMA engines: 2-D fp32 tensor maps.
#pragma once

#include <cuda.h>
#include <stdint.h>

namespace qla {

// 2-D fp32 tensor map: `rows` x `cols` row-major at `base`, box box_cols x
// box_rows, swizzle 0 (none), 32, 64 or 128 (bytes).  False when the driver
// entry point is missing or rejects the map.
bool make_map(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols, uint32_t box_rows,
              int swizzle);

}  // namespace qla
