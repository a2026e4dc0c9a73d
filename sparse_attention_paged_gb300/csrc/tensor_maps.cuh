// tensor_maps.cuh -- host-side TMA descriptors used by the kernels.
#pragma once

#include <cuda.h>

#include "dsa_common.cuh"

namespace dsa {

// Both maps count in 4-byte units (TMA throughput is per element); a 128-byte
// row block is 32 units and the second half of a 256-byte bf16 row starts at
// unit kHalfRowUnits.
constexpr int kHalfRowUnits = 32;

// Key pool: dims {row bytes / 4, 64 slots, num_pages}, page stride as given;
// box = one page's 128-byte column block, 128-byte swizzle.
bool encode_kcache_map(CUtensorMap* m, const RowsParams& p);

// Queries viewed as [rows * 64, 64 units]; box {32 units, box_rows rows},
// 128-byte swizzle.
bool encode_q_map(CUtensorMap* m, const RowsParams& p, int box_rows);

}  // namespace dsa
