// tensor_maps.cuh -- host-side TMA descriptors used by the kernels.
#pragma once

#include <cuda.h>

#include "dsa_common.cuh"

namespace dsa {

// Key pool: dims {128 values, 64 slots, num_pages}, page stride as given;
// box = one page (fp8: 128-byte rows; bf16: 64-value halves), 128-byte swizzle.
bool encode_kcache_map(CUtensorMap* m, const RowsParams& p);

// Queries viewed as [rows * 64, 128] bf16; box {64 values, box_rows rows},
// 128-byte swizzle.
bool encode_q_map(CUtensorMap* m, const RowsParams& p, int box_rows);

}  // namespace dsa
