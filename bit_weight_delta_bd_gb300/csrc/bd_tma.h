// Host-side encoding of TMA tensor maps (2-D, row-major) through the driver
// entry point fetched from the CUDA runtime, so the library needs no direct
// link against libcuda.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace bd {

// Encodes a 2-D tiled tensor map over a row-major [rows][cols] matrix whose
// rows are `row_bytes` apart.  Returns false if the driver rejects it.
bool encode_tma_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t cols, uint64_t rows,
                   uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle);

}  // namespace bd
