// Host-side encoding of TMA tensor maps (2-D, row-major) through the driver
// entry point fetched from the CUDA runtime, so the library needs no direct
// link against libcuda.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace bd {

// Encodes a 2-D tiled tensor map over a row-major [rows][cols] matrix whose
// rows are `row_bytes` apart.  Returns false if the driver rejects it.  A map
// depends only on its arguments, so encoded maps are kept in a bounded
// per-thread cache: repeated calls on the same buffers (W_base, the variants'
// sign tables, the workspace) do not call the driver again.
bool encode_tma_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t cols, uint64_t rows,
                   uint64_t row_bytes, uint32_t box_cols, uint32_t box_rows, CUtensorMapSwizzle swizzle);

// Raises a kernel's dynamic shared-memory limit on the current device to at
// least `bytes` and asks for the largest shared-memory carve-out, calling the
// runtime only the first time per device (the attributes persist);
// `per_device` is one counter array per kernel.
cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes, std::atomic<size_t>* per_device);

constexpr int kHostMaxDevices = 64;

}  // namespace bd
