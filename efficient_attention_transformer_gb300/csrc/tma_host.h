// Host-side TMA tensor-map encoding through the driver entry point (no link
// against libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace flashgau {

// Encodes a 2-D bf16 tensor map over a row-major [rows, cols] matrix with
// leading dimension `ld` elements, box = box_cols x box_rows elements and
// 128-byte swizzling (box_cols * 2 must be 128).  Returns cudaSuccess or
// cudaErrorInvalidValue when the driver rejects the map.
cudaError_t make_tmap_bf16_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                              uint64_t ld, uint32_t box_rows, uint32_t box_cols);

// Same for fp32 elements (box_cols * 4 must be 128).
cudaError_t make_tmap_f32_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                             uint64_t ld, uint32_t box_rows, uint32_t box_cols);

}  // namespace flashgau
