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

// A bf16 [rows, cols] matrix stored in 64 x 64 blocks: block (i, j) holds
// rows 64i .. 64i+63 and columns 64j .. 64j+63 as 8 KB of row-major data,
// blocks ordered row-block-major (rows, cols multiples of 64).  Encoded as
// a 4-D map {column in block, row in block, column block, row block} with
// 128-byte swizzling; a box covers box_rows rows (32, 64 or a multiple of
// 64) of one column block, loaded at coordinates {0, r % 64, c / 64, r / 64}
// and laid out in shared memory like the same rows of a row-major tile.
// box_cblocks > 1: a box of 64 rows spans that many adjacent column blocks
// (64 * box_cblocks columns, contiguous in memory, laid out block after block).
cudaError_t make_tmap_bf16_blocked(CUtensorMap *map, const void *base, uint64_t rows,
                                   uint64_t cols, uint32_t box_rows, uint32_t box_cblocks = 1);

// Same for fp32 elements (box_cols * 4 must be 128).
cudaError_t make_tmap_f32_2d(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols,
                             uint64_t ld, uint32_t box_rows, uint32_t box_cols);

}  // namespace flashgau
