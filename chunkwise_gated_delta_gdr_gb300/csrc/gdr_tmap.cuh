// gdr_tmap.cuh -- TMA tensor-map encoding shared by the fast-path launchers.
#pragma once

#include <cuda.h>
#include <stddef.h>

namespace gdr {
namespace fast {

// Tiled map with unit element strides, 128-byte L2 promotion and zero fill out
// of range. False when the driver entry point is missing or the driver rejects
// the layout (base or strides not 16-byte aligned, box too large, ...).
bool tmap_encode(CUtensorMap* map, CUtensorMapDataType type, int rank, const void* base,
                 const cuuint64_t* dims, const cuuint64_t* strides, const cuuint32_t* box,
                 CUtensorMapSwizzle swz);

// [B, T, heads, 128] bf16 tensor; box {64 channels, 1 head, 64 steps, 1},
// 128-byte swizzle (one 8 KB tile per box).
bool tmap_bthd(CUtensorMap* map, const void* base, int B, int T, int heads);

// `count` blocks of `rows` x `cols` elements of `esize` bytes, block i at
// base + i * block_bytes, rows packed; box {box_cols, box_rows, 1}.
bool tmap_blocks(CUtensorMap* map, const void* base, CUtensorMapDataType type, int esize,
                 int cols, int rows, size_t count, size_t block_bytes, int box_cols, int box_rows,
                 CUtensorMapSwizzle swz);

}  // namespace fast
}  // namespace gdr
