// tmap.cuh -- TMA tensor-map encoding (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace poetx {

// 2-D row-major tensor [rows, cols] of `elem_bytes`-byte elements; boxes of
// box_rows x box_cols (box_cols * elem_bytes <= 128 with the 128-byte
// swizzle).  Out-of-range elements load as zero.  Returns false on failure
// (base not 16-byte aligned, row pitch not a multiple of 16 bytes, ...).
bool make_tmap_2d(CUtensorMap* map, const void* base, CUtensorMapDataType dtype, int elem_bytes,
                  uint64_t rows, uint64_t cols, uint32_t box_rows, uint32_t box_cols,
                  CUtensorMapSwizzle swizzle);

}  // namespace poetx
