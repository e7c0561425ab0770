// Host-side construction of tensor-memory-access (TMA) descriptors for
// row-major bf16 matrices, loaded in 128-byte swizzled boxes.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace csa {

// True when the driver provides cuTensorMapEncodeTiled.
bool tma_available();

// A [rows, cols] bf16 row-major matrix (row stride cols * 2 bytes, a multiple
// of 16) as a TMA source: boxes of box_cols x box_rows (box_cols * 2 = 128
// bytes, the 128-byte swizzle span).  Loads outside the matrix fill zeros.
cudaError_t tma_map_bf16(CUtensorMap *m, const void *base, int64_t rows, int64_t cols, uint32_t box_cols,
                         uint32_t box_rows);

}  // namespace csa
