// Host-side encoding of TMA tensor maps (cuTensorMapEncodeTiled through the
// runtime's driver entry point, so the library needs no link to libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gqa {

// 2D map of a row-major [rows][cols] fp16 matrix with a 128-byte swizzle:
// boxes of box_cols (<= 64) x box_rows elements. Returns a CUDA error code
// (cudaErrorInvalidValue when the driver rejects the map).
cudaError_t encode_fp16_2d_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                                 uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows);

// 4D map of a (B, S, N, 128) fp16 query tensor (BSH layout, head size 128)
// with the 128-byte swizzle: boxes of 64 dims x G heads x 128/G positions x 1
// batch land as 128 rows of 128 bytes in (position, head) order, the layout of
// a 64-column K-major MMA operand box; positions past S read as zero.
// G must divide 128.
cudaError_t encode_fp16_query_sw128(CUtensorMap* map, const void* base, uint64_t B, uint64_t S, uint64_t N,
                                    uint32_t G);

// 4D map of a (B, S, N, 128) fp32 query tensor with the 128-byte swizzle:
// boxes of 32 dims x G heads x 128/G positions x 1 batch land as 128 rows of
// 128 bytes in (position, head) order; positions past S read as zero. G must
// divide 128.
cudaError_t encode_f32_query_sw128(CUtensorMap* map, const void* base, uint64_t B, uint64_t S, uint64_t N,
                                   uint32_t G);

// 2D map of a row-major [rows][cols] byte matrix without swizzle: boxes of
// box_cols (a multiple of 16, <= 256) x box_rows bytes land as box_rows dense
// rows; rows past the matrix read as zero.
cudaError_t encode_u8_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols, uint64_t row_stride_bytes,
                         uint32_t box_cols, uint32_t box_rows);

// 2D map of a row-major [rows][cols] byte matrix (int8 codes) with the
// 128-byte swizzle: boxes of box_cols (<= 128) x box_rows bytes.
cudaError_t encode_u8_2d_sw128(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                               uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows);

// 2D map of a row-major [rows][cols] fp32 matrix without swizzle: boxes of
// box_cols (<= 256) x box_rows elements land as box_rows rows of box_cols
// consecutive floats; elements past the matrix are read as zero.
cudaError_t encode_f32_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                          uint64_t row_stride_bytes, uint32_t box_cols, uint32_t box_rows);

}  // namespace gqa
