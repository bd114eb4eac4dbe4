// tmap.h — host-side creation of TMA tensor maps through the driver entry
// point (no link against libcuda).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cstdint>

namespace lrkv {

// Encode a 3-D tiled tensor map for a row-major [d2][d1][d0] tensor of 2-byte
// elements with box {b0, b1, 1} and the given swizzle.  Returns false on
// failure (driver entry point missing or arguments rejected).
bool make_tmap_3d_bf16(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2,
                       uint32_t b0, uint32_t b1, CUtensorMapSwizzle swizzle);

// Encode a 4-D tiled tensor map of 2-byte elements with explicit byte
// strides for dimensions 1..3 (any order; each a multiple of 16), box
// {b0, b1, b2, b3} and no swizzle.  Box elements outside the extents are
// filled with zeros.  Returns false on failure.
bool make_tmap_4d_bf16_strided(CUtensorMap* map, const void* base, const uint64_t dims[4],
                               const uint64_t strides_bytes[3], const uint32_t box[4]);

// As make_tmap_4d_bf16_strided, with the 128-byte swizzle (b0 * 2 <= 128).
bool make_tmap_4d_bf16_swizzled(CUtensorMap* map, const void* base, const uint64_t dims[4],
                                const uint64_t strides_bytes[3], const uint32_t box[4]);

// Encode a 2-D tiled tensor map for a row-major [d1][d0] fp32 tensor with box
// {b0, b1} (b0 may exceed d0: the excess is filled with zeros) and no swizzle.
bool make_tmap_2d_f32(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint32_t b0, uint32_t b1);

// Encode a 3-D tiled tensor map for a row-major [d2][d1][d0] fp32 tensor
// (d0 * 4 a multiple of 16) with box {b0, b1, 1} and no swizzle; box elements
// outside the extents are filled with zeros.
bool make_tmap_3d_f32(CUtensorMap* map, const void* base, uint64_t d0, uint64_t d1, uint64_t d2, uint32_t b0,
                      uint32_t b1);

}  // namespace lrkv
