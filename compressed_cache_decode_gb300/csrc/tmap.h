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

}  // namespace lrkv
