// decode_common.cuh — device helpers shared by the decode kernels.
#pragma once

#include <cuda_bf16.h>
#include <stdint.h>

#include "decode_plan.h"
#include "ptx.cuh"

namespace lrkv {
namespace dec {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

__host__ __device__ inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// CTA that owns global token g when N tokens are cut into G ranges
// [floor(c N / G), floor((c+1) N / G)).
__device__ __forceinline__ int cta_of_token(long long g, long long N, long long G) {
  return static_cast<int>(((g + 1) * G - 1) / N);
}

// Byte offset of 16-byte chunk `chunk` of row `row` in a TMA box written with
// the swizzle of span `span` bytes (128, 64 or 32): address bits [4, 4+k) are
// XORed with bits [7, 7+k), k = log2(span / 16).
__device__ __forceinline__ int swz_off(int row, int chunk, int span) {
  const int off = row * span + chunk * 16;
  return off ^ (((off >> 7) & (span / 16 - 1)) << 4);
}

// ---------------------------------------------------------- element loads --
template <bool BF16, int NE>
__device__ __forceinline__ void load_vec(const unsigned char* p, float* f) {
  if constexpr (BF16) {
    if constexpr (NE == 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(p);
      f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
      f[4] = bf_lo(u.z); f[5] = bf_hi(u.z); f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
    } else {
      static_assert(NE == 4, "bf16 latent vectors are 4 or 8 elements");
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
    }
  } else {
    static_assert(NE == 4, "fp32 latent vectors are 4 elements");
    const float4 v = *reinterpret_cast<const float4*>(p);
    f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
  }
}

__device__ __forceinline__ float load_elem(const void* base, size_t i, bool bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
  return reinterpret_cast<const float*>(base)[i];
}

// ------------------------------------------------------ token-range walk --
// A CTA's token range [g0, g1) of the concatenated histories, visited tile by
// tile; tiles never straddle two sequences.
struct TileWalk {
  int b;       // sequence
  int t0;      // first row of the tile within the sequence
  int t_end;   // one past the last row of this CTA's piece of the sequence
};

__device__ __forceinline__ bool walk_first(TileWalk& w, const int* pre, int B, int g0, int g1) {
  if (g0 >= g1) return false;
  int lo = 0, hi = B - 1;  // last b with pre[b] <= g0
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= g0) lo = mid; else hi = mid - 1;
  }
  int b = lo;
  while (b < B && pre[b + 1] <= g0) ++b;  // skip empty sequences at g0
  if (b >= B) return false;
  w.b = b;
  w.t0 = g0 - pre[b];
  w.t_end = min(pre[b + 1], g1) - pre[b];
  return true;
}

__device__ __forceinline__ bool walk_next(TileWalk& w, const int* pre, int B, int g1, int T) {
  w.t0 += T;
  if (w.t0 < w.t_end) return true;
  int b = w.b + 1;
  while (b < B && pre[b] < g1 && pre[b + 1] == pre[b]) ++b;
  if (b >= B || pre[b] >= g1) return false;
  w.b = b;
  w.t0 = 0;
  w.t_end = min(pre[b + 1], g1) - pre[b];
  return true;
}

}  // namespace dec
}  // namespace lrkv
