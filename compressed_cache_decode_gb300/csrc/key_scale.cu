// key_scale.cu — the joint reciprocal RMS of every cached key, for attention
// with post-projection RMSNorm of the keys ("Low-Rank Key Value Attention |
// What a shared cache can preserve", §8, "Post-projection normalization has a
// cache cost": one scale per head and token, computed at append time and
// multiplied into the summed score).  For head h and token j the key is
// k = s_j + z_j B_h^T (never the two parts normalised apart) and the scale is
// 1 / sqrt(mean_d k[d]^2 + eps), in fp32.
//
// The rebuild is a contraction per (sequence, head, block of 128 tokens):
// K = Z_h B_h^T (128 x d_h, inner dimension r) plus the shared rows, on the
// tensor cores (mma.sync m16n8k16: bf16 operands, exact products, fp32
// accumulation); the epilogue adds the shared row, squares and sums over d
// (thread, then quad), and writes 1 / sqrt(ss / d_h + eps).  B_h^K, the
// block's latent rows and shared rows are staged in shared memory by 16-byte
// asynchronous copies (all in flight at once) with padded row strides
// (conflict-free ldmatrix and epilogue reads).  Eight warps, 16 tokens each.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "host_cache.h"
#include "lrkv.h"
#include "ptx.cuh"

namespace lrkv {

namespace {

constexpr int kKsTok = 128;      // tokens per CTA (B_h is staged once for all of them)
constexpr int kKsThreads = 256;  // eight warps of 16 tokens
constexpr int kKsCols = 128;     // key columns per accumulator pass

struct KeyScaleParams {
  int B, H, dh, r, max_len, n_new;
  int rp;                     // rank padded to a multiple of 16 (zeros)
  int zs;                     // shared row stride (elements) of the B^K and latent rows: rp + 8
  int rvec;                   // rows copied in 16-byte pieces (r a multiple of 8, aligned bases)
  float eps;
  const __nv_bfloat16* k_s;   // [B][max_len][dh]
  const __nv_bfloat16* z_k;   // [B][max_len][H][r]
  const __nv_bfloat16* b_k;   // [H][dh][r]
  const int32_t* start_pos;   // [B]
  float* key_scale;           // [B][H][max_len]
};

// 16-byte asynchronous copy global -> shared; `valid` false fills zeros (no
// bytes are read; `src` is still a mapped address).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

}  // namespace

// DHC, RPC: head dim and padded rank as compile-time constants (0: read from
// the parameters), so that the staging loops' index arithmetic folds.
template <int DHC, int RPC>
__global__ void __launch_bounds__(kKsThreads) lrkv_key_scale_kernel(const KeyScaleParams p) {
  extern __shared__ __align__(16) unsigned char ks_raw[];
  const int dh = DHC ? DHC : p.dh, rp = RPC ? RPC : p.rp, zs = rp + 8;
  const int r = p.r;
  __nv_bfloat16* sB = reinterpret_cast<__nv_bfloat16*>(ks_raw);  // [dh][zs]
  __nv_bfloat16* sZ = sB + dh * zs;                              // [kKsTok][zs]
  __nv_bfloat16* sS = sZ + kKsTok * zs;                          // [kKsTok][dh + 8]
  const int h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, g = lane >> 2, q4 = lane & 3;
  const int t0 = blockIdx.x * kKsTok, start = p.start_pos[b];
  const int nt = min(kKsTok, p.n_new - t0);
  const __nv_bfloat16* bh = p.b_k + static_cast<size_t>(h) * dh * r;
  auto zrow = [&](int t) -> const __nv_bfloat16* {  // latent row of block token t, or null
    const int pos = start + t0 + t;
    if (t >= nt || pos < 0 || pos >= p.max_len) return nullptr;
    return p.z_k + ((static_cast<size_t>(b) * p.max_len + pos) * p.H + h) * r;
  };
  const uint4 zero4 = make_uint4(0u, 0u, 0u, 0u);
  const int ss_stride = dh + 8;  // staged shared rows, padded: the epilogue's quad reads hit distinct banks
  if (p.rvec) {
    // every row in 16-byte pieces, all copies in flight at once (cp.async,
    // zero-filled where a row lies outside the block or the cache)
    const int pr = rp / 8;  // 16-byte pieces per padded row
#pragma unroll 4
    for (int i = tid; i < dh * pr; i += kKsThreads) {
      const int d = i / pr, c8 = i - d * pr;
      const bool v = 8 * c8 < r;
      cp_async16(sB + d * zs + 8 * c8, v ? bh + static_cast<size_t>(d) * r + 8 * c8 : bh, v);
    }
#pragma unroll 4
    for (int i = tid; i < kKsTok * pr; i += kKsThreads) {
      const int t = i / pr, c8 = i - t * pr;
      const __nv_bfloat16* zr = zrow(t);
      const bool v = zr && 8 * c8 < r;
      cp_async16(sZ + t * zs + 8 * c8, v ? zr + 8 * c8 : bh, v);
    }
  } else {
    const __nv_bfloat16 zb = __float2bfloat16_rn(0.f);
    for (int i = tid; i < dh * rp; i += kKsThreads) {
      const int d = i / rp, c = i - d * rp;
      sB[d * zs + c] = c < r ? bh[static_cast<size_t>(d) * r + c] : zb;
    }
    for (int i = tid; i < kKsTok * rp; i += kKsThreads) {
      const int t = i / rp, c = i - t * rp;
      const __nv_bfloat16* zr = zrow(t);
      sZ[t * zs + c] = (zr && c < r) ? zr[c] : zb;
    }
  }
  const int pieces = dh / 8;
#pragma unroll 4
  for (int i = tid; i < kKsTok * pieces; i += kKsThreads) {
    const int t = i / pieces, c8 = i - t * pieces, pos = start + t0 + t;
    const bool v = t < nt && pos >= 0 && pos < p.max_len;
    cp_async16(sS + t * ss_stride + 8 * c8,
               v ? p.k_s + (static_cast<size_t>(b) * p.max_len + pos) * dh + 8 * c8 : p.k_s, v);
  }
  cp_async_wait_all();
  (void)zero4;
  __syncthreads();

  const int trow = 16 * warp;  // this warp's first token
  float ss0 = 0.f, ss1 = 0.f;  // sums of squares of tokens trow + g and trow + g + 8
  for (int dc = 0; dc < dh; dc += kKsCols) {
    const int nn = min(kKsCols, dh - dc) / 8;  // n tiles of 8 columns (a multiple of 4)
    float acc[kKsCols / 8][4];
#pragma unroll
    for (int j = 0; j < kKsCols / 8; ++j) acc[j][0] = acc[j][1] = acc[j][2] = acc[j][3] = 0.f;
    for (int kk = 0; kk < rp / 16; ++kk) {
      uint32_t a0, a1, a2, a3;
      ldsm_x4(a0, a1, a2, a3, sZ + (trow + (lane & 15)) * zs + 16 * kk + 8 * (lane >> 4));
      const int m = lane >> 3;
#pragma unroll
      for (int j = 0; j < kKsCols / 8; j += 2) {
        if (j < nn) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4(b0, b1, b2, b3, sB + (dc + 8 * (j + (m >> 1)) + (lane & 7)) * zs + 16 * kk + 8 * (m & 1));
          mma_bf16_16816(acc[j], a0, a1, a2, a3, b0, b1);
          mma_bf16_16816(acc[j + 1], a0, a1, a2, a3, b2, b3);
        }
      }
    }
#pragma unroll
    for (int j = 0; j < kKsCols / 8; ++j) {
      if (j < nn) {
        const int d = dc + 8 * j + 2 * q4;
        const uint32_t s0 = *reinterpret_cast<const uint32_t*>(sS + (trow + g) * ss_stride + d);
        const uint32_t s1 = *reinterpret_cast<const uint32_t*>(sS + (trow + g + 8) * ss_stride + d);
        const float k00 = acc[j][0] + bf_lo(s0), k01 = acc[j][1] + bf_hi(s0);
        const float k10 = acc[j][2] + bf_lo(s1), k11 = acc[j][3] + bf_hi(s1);
        ss0 = fmaf(k00, k00, fmaf(k01, k01, ss0));
        ss1 = fmaf(k10, k10, fmaf(k11, k11, ss1));
      }
    }
  }
  ss0 += __shfl_xor_sync(0xffffffffu, ss0, 1);
  ss0 += __shfl_xor_sync(0xffffffffu, ss0, 2);
  ss1 += __shfl_xor_sync(0xffffffffu, ss1, 1);
  ss1 += __shfl_xor_sync(0xffffffffu, ss1, 2);
  if (q4 == 0) {
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int t = trow + g + 8 * u, pos = start + t0 + t;
      if (t < nt && pos >= 0 && pos < p.max_len)
        p.key_scale[(static_cast<size_t>(b) * p.H + h) * p.max_len + pos] =
            1.f / sqrtf((u ? ss1 : ss0) / dh + p.eps);
    }
  }
}

lrkv_status key_scale_launch(const lrkv_dims& dm, float eps, int n_new, const void* k_s, const void* z_k,
                             const void* b_k, const int32_t* start_pos, float* key_scale, void* stream) {
  KeyScaleParams p;
  p.B = dm.batch; p.H = dm.heads; p.dh = dm.head_dim; p.r = dm.rank; p.max_len = dm.max_len; p.n_new = n_new;
  p.rp = (dm.rank + 15) / 16 * 16;
  p.zs = p.rp + 8;
  p.rvec = dm.rank % 8 == 0 && (reinterpret_cast<uintptr_t>(b_k) & 15u) == 0 &&
           (reinterpret_cast<uintptr_t>(z_k) & 15u) == 0;
  p.eps = eps;
  p.k_s = static_cast<const __nv_bfloat16*>(k_s);
  p.z_k = static_cast<const __nv_bfloat16*>(z_k);
  p.b_k = static_cast<const __nv_bfloat16*>(b_k);
  p.start_pos = start_pos;
  p.key_scale = key_scale;
  const int smem = ((dm.head_dim + kKsTok) * p.zs + kKsTok * (dm.head_dim + 8)) * 2;
  using Fn = void (*)(const KeyScaleParams);
  Fn kern = lrkv_key_scale_kernel<0, 0>;
  if (dm.head_dim == 128 && p.rp == 64) kern = lrkv_key_scale_kernel<128, 64>;
  else if (dm.head_dim == 128 && p.rp == 48) kern = lrkv_key_scale_kernel<128, 48>;
  else if (dm.head_dim == 128 && p.rp == 32) kern = lrkv_key_scale_kernel<128, 32>;
  else if (dm.head_dim == 64 && p.rp == 32) kern = lrkv_key_scale_kernel<64, 32>;
  if (ensure_kernel_smem(reinterpret_cast<const void*>(kern), smem) != cudaSuccess) return LRKV_ERR_CUDA;
  const dim3 grid((n_new + kKsTok - 1) / kKsTok, dm.heads, dm.batch);
  kern<<<grid, kKsThreads, smem, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

}  // namespace lrkv
