// key_scale.cu — the joint reciprocal RMS of every cached key, for attention
// with post-projection RMSNorm of the keys ("Low-Rank Key Value Attention |
// What a shared cache can preserve", §8, "Post-projection normalization has a
// cache cost": one scale per head and token, computed at append time and
// multiplied into the summed score).  For head h and token j the key is
// k = s_j + z_j B_h^T (never the two parts normalised apart) and the scale is
// 1 / sqrt(mean_d k[d]^2 + eps), in fp32.
//
// One CTA = (sequence b, head h, 64 new tokens): B_h^K, the tokens' shared rows
// and their latents of head h staged in shared memory as fp32; four threads
// per token rebuild a quarter of the key each and sum its squares.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "lrkv.h"
#include "ptx.cuh"

namespace lrkv {

namespace {

constexpr int kKsTokens = 64;
constexpr int kKsThreads = 256;  // 4 per token

struct KeyScaleParams {
  int B, H, dh, r, max_len, n_new;
  float eps;
  const __nv_bfloat16* k_s;   // [B][max_len][dh]
  const __nv_bfloat16* z_k;   // [B][max_len][H][r]
  const __nv_bfloat16* b_k;   // [H][dh][r]
  const int32_t* start_pos;   // [B]
  float* key_scale;           // [B][H][max_len]
};

}  // namespace

__global__ void __launch_bounds__(kKsThreads) lrkv_key_scale_kernel(const KeyScaleParams p) {
  extern __shared__ float ks_smem[];
  const int h = blockIdx.y, b = blockIdx.z;
  const int t_first = blockIdx.x * kKsTokens;
  const int dh = p.dh, r = p.r;
  float* sB = ks_smem;                       // [dh][r]
  float* sZ = sB + dh * r;                   // [64][r]
  float* sS = sZ + kKsTokens * r;            // [64][dh]
  const int start = p.start_pos[b];
  const int tid = threadIdx.x;
  for (int i = tid; i < dh * r; i += blockDim.x)
    sB[i] = __bfloat162float(p.b_k[static_cast<size_t>(h) * dh * r + i]);
  for (int i = tid; i < kKsTokens * r; i += blockDim.x) {
    const int t = i / r, c = i - t * r, pos = start + t_first + t;
    const bool in = t_first + t < p.n_new && pos >= 0 && pos < p.max_len;
    sZ[i] = in ? __bfloat162float(p.z_k[((static_cast<size_t>(b) * p.max_len + pos) * p.H + h) * r + c]) : 0.f;
  }
  for (int i = tid; i < kKsTokens * dh; i += blockDim.x) {
    const int t = i / dh, d = i - t * dh, pos = start + t_first + t;
    const bool in = t_first + t < p.n_new && pos >= 0 && pos < p.max_len;
    sS[i] = in ? __bfloat162float(p.k_s[(static_cast<size_t>(b) * p.max_len + pos) * dh + d]) : 0.f;
  }
  __syncthreads();
  const int t = tid >> 2, part = tid & 3;    // token, quarter of the key
  const float* z = sZ + t * r;
  float ss = 0.f;
  for (int d = part; d < dh; d += 4) {
    const float* bd = sB + d * r;
    float k = sS[t * dh + d];
    for (int c = 0; c < r; ++c) k = fmaf(z[c], bd[c], k);
    ss = fmaf(k, k, ss);
  }
  ss += __shfl_xor_sync(0xffffffffu, ss, 1);
  ss += __shfl_xor_sync(0xffffffffu, ss, 2);
  const int pos = start + t_first + t;
  if (part == 0 && t_first + t < p.n_new && pos >= 0 && pos < p.max_len)
    p.key_scale[(static_cast<size_t>(b) * p.H + h) * p.max_len + pos] = 1.f / sqrtf(ss / dh + p.eps);
}

lrkv_status key_scale_launch(const lrkv_dims& dm, float eps, int n_new, const void* k_s, const void* z_k,
                             const void* b_k, const int32_t* start_pos, float* key_scale, void* stream) {
  KeyScaleParams p;
  p.B = dm.batch; p.H = dm.heads; p.dh = dm.head_dim; p.r = dm.rank; p.max_len = dm.max_len; p.n_new = n_new;
  p.eps = eps;
  p.k_s = static_cast<const __nv_bfloat16*>(k_s);
  p.z_k = static_cast<const __nv_bfloat16*>(z_k);
  p.b_k = static_cast<const __nv_bfloat16*>(b_k);
  p.start_pos = start_pos;
  p.key_scale = key_scale;
  const int smem = (dm.head_dim * dm.rank + kKsTokens * dm.rank + kKsTokens * dm.head_dim) * 4;
  static int have = 0;
  if (smem > 48 * 1024 && smem > have) {
    if (cudaFuncSetAttribute(lrkv_key_scale_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return LRKV_ERR_CUDA;
    have = smem;
  }
  const dim3 grid((n_new + kKsTokens - 1) / kKsTokens, dm.heads, dm.batch);
  lrkv_key_scale_kernel<<<grid, kKsThreads, smem, static_cast<cudaStream_t>(stream)>>>(p);
  return cudaGetLastError() == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

}  // namespace lrkv
