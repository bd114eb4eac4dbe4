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
#include <cstdlib>
#include <cstring>

#include "host_cache.h"
#include "lrkv.h"
#include "ptx.cuh"
#include "tmap.h"

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

bool a16(const void* q) { return (reinterpret_cast<uintptr_t>(q) & 15u) == 0; }

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

// ---------------------------------------------------------------------------
// The same scales on the 5th-generation tensor cores (tcgen05, TMEM), for
// d_h in {64, 128} and r <= 64 a multiple of 8.  CTA = (128-token tile of one
// sequence, group of kKtHeads heads).  The tile's shared rows are copied once
// (TMA, 128-byte swizzle); per head, Z_h (128 tokens x r, padded to 64 with
// zeros by the copy) and B_h (d_h x r) land in a two-stage ring and one
// thread issues K = Z_h B_h^T as 4 MMAs (M 128, N d_h, K 16 each) into one of
// two TMEM accumulators, so that the epilogue of head i (8 warps: one token
// and half of the columns per thread, TMEM row + shared row, squared and
// summed; the halves meet in shared memory) overlaps the MMAs of head i + 1.
// Measured on 2 x 4096 tokens of 32 heads (d_h 128, r 64): 14.6 us per launch
// (ncu; the mma.sync form 27 us), latency-bound (DRAM 31%, L2 21% busy).
// Slower on the same box: the shared rows held in registers with a
// three-stage ring, and an L2 prefetch of the group's latents at entry.
constexpr int kKtHeads = 8;      // heads per CTA
constexpr int kKtStages = 2;     // ring stages of (Z_h, B_h)
constexpr int kKtThreads = 320;  // warp 0 copies, warp 1 MMAs, warps 2-9 epilogue (two per lane quadrant)
constexpr int kKtZBytes = 128 * 128;      // 128 rows x 64 bf16
constexpr int kKtBBytes = 128 * 128;      // up to 128 rows (d) x 64 bf16

struct KtMaps {
  CUtensorMap z;  // z_k as (r, H, max_len, B), box (64, 1, 128, 1)
  CUtensorMap b;  // b_k as (r, d_h, H), box (64, d_h, 1)
  CUtensorMap s;  // k_s as (d_h, max_len, B), box (64, 128, 1)
};

template <int DH>
__global__ void __launch_bounds__(kKtThreads, 1)
    lrkv_key_scale_tc_kernel(const KeyScaleParams p, const __grid_constant__ KtMaps maps) {
  constexpr int NSB = DH / 64;                // 64-column boxes of a shared row
  constexpr int kSBytes = NSB * 128 * 128;    // shared rows of the tile
  constexpr uint32_t kTCols = 2 * DH;         // two accumulators of DH columns
  extern __shared__ __align__(16) unsigned char kt_raw[];
  __shared__ uint64_t full[kKtStages], empty[kKtStages], sfull, accf[2], acce[2];
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail, s_issued, s_mmas;  // heads whose copies / MMAs were issued
  __shared__ float s_half[2][128];           // second-half sums of squares per accumulator and token
  unsigned char* smem = kt_raw + ((1024u - (smem_u32(kt_raw) & 1023u)) & 1023u);
  unsigned char* s_rows = smem;                                  // [NSB][128 rows][128 B], swizzled
  unsigned char* ring = smem + kSBytes;                          // [stage] {Z 16 KB, B 16 KB}
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.z, h0 = blockIdx.y * kKtHeads, t0 = blockIdx.x * 128;
  const int nh = min(kKtHeads, p.H - h0);
  const int pos0 = p.start_pos[b] + t0;

  if (threadIdx.x == 0) {
    for (int st = 0; st < kKtStages; ++st) {
      mbar_init(&full[st], 1);
      mbar_init(&empty[st], 1);
    }
    mbar_init(&sfull, 1);
    for (int j = 0; j < 2; ++j) {
      mbar_init(&accf[j], 1);
      mbar_init(&acce[j], 8);  // one arrival per epilogue warp
    }
    s_fail = 0;
    s_issued = 0;
    s_mmas = 0;
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&tmem_base, kTCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  if (warp == 0) {
    if (lane == 0) {
      // ---- copies: the shared rows, then (Z_h, B_h) per head -----------------
      mbar_arrive_expect_tx(&sfull, kSBytes);
      for (int c = 0; c < NSB; ++c) tma_load_3d(s_rows + c * 128 * 128, &maps.s, 64 * c, pos0, b, &sfull);
      for (int i = 0; i < nh; ++i) {
        const int st = i % kKtStages;
        if (i >= kKtStages &&
            !mbar_wait_bounded(&empty[st], static_cast<uint32_t>(i / kKtStages - 1) & 1u)) {
          s_fail = 1;
          break;
        }
        unsigned char* zs = ring + st * (kKtZBytes + kKtBBytes);
        mbar_arrive_expect_tx(&full[st], kKtZBytes + DH * 128);
        tma_load_4d(zs, &maps.z, 0, h0 + i, pos0, b, &full[st]);
        tma_load_3d(zs + kKtZBytes, &maps.b, 0, 0, h0 + i, &full[st]);
        s_issued = i + 1;
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---- MMAs: head i into accumulator i & 1 ---------------------------------
      constexpr uint32_t idesc = idesc_bf16(128, DH, 0, 0);
      for (int i = 0; i < nh; ++i) {
        const int st = i % kKtStages, j = i & 1;
        if (*reinterpret_cast<volatile int*>(&s_fail) ||
            !mbar_wait_bounded(&full[st], static_cast<uint32_t>(i / kKtStages) & 1u) ||
            (i >= 2 && !mbar_wait_bounded(&acce[j], static_cast<uint32_t>(i / 2 - 1) & 1u))) {
          s_fail = 1;
          break;
        }
        tc_fence_after();
        const uint32_t za = smem_u32(ring + st * (kKtZBytes + kKtBBytes));
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t ad = smem_desc(za + kk * 32, 16, 1024, 2);
          const uint64_t bd = smem_desc(za + kKtZBytes + kk * 32, 16, 1024, 2);
          tc_mma_ss(tmem + j * DH, ad, bd, idesc, kk > 0 ? 1u : 0u);
        }
        tc_commit(&empty[st]);
        tc_commit(&accf[j]);
        s_mmas = i + 1;
      }
    }
  } else {
    // ---- epilogue: token (TMEM lane) 32 q + lane of the tile, q = warp % 4;
    // columns [half DH / 2, (half + 1) DH / 2) ----------------------------------
    const int q = warp & 3, half = (warp - 2) >> 2, row = 32 * q + lane;
    const int t = t0 + row, pos = pos0 + row;
    const bool live = t < p.n_new && pos >= 0 && pos < p.max_len;
    bool ok = mbar_wait_bounded(&sfull, 0u);
    for (int i = 0; i < nh; ++i) {
      const int j = i & 1;
      float ss = 0.f;
      if (ok && !*reinterpret_cast<volatile int*>(&s_fail)) {
        ok = mbar_wait_bounded(&accf[j], static_cast<uint32_t>(i / 2) & 1u);
        if (ok) {
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < DH / 64; ++cc) {
            const int c = half * (DH / 64) + cc;  // 32-column chunk
            uint32_t v[32];
            tmem_ld32(tmem + (static_cast<uint32_t>(32 * q) << 16) + j * DH + 32 * c, v);
            tmem_wait_ld();
            // shared row columns 32 c .. 32 c + 31: four 16-byte chunks of box
            // (32 c) / 64, chunk index XORed with the row's low bits
            const unsigned char* sb = s_rows + ((32 * c) >> 6) * 128 * 128 + row * 128;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int chunk = (((32 * c) & 63) >> 3) + u;
              const uint4 w = *reinterpret_cast<const uint4*>(sb + ((chunk ^ (row & 7)) << 4));
              const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                const float k0 = __uint_as_float(v[8 * u + 2 * e]) + bf_lo(ww[e]);
                const float k1 = __uint_as_float(v[8 * u + 2 * e + 1]) + bf_hi(ww[e]);
                ss = fmaf(k0, k0, fmaf(k1, k1, ss));
              }
            }
          }
          tc_fence_before();
        } else {
          s_fail = 1;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_cta(&acce[j]);
      // the halves meet: the second writes, the first adds and stores (the
      // buffer of accumulator j is written again only two heads later, after
      // the next barrier, by when the first half has read it)
      if (half == 1) s_half[j][row] = ok ? ss : __int_as_float(0x7fc00000);
      asm volatile("bar.sync 1, 256;" ::: "memory");
      if (half == 0 && live)
        p.key_scale[(static_cast<size_t>(b) * p.H + h0 + i) * p.max_len + pos] =
            ok ? 1.f / sqrtf((ss + s_half[j][row]) / DH + p.eps) : __int_as_float(0x7fc00000);
    }
  }
  // every copy and MMA issued must be complete before the block releases its
  // shared memory and tensor memory (bounded waits: the full bound)
  __syncthreads();
  if (threadIdx.x == 0) {
    // the last copy issued into each stage, the shared rows, the last MMAs
    // committed into each accumulator
    for (int i = max(0, s_issued - kKtStages); i < s_issued; ++i)
      mbar_wait_bounded(&full[i % kKtStages], static_cast<uint32_t>(i / kKtStages) & 1u);
    mbar_wait_bounded(&sfull, 0u);
    for (int i = max(0, s_mmas - 2); i < s_mmas; ++i)
      mbar_wait_bounded(&accf[i & 1], static_cast<uint32_t>(i / 2) & 1u);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTCols);
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
  // the tensor-core form where it applies (LRKV_KEY_SCALE_TC=0: tuning, the
  // mma.sync form everywhere)
  const char* tc_env = std::getenv("LRKV_KEY_SCALE_TC");
  const bool tc_ok = !(tc_env && *tc_env && std::atoi(tc_env) == 0) &&
                     (dm.head_dim == 64 || dm.head_dim == 128) && dm.rank >= 8 && dm.rank <= 64 &&
                     dm.rank % 8 == 0 && a16(k_s) && a16(z_k) && a16(b_k);
  if (tc_ok) {
    KtMaps m;
    std::memset(&m, 0, sizeof(m));
    const uint64_t r = dm.rank, H = dm.heads, L = dm.max_len, Bq = dm.batch, dh = dm.head_dim;
    const uint64_t zd[4] = {r, H, L, Bq};
    const uint64_t zst[3] = {r * 2, H * r * 2, L * H * r * 2};
    const uint32_t zbox[4] = {64u, 1u, 128u, 1u};
    if (!make_tmap_4d_bf16_swizzled(&m.z, z_k, zd, zst, zbox) ||
        !make_tmap_3d_bf16(&m.b, b_k, r, dh, H, 64u, static_cast<uint32_t>(dh), CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_tmap_3d_bf16(&m.s, k_s, dh, L, Bq, 64u, 128u, CU_TENSOR_MAP_SWIZZLE_128B))
      return LRKV_ERR_CUDA;
    using TcFn = void (*)(const KeyScaleParams, const KtMaps);
    const TcFn kern = dm.head_dim == 128 ? lrkv_key_scale_tc_kernel<128> : lrkv_key_scale_tc_kernel<64>;
    const int smem = 1024 + (dm.head_dim / 64) * 128 * 128 + kKtStages * (kKtZBytes + kKtBBytes);
    if (ensure_kernel_smem(reinterpret_cast<const void*>(kern), smem, true) != cudaSuccess) return LRKV_ERR_CUDA;
    const dim3 grid((n_new + 127) / 128, (dm.heads + kKtHeads - 1) / kKtHeads, dm.batch);
    kern<<<grid, kKtThreads, smem, static_cast<cudaStream_t>(stream)>>>(p, m);
    return cudaGetLastError() == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
  }
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
