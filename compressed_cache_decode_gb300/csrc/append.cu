// append.cu — build factored-cache rows from layer activations on the
// tensor cores (tcgen05 + TMEM, sm_103a).
//
// Algorithm 1 of "Low-Rank Key Value Attention | What a shared cache can
// preserve" (§3): S_K = X W_sK, S_V = X W_sV once for all heads, and per head
// R_K[h] = X U_K[h], R_V[h] = X U_V[h], appended at the tokens' own rows
// ("Low-Rank Key Value Attention：中文研读笔记", §2.3).  All four products share
// X, so they run as one GEMM  C[M, N] = X[M, d] W_cat[N, d]^T  with
// N = 2 d_h + 2 H r, and the epilogue scatters each column range into its
// cache tensor at row start_pos[b] + t of sequence b.
//
// Tile 256 x 256, K step 64 (one 128-byte swizzle atom of bf16): two M = 128
// MMAs per K step share the B tile, into two accumulators of 256 TMEM
// columns each (all 512), so that a K step moves 64 KB of operands for
// 256 x 256 outputs (a 128 x 256 tile moved 48 KB for half as many; it ran
// the tensor pipe 56% busy, its 4-stage ring covering ~1.3 us of load
// latency).  Warp 0 issues TMA loads into a 3-stage ring, warp 1 issues the
// MMAs (one thread) and frees each stage with tcgen05.commit; then all four
// warps read the accumulators back (tcgen05.ld), round to bf16 and store.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstring>

#include "lrkv.h"
#include "trace.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lrkv {

namespace {

constexpr int kBM = 256, kBN = 256, kBK = 64, kStages = 3;
constexpr int kABytes = kBM * kBK * 2;   // 32 KB (two 128-row halves)
constexpr int kBBytes = kBN * kBK * 2;   // 32 KB
constexpr int kSub = 64;                 // rows of one weight box
constexpr uint32_t kStatusBounds = 2u;

struct AppendParams {
  int M, N, K;            // rows (B * n_new), columns (2 dh + 2 H r), depth (d_model)
  int n_new, max_len, dh, hr;
  const int32_t* start_pos;
  // paged cache: row t of sequence b is row t & (2^page_shift - 1) of page
  // block_table[b][t >> page_shift] of pools [num_pages][2^page_shift]; NULL: [B][max_len]
  const int32_t* block_table;
  int max_blocks, page_shift, num_pages;
  __nv_bfloat16* k_s;
  __nv_bfloat16* v_s;
  __nv_bfloat16* z_k;
  __nv_bfloat16* z_v;
  uint32_t* status;
};

struct AppendMaps {
  CUtensorMap x;
  CUtensorMap w[4];
};

}  // namespace

__global__ void __launch_bounds__(128, 1)
    lrkv_append_gemm_kernel(const AppendParams p, const __grid_constant__ AppendMaps maps) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ uint64_t full[kStages], empty[kStages], done;
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* a_st = smem;                         // kStages x 16 KB
  unsigned char* b_st = smem + kStages * kABytes;     // kStages x 32 KB

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n0 = blockIdx.x * kBN, m0 = blockIdx.y * kBM;
  const int kblocks = (p.K + kBK - 1) / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(&done, 1);
    s_fail = 0;
    fence_barrier_init();
  }
  if (warp == 0) tmem_alloc(&tmem_base, 2 * kBN);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;

  // segment boundaries of W_cat rows
  const int seg_end[4] = {p.dh, 2 * p.dh, 2 * p.dh + p.hr, 2 * p.dh + 2 * p.hr};
  const int seg_beg[4] = {0, p.dh, 2 * p.dh, 2 * p.dh + p.hr};

  if (warp == 0 && lane == 0) {
    // ---- producer: TMA ring ------------------------------------------------
    int nsub = 0;
    for (int j = 0; j < kBN / kSub; ++j)
      if (n0 + j * kSub < p.N) ++nsub;
    const uint32_t bytes = kABytes + nsub * kSub * kBK * 2;
    for (int kb = 0; kb < kblocks; ++kb) {
      const int s = kb % kStages;
      if (kb >= kStages && !mbar_wait_bounded(&empty[s], static_cast<uint32_t>(kb / kStages - 1) & 1u)) {
        s_fail = 1;
        break;
      }
      mbar_arrive_expect_tx(&full[s], bytes);
      tma_load_3d(a_st + s * kABytes, &maps.x, kb * kBK, m0, 0, &full[s]);
      for (int j = 0; j < nsub; ++j) {
        const int row = n0 + j * kSub;
        int seg = 0;
        while (seg < 3 && row >= seg_end[seg]) ++seg;
        tma_load_3d(b_st + s * kBBytes + j * kSub * kBK * 2, &maps.w[seg], kb * kBK, row - seg_beg[seg], 0,
                    &full[s]);
      }
    }
  } else if (warp == 1 && lane == 0) {
    // ---- MMA issuer ----------------------------------------------------------
    constexpr uint32_t idesc = idesc_bf16(128, kBN, 0, 0);
    bool ok = true;
    for (int kb = 0; kb < kblocks && ok; ++kb) {
      const int s = kb % kStages;
      if (!mbar_wait_bounded(&full[s], static_cast<uint32_t>(kb / kStages) & 1u)) {
        ok = false;
        s_fail = 1;
        break;
      }
      tc_fence_after();
      const uint32_t a0 = smem_u32(a_st + s * kABytes), b0 = smem_u32(b_st + s * kBBytes);
#pragma unroll
      for (int kk = 0; kk < kBK / 16; ++kk) {
        const uint64_t bd = smem_desc(b0 + kk * 32, 16, 1024, 2);
#pragma unroll
        for (int half = 0; half < 2; ++half) {  // rows 128 half .. 128 half + 127 into columns 256 half ..
          const uint64_t ad = smem_desc(a0 + half * (128 * 128) + kk * 32, 16, 1024, 2);
          tc_mma_ss(tmem + half * kBN, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
        }
      }
      tc_commit(&empty[s]);
    }
    tc_commit(&done);
  }

  // ---- epilogue: TMEM -> registers -> bf16 cache rows ----------------------
  __syncwarp();
  const bool got = mbar_wait_bounded(&done, 0u);
  tc_fence_after();
  if (!got || s_fail) {
    if (threadIdx.x == 0) atomicOr(p.status, 1u);
  } else {
    for (int half = 0; half < 2; ++half) {
    const int m = m0 + half * 128 + warp * 32 + lane;  // this thread's output row
    size_t crow = 0;
    bool row_ok = m < p.M;
    if (row_ok) {
      const int b = m / p.n_new, t = m % p.n_new;
      const int pos = p.start_pos[b] + t;
      if (pos < 0 || pos >= p.max_len) {
        row_ok = false;
        atomicOr(p.status, kStatusBounds);
      } else if (!p.block_table) {
        crow = static_cast<size_t>(b) * p.max_len + pos;
      } else {
        const int pg = p.block_table[static_cast<size_t>(b) * p.max_blocks + (pos >> p.page_shift)];
        if (pg < 0 || pg >= p.num_pages) {  // no page of the pool: the row is not written
          row_ok = false;
          atomicOr(p.status, kStatusBounds);
        } else {
          crow = (static_cast<size_t>(pg) << p.page_shift) + (pos & ((1 << p.page_shift) - 1));
        }
      }
    }
    for (int c = 0; c < kBN / 32; ++c) {
      const int n = n0 + c * 32;
      uint32_t v[32];
      tmem_ld32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + half * kBN + c * 32, v);
      tmem_wait_ld();
      if (!row_ok || n >= p.N) continue;
      int seg = 0;
      while (seg < 3 && n >= seg_end[seg]) ++seg;
      __nv_bfloat16* base = seg == 0 ? p.k_s : seg == 1 ? p.v_s : seg == 2 ? p.z_k : p.z_v;
      const int width = seg < 2 ? p.dh : p.hr;
      uint4* dst = reinterpret_cast<uint4*>(base + crow * width + (n - seg_beg[seg]));
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 w;
        uint32_t* wp = reinterpret_cast<uint32_t*>(&w);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(v[q * 8 + 2 * e]),
                                                          __uint_as_float(v[q * 8 + 2 * e + 1]));
          wp[e] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        dst[q] = w;
      }
    }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, 2 * kBN);
}

}  // namespace lrkv

namespace {

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool make_map_2d(CUtensorMap* map, const void* base, uint64_t inner, uint64_t rows, uint32_t box_inner,
                 uint32_t box_rows) {
  // a 2-D bf16 map as a 3-D one with a unit outer dimension
  return lrkv::make_tmap_3d_bf16(map, base, inner, rows, 1, box_inner, box_rows, CU_TENSOR_MAP_SWIZZLE_128B);
}

}  // namespace

static lrkv_status append_impl(const lrkv_dims* dims, int d_model, int n_new, const void* x, const void* w_sk,
                               const void* w_sv, const void* u_k, const void* u_v, const int32_t* start_pos,
                               const int32_t* block_table, int page_size, int num_pages, void* k_s, void* v_s,
                               void* z_k, void* z_v, void* ws, size_t ws_bytes, lrkv_stream_t stream) {
  if (!dims) return LRKV_ERR_INVALID_ARG;
  const lrkv_dims& d = *dims;
  if (d.batch < 1 || d.heads < 1 || d.head_dim < 1 || d.rank < 0 || d.max_len < 1 || d_model < 1 || n_new < 1)
    return LRKV_ERR_INVALID_ARG;
  if (d.dtype != LRKV_BF16 && d.dtype != LRKV_F32) return LRKV_ERR_INVALID_ARG;
  if (d.dtype != LRKV_BF16) return LRKV_ERR_UNSUPPORTED;
  const int hr = d.heads * d.rank;
  if (d_model % 64 != 0 || d.head_dim % 64 != 0 || hr % 64 != 0) return LRKV_ERR_UNSUPPORTED;
  if (static_cast<long long>(d.batch) * n_new > (1LL << 31) - 1) return LRKV_ERR_UNSUPPORTED;
  if (!x || !w_sk || !w_sv || !start_pos || !k_s || !v_s) return LRKV_ERR_INVALID_ARG;
  if (hr > 0 && (!u_k || !u_v || !z_k || !z_v)) return LRKV_ERR_INVALID_ARG;
  if (!a16(x) || !a16(w_sk) || !a16(w_sv) || !a16(k_s) || !a16(v_s)) return LRKV_ERR_INVALID_ARG;
  if (hr > 0 && (!a16(u_k) || !a16(u_v) || !a16(z_k) || !a16(z_v))) return LRKV_ERR_INVALID_ARG;
  if (!ws || ws_bytes < 16) return LRKV_ERR_WORKSPACE;

  lrkv::AppendParams p;
  p.M = d.batch * n_new;
  p.N = 2 * d.head_dim + 2 * hr;
  p.K = d_model;
  p.n_new = n_new;
  p.max_len = d.max_len;
  p.dh = d.head_dim;
  p.hr = hr;
  p.start_pos = start_pos;
  p.block_table = block_table;
  p.max_blocks = block_table ? d.max_len / page_size : 0;
  p.page_shift = 0;
  while (block_table && (1 << p.page_shift) < page_size) ++p.page_shift;
  p.num_pages = num_pages;
  p.k_s = static_cast<__nv_bfloat16*>(k_s);
  p.v_s = static_cast<__nv_bfloat16*>(v_s);
  p.z_k = static_cast<__nv_bfloat16*>(z_k);
  p.z_v = static_cast<__nv_bfloat16*>(z_v);
  p.status = static_cast<uint32_t*>(ws);

  lrkv::AppendMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  if (!make_map_2d(&maps.x, x, d_model, p.M, 64, lrkv::kBM) ||
      !make_map_2d(&maps.w[0], w_sk, d_model, d.head_dim, 64, 64) ||
      !make_map_2d(&maps.w[1], w_sv, d_model, d.head_dim, 64, 64))
    return LRKV_ERR_CUDA;
  if (hr > 0 && (!make_map_2d(&maps.w[2], u_k, d_model, hr, 64, 64) ||
                 !make_map_2d(&maps.w[3], u_v, d_model, hr, 64, 64)))
    return LRKV_ERR_CUDA;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, 4, s) != cudaSuccess) return LRKV_ERR_CUDA;
  const int smem = lrkv::kStages * (lrkv::kABytes + lrkv::kBBytes) + 1024;
  if (cudaFuncSetAttribute(lrkv::lrkv_append_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
      cudaSuccess)
    return LRKV_ERR_CUDA;
  const dim3 grid((p.N + lrkv::kBN - 1) / lrkv::kBN, (p.M + lrkv::kBM - 1) / lrkv::kBM);
  lrkv::lrkv_append_gemm_kernel<<<grid, 128, smem, s>>>(p, maps);
  return cudaGetLastError() == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

extern "C" lrkv_status lrkv_append(const lrkv_dims* dims, int d_model, int n_new, const void* x,
                                   const void* w_sk, const void* w_sv, const void* u_k, const void* u_v,
                                   const int32_t* start_pos, void* k_s, void* v_s, void* z_k, void* z_v,
                                   void* ws, size_t ws_bytes, lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_append");
  return append_impl(dims, d_model, n_new, x, w_sk, w_sv, u_k, u_v, start_pos, nullptr, 0, 0, k_s, v_s, z_k, z_v,
                     ws, ws_bytes, stream);
}

extern "C" lrkv_status lrkv_append_paged(const lrkv_dims* dims, int d_model, int n_new, const void* x,
                                         const void* w_sk, const void* w_sv, const void* u_k, const void* u_v,
                                         const int32_t* start_pos, int page_size, int num_pages,
                                         const int32_t* block_table, void* k_s, void* v_s, void* z_k, void* z_v,
                                         void* ws, size_t ws_bytes, lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_append_paged");
  if (!dims || !block_table) return LRKV_ERR_INVALID_ARG;
  if (page_size < 16 || (page_size & (page_size - 1)) != 0 || num_pages < 1) return LRKV_ERR_INVALID_ARG;
  if (dims->max_len % page_size != 0) return LRKV_ERR_INVALID_ARG;
  if (static_cast<long long>(num_pages) * page_size > (1LL << 31) - 1) return LRKV_ERR_UNSUPPORTED;
  return append_impl(dims, d_model, n_new, x, w_sk, w_sv, u_k, u_v, start_pos, block_table, page_size, num_pages,
                     k_s, v_s, z_k, z_v, ws, ws_bytes, stream);
}
