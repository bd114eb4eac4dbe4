// decode_step.cu — one decode step of an attention layer: the new token's
// cache rows from its layer input x ("Low-Rank Key Value Attention | What a
// shared cache can preserve", §3, Algorithm 1, for one token; "Low-Rank Key
// Value Attention：中文研读笔记", §2.3), then attention over the cache that
// now holds them (Algorithm 2).  Two programmatically dependent launches:
// this kernel writes the rows, the decode scan waits for it before it reads
// the cache (its set-up overlaps this kernel).
//
// For a batch of one-token steps the projection is a matrix-vector product
// per sequence, bound by reading the weights once: one warp per output
// column (grid-stride), the weight row streamed with 16-byte loads, the batch's
// x rows in shared memory, fp32 accumulation, bf16 (round to nearest even)
// stores at cache row seq_lens[b] - 1.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdlib>
#include <cstdint>

#include "host_cache.h"
#include "lrkv.h"
#include "ptx.cuh"

namespace lrkv {

namespace {

constexpr int kStepThreads = 256;
constexpr int kStepWarps = kStepThreads / 32;
constexpr int kStepSmem = 200 * 1024;      // x rows of one pass + the warps' first weight rows
constexpr int kStepWRows = 64 * 1024;      // weight rows staged when 8 of them fit here

struct StepParams {
  int B, H, dh, r, d, max_len, bc;
  int wstage;                              // the warps' first weight rows staged in shared memory
  const __nv_bfloat16* x;                  // [B][d]
  const __nv_bfloat16* w_sk;               // [dh][d]
  const __nv_bfloat16* w_sv;               // [dh][d]
  const __nv_bfloat16* u_k;                // [H r][d]
  const __nv_bfloat16* u_v;                // [H r][d]
  const int32_t* seq_lens;                 // [B], rows [0, seq_lens[b]) incl. the new one
  __nv_bfloat16 *k_s, *v_s, *z_k, *z_v;
  // paged cache: row t of sequence b is row t & (2^page_shift - 1) of page
  // block_table[b][t >> page_shift]; NULL: [B][max_len]
  const int32_t* block_table;
  int max_blocks, page_shift, num_pages;
};

__device__ __forceinline__ float dot8(const uint4 w, const uint4 x, float acc) {
  acc = fmaf(bf_lo(w.x), bf_lo(x.x), acc); acc = fmaf(bf_hi(w.x), bf_hi(x.x), acc);
  acc = fmaf(bf_lo(w.y), bf_lo(x.y), acc); acc = fmaf(bf_hi(w.y), bf_hi(x.y), acc);
  acc = fmaf(bf_lo(w.z), bf_lo(x.z), acc); acc = fmaf(bf_hi(w.z), bf_hi(x.z), acc);
  acc = fmaf(bf_lo(w.w), bf_lo(x.w), acc); acc = fmaf(bf_hi(w.w), bf_hi(x.w), acc);
  return acc;
}

__device__ __forceinline__ void cp_async16(void* smem_dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(smem_dst)), "l"(src) : "memory");
}

// Warp sums of M values per lane (M a power of two <= 32) by halving
// exchanges: after log2(M) steps each lane holds one partially summed value,
// whose index is given by the lane bits 16, 8, ...; the remaining lane bits
// are summed by xor shuffles.  Returns the full sum of value `idx` (every
// lane holds one; the lanes with the same idx hold the same sum).
template <int M>
__device__ __forceinline__ float warp_sums(float (&v)[M], int lane, int& idx) {
  int off = 16;
  idx = 0;
#pragma unroll
  for (int half = M / 2; half >= 1; half /= 2) {
    const bool up = (lane & off) != 0;
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float send = up ? v[i] : v[i + half];
      const float keep = up ? v[i + half] : v[i];
      v[i] = keep + __shfl_xor_sync(0xffffffffu, send, off);
    }
    if (up) idx += half;
    off >>= 1;
  }
  float s = v[0];
  for (; off >= 1; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  return s;
}

}  // namespace

// M: sequences per pass over the weights (8 or 16)
template <int M>
__global__ void __launch_bounds__(kStepThreads) lrkv_append_token_kernel(const StepParams p) {
  extern __shared__ __align__(16) unsigned char sx_raw[];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = gridDim.x * kStepWarps, gw = blockIdx.x * kStepWarps + warp;
  const int HR = p.H * p.r, N = 2 * p.dh + 2 * HR;
  const int chunks = p.d / 8;  // 16-byte chunks per row
  uint4* xs = reinterpret_cast<uint4*>(sx_raw);                    // [bc][chunks]
  uint4* wsm = xs + static_cast<size_t>(p.bc) * chunks + warp * chunks;  // this warp's first row
  auto weight_row = [&](int n) {
    return n < p.dh ? p.w_sk + static_cast<size_t>(n) * p.d
           : n < 2 * p.dh ? p.w_sv + static_cast<size_t>(n - p.dh) * p.d
           : n < 2 * p.dh + HR ? p.u_k + static_cast<size_t>(n - 2 * p.dh) * p.d
                               : p.u_v + static_cast<size_t>(n - 2 * p.dh - HR) * p.d;
  };
  // The weights are inputs of the call (no launch before writes them): the
  // warp's first column's row is copied into shared memory while the launch
  // before finishes, and its later columns start moving into L2 (a prefetch
  // reads nothing that could be stale: L2 is coherent).
  const bool staged = p.wstage && gw < N;
  if (staged) {
    const uint4* wv = reinterpret_cast<const uint4*>(weight_row(gw));
    for (int c = lane; c < chunks; c += 32) cp_async16(wsm + c, wv + c);
  }
  asm volatile("cp.async.commit_group;" ::: "memory");
  for (int n = gw + (staged ? nwarps : 0); n < N; n += nwarps) {
    const char* row = reinterpret_cast<const char*>(weight_row(n));
    for (int off = lane * 128; off < p.d * 2; off += 32 * 128)
      asm volatile("prefetch.global.L2 [%0];" ::"l"(row + off));
  }
  // x may come from the launch before: wait for it; only then may the decode
  // scan launch (its set-up reads q and the lengths, which the launch before
  // may also write; it waits for this grid before it reads the cache)
  pdl_wait();
  pdl_trigger();
  asm volatile("cp.async.wait_group 0;" ::: "memory");
  for (int b0 = 0; b0 < p.B; b0 += p.bc) {
    const int nb = min(p.bc, p.B - b0);
    __syncthreads();  // the previous pass is done with xs (first pass: the staged rows are in)
    const uint4* xg = reinterpret_cast<const uint4*>(p.x) + static_cast<size_t>(b0) * chunks;
    for (int i = tid; i < nb * chunks; i += blockDim.x) xs[i] = xg[i];
    __syncthreads();
    for (int n = gw; n < N; n += nwarps) {
      const uint4* wv = (staged && n == gw) ? wsm : reinterpret_cast<const uint4*>(weight_row(n));
      float acc[M];
#pragma unroll
      for (int b = 0; b < M; ++b) acc[b] = 0.f;
      for (int c = lane; c < chunks; c += 32) {
        const uint4 w = wv[c];
#pragma unroll
        for (int b = 0; b < M; ++b)
          if (b < nb) acc[b] = dot8(w, xs[b * chunks + c], acc[b]);
      }
      int idx;
      const float tot = warp_sums<M>(acc, lane, idx);  // sequence b0 + idx
      if ((lane & (32 / M - 1)) == 0 && idx < nb) {
        const int b = b0 + idx;
        const int pos = p.seq_lens[b] - 1;  // the new token's row (lengths out of range: no row;
                                            // the decode flags them)
        int pg = b, rw = pos;  // pool page (or sequence) and row of the new token
        if (p.block_table && pos >= 0 && pos < p.max_len) {
          pg = p.block_table[static_cast<size_t>(b) * p.max_blocks + (pos >> p.page_shift)];
          rw = pos & ((1 << p.page_shift) - 1);
        }
        // lengths out of range, or a page outside the pool: no row (the decode flags both)
        if (pos >= 0 && pos < p.max_len && (!p.block_table || (pg >= 0 && pg < p.num_pages))) {
          const size_t row = p.block_table ? (static_cast<size_t>(pg) << p.page_shift) + rw
                                           : static_cast<size_t>(b) * p.max_len + pos;
          __nv_bfloat16* dst = n < p.dh ? p.k_s + row * p.dh + n
                               : n < 2 * p.dh ? p.v_s + row * p.dh + (n - p.dh)
                               : n < 2 * p.dh + HR ? p.z_k + row * HR + (n - 2 * p.dh)
                                                   : p.z_v + row * HR + (n - 2 * p.dh - HR);
          *dst = __float2bfloat16_rn(tot);
        }
      }
    }
  }
}

// Host launch of the token rows (programmatic dependent launch after the
// caller's previous work).  Checks were done by the caller.
lrkv_status step_append_launch(const lrkv_dims& dm, int d_model, const void* x, const void* w_sk,
                               const void* w_sv, const void* u_k, const void* u_v, const int32_t* seq_lens,
                               void* k_s, void* v_s, void* z_k, void* z_v, int num_sms, void* stream,
                               const int32_t* block_table, int page_size, int num_pages) {
  StepParams p;
  p.block_table = block_table;
  p.max_blocks = block_table ? dm.max_len / page_size : 0;
  p.page_shift = 0;
  while (block_table && (1 << p.page_shift) < page_size) ++p.page_shift;
  p.num_pages = num_pages;
  p.B = dm.batch; p.H = dm.heads; p.dh = dm.head_dim; p.r = dm.rank; p.d = d_model; p.max_len = dm.max_len;
  const long long row_bytes = static_cast<long long>(d_model) * 2;
  const int M = dm.batch > 8 ? 16 : 8;
  p.wstage = kStepWarps * row_bytes <= kStepWRows;
  const long long x_budget = kStepSmem - (p.wstage ? kStepWarps * row_bytes : 0);
  p.bc = static_cast<int>(std::min<long long>(std::min(M, dm.batch), x_budget / row_bytes));
  if (p.bc < 1) return LRKV_ERR_UNSUPPORTED;
  p.x = static_cast<const __nv_bfloat16*>(x);
  p.w_sk = static_cast<const __nv_bfloat16*>(w_sk); p.w_sv = static_cast<const __nv_bfloat16*>(w_sv);
  p.u_k = static_cast<const __nv_bfloat16*>(u_k); p.u_v = static_cast<const __nv_bfloat16*>(u_v);
  p.seq_lens = seq_lens;
  p.k_s = static_cast<__nv_bfloat16*>(k_s); p.v_s = static_cast<__nv_bfloat16*>(v_s);
  p.z_k = static_cast<__nv_bfloat16*>(z_k); p.z_v = static_cast<__nv_bfloat16*>(z_v);
  const int smem = static_cast<int>((p.bc + (p.wstage ? kStepWarps : 0)) * row_bytes);
  auto kern = M == 8 ? lrkv_append_token_kernel<8> : lrkv_append_token_kernel<16>;
  // the largest shared-memory carveout, as the scan after it asks for (no
  // reconfiguration of the SMs between the two launches)
  if (ensure_kernel_smem(reinterpret_cast<const void*>(kern), smem, true) != cudaSuccess) return LRKV_ERR_CUDA;
  // one warp per output column, at most one CTA per SM
  const long long N = 2ll * dm.head_dim + 2ll * dm.heads * dm.rank;
  const long long wpc = kStepWarps;
  const char* cap_env = std::getenv("LRKV_STEP_GRID");  // tuning: at most this many CTAs
  const long long cap = (cap_env && *cap_env) ? std::max(1, std::atoi(cap_env)) : num_sms;
  const int grid = static_cast<int>(std::max<long long>(1, std::min<long long>(std::min<long long>(num_sms, cap),
                                                                               (N + wpc - 1) / wpc)));
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kStepThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p) == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

}  // namespace lrkv
