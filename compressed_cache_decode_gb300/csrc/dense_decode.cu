// dense_decode.cu — the comparison decode on the same box: attention over
// materialised K/V with grouped heads (MHA, GQA, MQA), so that the factored
// cache's decode can be measured against the layouts it replaces ("Low-Rank
// Key Value Attention | What a shared cache can preserve", §4 "Weight count
// and the two decode regimes" and §5, which asks for optimized GQA and MHA
// at the same batch, length and dtype).
//
// K, V [B][max_len][H_kv][d] bf16; query head h reads KV head h / (H / H_kv).
// Grid (range CTAs, groups of up to 8 KV heads); one warp per KV head, its
// group's query heads (up to 8) are the N columns of the tensor-core
// products (bf16 mma.sync, fp32 accumulation):
//   S^T = K q^T (tokens x query heads), ONE online softmax per query head,
//   O^T += V^T P^T (rows of the head dim), the probabilities transposed in
//   registers (movmatrix) into the B operand.
// 16-token tiles of the group's K and V stream through a ring of shared-memory
// stages (TMA; each head's 16 rows land contiguously with the 128-byte
// swizzle: conflict-free ldmatrix); every warp consumes every stage and the
// last of them to finish refills it.  Each (piece, query head) leaves a
// partial in the workspace layout of the LRKV decode at rank 0, and the same
// merge finishes.
#include <cuda.h>
#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstring>

#include "decode_common.cuh"
#include "decode_plan.h"
#include "host_cache.h"
#include "lrkv.h"
#include "trace.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lrkv {

using namespace dec;

namespace {

constexpr int kDT = 16;         // tokens per tile
constexpr int kDMaxWarps = 8;   // KV heads per CTA (one warp each)
constexpr int kDHeader = 1024;  // barriers and stage records
constexpr int kDMaxStages = 16;
constexpr float kDRescaleLog2 = 8.f;  // raise the reference max only past 2^8

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

}  // namespace

// D: head dim; NG: query heads per KV head (<= 8, the useful MMA columns).
template <int D, int NG>
__global__ void __launch_bounds__(32 * kDMaxWarps, 1)
    lrkv_dense_decode_kernel(const __grid_constant__ DecodePlan P, const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v) {
  constexpr int KS = D / 16;       // 16-wide head-dim steps
  constexpr int NB = D / 64;       // 64-column boxes per row
  constexpr int KB = KS > 4 ? 4 : KS;
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_timeout;
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  pdl_trigger();  // the merge may launch: it waits for this grid before it reads
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int g = lane >> 2, q4 = lane & 3;
  const int B = P.B, H = P.H;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  int* cons = reinterpret_cast<int*>(smem + 128);
  int* issued = reinterpret_cast<int*>(smem + 256);
  int* pre = reinterpret_cast<int*>(smem + kDHeader);

  if (tid == 0) {
    s_timeout = 0;
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(&full[s], 1);
      cons[s] = 0;
      issued[s] = -1;
    }
    fence_barrier_init();
  }
  int bad = 0;
  for (int b = tid; b < B; b += blockDim.x) {
    int L = P.seq_lens[b];
    if (L < 0 || L > P.max_len) {
      bad = 1;
      L = min(max(L, 0), P.max_len);
    }
    pre[b + 1] = L;
  }
  if (tid == 0) pre[0] = 0;
  bad = __syncthreads_or(bad);
  if (warp == 0) {
    int carry = 0;
    for (int base = 1; base <= B; base += 32) {
      const int i = base + lane;
      int v = (i <= B) ? pre[i] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (i <= B) pre[i] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
  const int N = pre[B];
  const int G = max(1, min(static_cast<int>(gridDim.x), (N + P.min_tokens - 1) / max(P.min_tokens, 1)));
  uint32_t* cta_status = P.cta_status + blockIdx.y * gridDim.x + blockIdx.x;
  if (N == 0 || static_cast<int>(blockIdx.x) >= G) {
    pdl_wait();  // the launch before may still read the workspace
    if (blockIdx.x == 0 && blockIdx.y == 0) {
      for (int b = tid; b <= B; b += blockDim.x) P.prefix[b] = pre[b];
      if (tid == 0) { P.meta[0] = N; P.meta[1] = G; }
    }
    if (tid == 0) *cta_status = bad ? kDevBounds : 0u;
    return;
  }
  const int c = blockIdx.x;
  const int g0 = static_cast<int>(static_cast<long long>(c) * N / G);
  const int g1 = static_cast<int>(static_cast<long long>(c + 1) * N / G);
  const int kvg = nwarps;                    // KV heads of this CTA
  const int hk0 = blockIdx.y * kvg;          // its first KV head
  const int box_bytes = kvg * kDT * 128;     // one 64-column box of the group

  auto issue = [&](int s, int j, const TileWalk& t) {
    unsigned char* ks = smem + P.off_kv + static_cast<size_t>(s) * P.stage_bytes;
    unsigned char* vs = ks + P.kv_bytes;
    mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(2 * P.kv_bytes));
#pragma unroll
    for (int cb = 0; cb < NB; ++cb) {
      tma_load_4d(ks + cb * box_bytes, &tm_k, cb * 64, t.t0, hk0, t.b, &full[s]);
      tma_load_4d(vs + cb * box_bytes, &tm_v, cb * 64, t.t0, hk0, t.b, &full[s]);
    }
    *reinterpret_cast<volatile int*>(&issued[s]) = j;
  };
  TileWalk ahead;
  bool ahead_more = walk_first(ahead, pre, B, g0, g1);
  for (int j = 0; j < P.stages && ahead_more; ++j) {
    if (tid == 0) issue(j, j, ahead);
    ahead_more = walk_next(ahead, pre, B, g1, kDT);
  }

  // ---- this warp: KV head hk, query heads h0 .. h0 + NG - 1 ----
  const int hk = hk0 + warp;
  const int h0 = hk * NG;
  // q as the B operand (k = head dim, n = query head g of the group; zero
  // for the columns past the group)
  uint32_t qb[KS][2];
#pragma unroll
  for (int kk = 0; kk < KS; ++kk) qb[kk][0] = qb[kk][1] = 0u;
  const int arow = lane & 15, ahalf = lane >> 4;
  const int trow = (lane & 7) + 8 * (lane >> 4), tcol = (lane >> 3) & 1;
  const int hoff = warp * kDT * 128;  // this head's rows inside a box

  float acc[KS][4];
  float mc[2], lc[2];
  TileWalk w;
  bool more = walk_first(w, pre, B, g0, g1);
  bool ok = true, waited = false;
  int cur_b = -1;

  auto write_partial = [&](int b) {
    if (!waited) {
      pdl_wait();  // the launch before may still read the workspace
      waited = true;
    }
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lc[0] += __shfl_xor_sync(0xffffffffu, lc[0], o);
      lc[1] += __shfl_xor_sync(0xffffffffu, lc[1], o);
    }
    const size_t slot = static_cast<size_t>(b + c);
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int n = 2 * q4 + e;
      if (n < NG) {
        const int h = h0 + n;
        if (g == 0) {
          float* pml = P.part_ml + (slot * H + h) * 2;
          pml[0] = mc[e];
          pml[1] = lc[e];
        }
        float* o = P.part_acc + (slot * H + h) * (D + P.r);
#pragma unroll
        for (int m = 0; m < KS; ++m) {
          o[16 * m + g] = acc[m][e];
          o[16 * m + g + 8] = acc[m][2 + e];
        }
      }
    }
  };

  for (int j = 0; more; ++j) {
    if (w.b != cur_b) {
      if (cur_b >= 0) write_partial(cur_b);
      cur_b = w.b;
      mc[0] = mc[1] = -INFINITY;
      lc[0] = lc[1] = 0.f;
#pragma unroll
      for (int m = 0; m < KS; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
      if (g < NG) {
        const __nv_bfloat16* qr = static_cast<const __nv_bfloat16*>(P.q) + (static_cast<size_t>(w.b) * H + h0 + g) * D;
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          qb[kk][0] = *reinterpret_cast<const uint32_t*>(qr + 16 * kk + 2 * q4);
          qb[kk][1] = *reinterpret_cast<const uint32_t*>(qr + 16 * kk + 2 * q4 + 8);
        }
      }
    }
    const int s = j % P.stages;
    const int nvalid = min(kDT, w.t_end - w.t0);
    if (ok && *reinterpret_cast<volatile int*>(&s_timeout)) ok = false;
    if (ok) {
      ok = mbar_wait_bounded(&full[s], static_cast<uint32_t>(j / P.stages) & 1u, P.wait_limit);
      if (!ok) *reinterpret_cast<volatile int*>(&s_timeout) = 1;
    }
    if (ok) {
      const unsigned char* ks = smem + P.off_kv + static_cast<size_t>(s) * P.stage_bytes;
      const unsigned char* vs = ks + P.kv_bytes;
      // scores S^T: rows tokens g / g + 8, columns query heads 2 q4 + e
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int k0 = 0; k0 < KS; k0 += KB) {
        uint32_t a[KB][4];
#pragma unroll
        for (int u = 0; u < KB; ++u) {
          const int ch = 2 * (k0 + u) + ahalf;  // 16-byte chunk along the head dim
          ldsm_x4(a[u][0], a[u][1], a[u][2], a[u][3],
                  ks + (ch >> 3) * box_bytes + hoff + swz_off(arow, ch & 7, 128));
        }
#pragma unroll
        for (int u = 0; u < KB; ++u)
          mma_bf16_16816(((k0 + u) & 1) ? sb : sa, a[u][0], a[u][1], a[u][2], a[u][3], qb[k0 + u][0],
                         qb[k0 + u][1]);
      }
      const bool v0 = g < nvalid, v1 = g + 8 < nvalid;
      float sc[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) sc[u] = (u < 2 ? v0 : v1) ? (sa[u] + sb[u]) * P.scale_log2 : -INFINITY;
      float mx[2] = {fmaxf(sc[0], sc[2]), fmaxf(sc[1], sc[3])};
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], o));
        mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], o));
      }
      const bool up = mx[0] > mc[0] + kDRescaleLog2 || mx[1] > mc[1] + kDRescaleLog2;
      if (__any_sync(0xffffffffu, up)) {
        float al[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float mn = mx[e] > mc[e] + kDRescaleLog2 ? mx[e] : mc[e];
          al[e] = mc[e] == -INFINITY ? 0.f : exp2f(mc[e] - mn);
          mc[e] = mn;
          lc[e] *= al[e];
        }
#pragma unroll
        for (int m = 0; m < KS; ++m) {
          acc[m][0] *= al[0]; acc[m][1] *= al[1]; acc[m][2] *= al[0]; acc[m][3] *= al[1];
        }
      }
      const float p0 = exp2f(sc[0] - mc[0]), p1 = exp2f(sc[1] - mc[1]);
      const float p2 = exp2f(sc[2] - mc[0]), p3 = exp2f(sc[3] - mc[1]);
      lc[0] += p0 + p2;
      lc[1] += p1 + p3;
      const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));  // tokens 0-7
      const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));  // tokens 8-15
      // rows past the history may hold anything: keep them out of the A operand
      auto valid = [&](int row) { return row < nvalid; };
      const uint32_t keep0 = (valid(2 * q4) ? 0x0000ffffu : 0u) | (valid(2 * q4 + 1) ? 0xffff0000u : 0u);
      const uint32_t keep1 = (valid(2 * q4 + 8) ? 0x0000ffffu : 0u) | (valid(2 * q4 + 9) ? 0xffff0000u : 0u);
#pragma unroll
      for (int n0 = 0; n0 < KS; n0 += KB) {
        uint32_t a[KB][4];
#pragma unroll
        for (int u = 0; u < KB; ++u) {
          const int ch = 2 * (n0 + u) + tcol;
          ldsm_x4_trans(a[u][0], a[u][1], a[u][2], a[u][3],
                        vs + (ch >> 3) * box_bytes + hoff + swz_off(trow, ch & 7, 128));
        }
#pragma unroll
        for (int u = 0; u < KB; ++u)
          mma_bf16_16816(acc[n0 + u], a[u][0] & keep0, a[u][1] & keep0, a[u][2] & keep1, a[u][3] & keep1, pb0,
                         pb1);
      }
      // the stage is free once every warp is done with it: the last to finish
      // refills it (a warp counts only after it saw the stage's copy land)
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        const bool last = (atomicAdd(&cons[s], 1) % nwarps) == nwarps - 1;
        __threadfence_block();
        if (last && ahead_more && !*reinterpret_cast<volatile int*>(&s_timeout)) {
          fence_proxy_async_smem();
          issue(s, j + P.stages, ahead);
        }
      }
      __syncwarp();
    }
    more = walk_next(w, pre, B, g1, kDT);
    if (ahead_more) ahead_more = walk_next(ahead, pre, B, g1, kDT);
  }
  if (cur_b >= 0) write_partial(cur_b);

  // ---- every copy this CTA issued has landed before it exits ----
  __syncthreads();
  if (tid == 0) {
    pdl_wait();
    bool drained = true;
    for (int st = 0; st < P.stages; ++st) {
      const int jj = *reinterpret_cast<volatile int*>(&issued[st]);
      if (jj >= 0) drained = mbar_wait_bounded(&full[st], static_cast<uint32_t>(jj / P.stages) & 1u) && drained;
    }
    if (!drained) *reinterpret_cast<volatile int*>(&s_timeout) = 1;
    if (blockIdx.x == 0 && blockIdx.y == 0) {
      P.meta[0] = N;
      P.meta[1] = G;
    }
    *cta_status = (bad ? kDevBounds : 0u) | (*reinterpret_cast<volatile int*>(&s_timeout) ? kDevTimeout : 0u);
  }
  if (blockIdx.x == 0 && blockIdx.y == 0) {
    pdl_wait();
    for (int b = tid; b <= B; b += blockDim.x) P.prefix[b] = pre[b];
  }
}

// ======================================================================== MLA
// Absorbed multi-head latent attention decode (review §5: a head computes
// (q_h A_h) Z^T without materialising its keys, the values likewise): one
// latent row c_j of width DC per token for all heads.
//   q_c,h = q_h W_uk[h]          (lrkv_mla_absorb_kernel, fp32, in the workspace)
//   s_{h,j} = q_c,h . c_j / sqrt(d_h), one softmax per head
//   o_c,h = sum_j a_{h,j} c_j    (this kernel; partials per (piece, head))
//   o_h = o_c,h W_uv[h]^T        (the merge's lift)
// Grid: range CTAs; 2 H / 8 warps: warp w takes query group w / 2 (8 heads,
// the N columns of the MMAs) and latent half w % 2 for the values; both warps
// of a group compute the group's scores (32 k steps, q_c as bf16 high + low
// parts from a conflict-free shared table).  16-token tiles of c stream
// through a ring (TMA, 128-byte swizzle); the last warp to finish a stage
// refills it.

__global__ void lrkv_mla_absorb_kernel(const DecodePlan P, const __nv_bfloat16* w_uk) {
  extern __shared__ float qs[];  // [d_h]
  const int h = blockIdx.x, b = blockIdx.y, dh = P.dh, dc = P.r;
  const __nv_bfloat16* q = static_cast<const __nv_bfloat16*>(P.q) + (static_cast<size_t>(b) * P.H + h) * dh;
  for (int d = threadIdx.x; d < dh; d += blockDim.x) qs[d] = __bfloat162float(q[d]);
  __syncthreads();
  const __nv_bfloat16* w = w_uk + static_cast<size_t>(h) * dh * dc;
  for (int cc = threadIdx.x; cc < dc; cc += blockDim.x) {
    float a = 0.f;
    for (int d = 0; d < dh; ++d) a = fmaf(qs[d], __bfloat162float(w[static_cast<size_t>(d) * dc + cc]), a);
    P.p_abs[(static_cast<size_t>(b) * P.H + h) * dc + cc] = a;
  }
}

template <int DC>
__global__ void __launch_bounds__(32 * kDMaxWarps, 1)
    lrkv_mla_decode_kernel(const __grid_constant__ DecodePlan P, const __grid_constant__ CUtensorMap tm_c) {
  constexpr int KS = DC / 16;     // 16-wide latent steps of the scores
  constexpr int NB = DC / 64;     // 64-column boxes per row
  constexpr int MH = DC / 32;     // 16-row value tiles per latent half
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_timeout;
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int g = lane >> 2, q4 = lane & 3;
  const int B = P.B, H = P.H;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  int* cons = reinterpret_cast<int*>(smem + 128);
  int* issued = reinterpret_cast<int*>(smem + 256);
  int* pre = reinterpret_cast<int*>(smem + kDHeader);
  uint4* qtab = reinterpret_cast<uint4*>(smem + P.off_pq);  // [group][KS][32] {hi b0, hi b1, lo b0, lo b1}

  if (tid == 0) {
    s_timeout = 0;
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(&full[s], 1);
      cons[s] = 0;
      issued[s] = -1;
    }
    fence_barrier_init();
  }
  int bad = 0;
  for (int b = tid; b < B; b += blockDim.x) {
    int L = P.seq_lens[b];
    if (L < 0 || L > P.max_len) {
      bad = 1;
      L = min(max(L, 0), P.max_len);
    }
    pre[b + 1] = L;
  }
  if (tid == 0) pre[0] = 0;
  bad = __syncthreads_or(bad);
  if (warp == 0) {
    int carry = 0;
    for (int base = 1; base <= B; base += 32) {
      const int i = base + lane;
      int v = (i <= B) ? pre[i] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
      }
      if (i <= B) pre[i] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  __syncthreads();
  const int N = pre[B];
  const int G = max(1, min(static_cast<int>(gridDim.x), (N + P.min_tokens - 1) / max(P.min_tokens, 1)));
  uint32_t* cta_status = P.cta_status + blockIdx.x;
  if (N == 0 || static_cast<int>(blockIdx.x) >= G) {
    pdl_wait();
    if (blockIdx.x == 0) {
      for (int b = tid; b <= B; b += blockDim.x) P.prefix[b] = pre[b];
      if (tid == 0) { P.meta[0] = N; P.meta[1] = G; }
    }
    if (tid == 0) *cta_status = bad ? kDevBounds : 0u;
    return;
  }
  const int c = blockIdx.x;
  const int g0 = static_cast<int>(static_cast<long long>(c) * N / G);
  const int g1 = static_cast<int>(static_cast<long long>(c + 1) * N / G);

  auto issue = [&](int s, int j, const TileWalk& t) {
    unsigned char* cs = smem + P.off_kv + static_cast<size_t>(s) * P.stage_bytes;
    mbar_arrive_expect_tx(&full[s], static_cast<uint32_t>(P.stage_bytes));
#pragma unroll
    for (int cb = 0; cb < NB; ++cb) tma_load_3d(cs + cb * kDT * 128, &tm_c, cb * 64, t.t0, t.b, &full[s]);
    *reinterpret_cast<volatile int*>(&issued[s]) = j;
  };
  // q_c is written by the launch before (the absorb): wait for it before the
  // first table is built (the first copies overlap the wait)
  TileWalk ahead;
  bool ahead_more = walk_first(ahead, pre, B, g0, g1);
  for (int j = 0; j < P.stages && ahead_more; ++j) {
    if (tid == 0) issue(j, j, ahead);
    ahead_more = walk_next(ahead, pre, B, g1, kDT);
  }
  pdl_wait();

  const int qg = warp >> 1, dhf = warp & 1;  // query group (8 heads), latent half of the values
  const int h0 = 8 * qg;
  const int arow = lane & 15, ahalf = lane >> 4;
  const int trow = (lane & 7) + 8 * (lane >> 4), tcol = (lane >> 3) & 1;
  uint4* qt = qtab + qg * KS * 32;
  float acc[MH][4];
  float mc[2], lc[2];
  TileWalk w;
  bool more = walk_first(w, pre, B, g0, g1);
  bool ok = true;
  int cur_b = -1;

  auto write_partial = [&](int b) {
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lc[0] += __shfl_xor_sync(0xffffffffu, lc[0], o);
      lc[1] += __shfl_xor_sync(0xffffffffu, lc[1], o);
    }
    const size_t slot = static_cast<size_t>(b + c);
    const int W = P.dh + DC;
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int h = h0 + 2 * q4 + e;
      float* o = P.part_acc + (slot * H + h) * W;
      if (dhf == 0) {
        if (g == 0) {
          float* pml = P.part_ml + (slot * H + h) * 2;
          pml[0] = mc[e];
          pml[1] = lc[e];
        }
        for (int i = g; i < P.dh; i += 8) o[i] = 0.f;  // no shared part: the merge lifts the latent sum
      }
#pragma unroll
      for (int m = 0; m < MH; ++m) {
        o[P.dh + 16 * (dhf * MH + m) + g] = acc[m][e];
        o[P.dh + 16 * (dhf * MH + m) + g + 8] = acc[m][2 + e];
      }
    }
  };

  for (int j = 0; more; ++j) {
    if (w.b != cur_b) {
      if (cur_b >= 0) write_partial(cur_b);
      cur_b = w.b;
      mc[0] = mc[1] = -INFINITY;
      lc[0] = lc[1] = 0.f;
#pragma unroll
      for (int m = 0; m < MH; ++m) acc[m][0] = acc[m][1] = acc[m][2] = acc[m][3] = 0.f;
      // the group's q table for this sequence (the two warps split the steps)
      named_bar_sync(1 + qg, 64);  // both warps are done with the previous table
      const float* qc = P.p_abs + (static_cast<size_t>(w.b) * H + h0 + g) * DC;
      for (int kk = dhf; kk < KS; kk += 2) {
        const int k0 = 16 * kk + 2 * q4;
        float v[4] = {qc[k0], qc[k0 + 1], qc[k0 + 8], qc[k0 + 9]};
        float hi[4], lo[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          hi[u] = __bfloat162float(__float2bfloat16_rn(v[u]));
          lo[u] = v[u] - hi[u];
        }
        qt[kk * 32 + lane] = make_uint4(pack_bf16x2(hi[0], hi[1]), pack_bf16x2(hi[2], hi[3]),
                                        pack_bf16x2(lo[0], lo[1]), pack_bf16x2(lo[2], lo[3]));
      }
      named_bar_sync(1 + qg, 64);  // the table is complete
    }
    const int s = j % P.stages;
    const int nvalid = min(kDT, w.t_end - w.t0);
    if (ok && *reinterpret_cast<volatile int*>(&s_timeout)) ok = false;
    if (ok) {
      ok = mbar_wait_bounded(&full[s], static_cast<uint32_t>(j / P.stages) & 1u, P.wait_limit);
      if (!ok) *reinterpret_cast<volatile int*>(&s_timeout) = 1;
    }
    if (ok) {
      const unsigned char* cs = smem + P.off_kv + static_cast<size_t>(s) * P.stage_bytes;
      float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
      float la[4] = {0.f, 0.f, 0.f, 0.f}, lb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
      for (int kk = 0; kk < KS; ++kk) {
        const int ch = 2 * kk + ahalf;
        uint32_t a0, a1, a2, a3;
        ldsm_x4(a0, a1, a2, a3, cs + (ch >> 3) * (kDT * 128) + swz_off(arow, ch & 7, 128));
        const uint4 f = qt[kk * 32 + lane];
        mma_bf16_16816((kk & 1) ? sb : sa, a0, a1, a2, a3, f.x, f.y);
        mma_bf16_16816((kk & 1) ? lb : la, a0, a1, a2, a3, f.z, f.w);
      }
      const bool v0 = g < nvalid, v1 = g + 8 < nvalid;
      float sc[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        sc[u] = (u < 2 ? v0 : v1) ? ((sa[u] + sb[u]) + (la[u] + lb[u])) * P.scale_log2 : -INFINITY;
      float mx[2] = {fmaxf(sc[0], sc[2]), fmaxf(sc[1], sc[3])};
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], o));
        mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], o));
      }
      const bool up = mx[0] > mc[0] + kDRescaleLog2 || mx[1] > mc[1] + kDRescaleLog2;
      if (__any_sync(0xffffffffu, up)) {
        float al[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const float mn = mx[e] > mc[e] + kDRescaleLog2 ? mx[e] : mc[e];
          al[e] = mc[e] == -INFINITY ? 0.f : exp2f(mc[e] - mn);
          mc[e] = mn;
          lc[e] *= al[e];
        }
#pragma unroll
        for (int m = 0; m < MH; ++m) {
          acc[m][0] *= al[0]; acc[m][1] *= al[1]; acc[m][2] *= al[0]; acc[m][3] *= al[1];
        }
      }
      const float p0 = exp2f(sc[0] - mc[0]), p1 = exp2f(sc[1] - mc[1]);
      const float p2 = exp2f(sc[2] - mc[0]), p3 = exp2f(sc[3] - mc[1]);
      lc[0] += p0 + p2;
      lc[1] += p1 + p3;
      const uint32_t pb0 = movmatrix_trans(pack_bf16x2(p0, p1));
      const uint32_t pb1 = movmatrix_trans(pack_bf16x2(p2, p3));
      auto valid = [&](int row) { return row < nvalid; };
      const uint32_t keep0 = (valid(2 * q4) ? 0x0000ffffu : 0u) | (valid(2 * q4 + 1) ? 0xffff0000u : 0u);
      const uint32_t keep1 = (valid(2 * q4 + 8) ? 0x0000ffffu : 0u) | (valid(2 * q4 + 9) ? 0xffff0000u : 0u);
#pragma unroll
      for (int m0 = 0; m0 < MH; m0 += 4) {
        uint32_t a[4][4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ch = 2 * (dhf * MH + m0 + u) + tcol;
          ldsm_x4_trans(a[u][0], a[u][1], a[u][2], a[u][3], cs + (ch >> 3) * (kDT * 128) + swz_off(trow, ch & 7, 128));
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          mma_bf16_16816(acc[m0 + u], a[u][0] & keep0, a[u][1] & keep0, a[u][2] & keep1, a[u][3] & keep1, pb0, pb1);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();
        const bool last = (atomicAdd(&cons[s], 1) % nwarps) == nwarps - 1;
        __threadfence_block();
        if (last && ahead_more && !*reinterpret_cast<volatile int*>(&s_timeout)) {
          fence_proxy_async_smem();
          issue(s, j + P.stages, ahead);
        }
      }
      __syncwarp();
    }
    more = walk_next(w, pre, B, g1, kDT);
    if (ahead_more) ahead_more = walk_next(ahead, pre, B, g1, kDT);
  }
  if (cur_b >= 0) write_partial(cur_b);

  __syncthreads();
  if (tid == 0) {
    bool drained = true;
    for (int st = 0; st < P.stages; ++st) {
      const int jj = *reinterpret_cast<volatile int*>(&issued[st]);
      if (jj >= 0) drained = mbar_wait_bounded(&full[st], static_cast<uint32_t>(jj / P.stages) & 1u) && drained;
    }
    if (!drained) *reinterpret_cast<volatile int*>(&s_timeout) = 1;
    if (blockIdx.x == 0) {
      P.meta[0] = N;
      P.meta[1] = G;
    }
    *cta_status = (bad ? kDevBounds : 0u) | (*reinterpret_cast<volatile int*>(&s_timeout) ? kDevTimeout : 0u);
  }
  if (blockIdx.x == 0)
    for (int b = tid; b <= B; b += blockDim.x) P.prefix[b] = pre[b];
}

// ======================================================================= host
namespace {

using DenseFn = void (*)(const DecodePlan, const CUtensorMap, const CUtensorMap);

template <int D>
DenseFn dense_fn_g(int ng) {
  switch (ng) {
    case 1: return lrkv_dense_decode_kernel<D, 1>;
    case 2: return lrkv_dense_decode_kernel<D, 2>;
    case 4: return lrkv_dense_decode_kernel<D, 4>;
    case 8: return lrkv_dense_decode_kernel<D, 8>;
    default: return nullptr;
  }
}

DenseFn dense_fn(int d, int ng) {
  if (d == 64) return dense_fn_g<64>(ng);
  if (d == 128) return dense_fn_g<128>(ng);
  return nullptr;
}

lrkv_status dense_check(const lrkv_dense_dims* d) {
  if (!d) return LRKV_ERR_INVALID_ARG;
  if (d->batch < 1 || d->heads < 1 || d->kv_heads < 1 || d->head_dim < 1 || d->max_len < 1)
    return LRKV_ERR_INVALID_ARG;
  if (!(d->scale == d->scale)) return LRKV_ERR_INVALID_ARG;
  if (d->heads % d->kv_heads != 0) return LRKV_ERR_INVALID_ARG;
  if (!dense_fn(d->head_dim, d->heads / d->kv_heads)) return LRKV_ERR_UNSUPPORTED;
  if (d->batch > kMaxBatch || static_cast<long long>(d->batch) * d->max_len > (1LL << 31) - 1)
    return LRKV_ERR_UNSUPPORTED;
  return LRKV_OK;
}

lrkv_status dense_make_plan(const lrkv_dense_dims& d, int num_sms, DecodePlan& P, size_t* ws_bytes) {
  std::memset(&P, 0, sizeof(P));
  P.B = d.batch; P.H = d.heads; P.dh = d.head_dim; P.r = 0; P.max_len = d.max_len;
  P.map_len = d.max_len; P.map_seqs = d.batch;
  const float scale = d.scale > 0.f ? d.scale : 1.f / std::sqrt(static_cast<float>(d.head_dim));
  P.scale_log2 = scale * kLog2e;
  P.bf16 = 1; P.esz = 2; P.T = kDT; P.stream = 1;
  {
    const char* v = std::getenv("LRKV_WAIT_LIMIT_CYCLES");
    const long long x = (v && *v) ? std::atoll(v) : 0;
    P.wait_limit = x > 0 ? x : kWaitLimitCycles;
  }
  int kvg = kDMaxWarps;
  while (kvg > 1 && d.kv_heads % kvg != 0) kvg >>= 1;
  P.nthreads = 32 * kvg;
  P.mt = d.kv_heads / kvg;
  P.grid = std::max(1, num_sms / P.mt);
  P.ngw = 1;
  P.kv_bytes = kvg * kDT * d.head_dim * 2;  // a multiple of 2048 (d a multiple of 64)
  P.stage_bytes = 2 * P.kv_bytes;
  P.off_prefix = kDHeader;
  P.off_kv = round_up(kDHeader + (P.B + 1) * 4, 1024);
  const int budget = 226 * 1024;
  P.stages = std::min(kDMaxStages, (budget - P.off_kv - 1024) / P.stage_bytes);
  if (P.stages < 2) return LRKV_ERR_UNSUPPORTED;
  P.smem_bytes = P.off_kv + P.stages * P.stage_bytes + 1024;
  P.min_tokens = 8 * kDT;
  P.wide_merge = 1;
  P.wide_warps = 8;
  P.combine_ctas = static_cast<int>(std::min<long long>(static_cast<long long>(P.B) * P.H, 4ll * num_sms));
  *ws_bytes = decode_workspace_bytes(P);
  return LRKV_OK;
}

bool d16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

using MlaFn = void (*)(const DecodePlan, const CUtensorMap);

MlaFn mla_fn(int dc) {
  if (dc == 256) return lrkv_mla_decode_kernel<256>;
  if (dc == 512) return lrkv_mla_decode_kernel<512>;
  return nullptr;
}

lrkv_status mla_check(const lrkv_mla_dims* d) {
  if (!d) return LRKV_ERR_INVALID_ARG;
  if (d->batch < 1 || d->heads < 1 || d->head_dim < 1 || d->latent_dim < 1 || d->max_len < 1)
    return LRKV_ERR_INVALID_ARG;
  if (!(d->scale == d->scale)) return LRKV_ERR_INVALID_ARG;
  if (!mla_fn(d->latent_dim) || !(d->heads == 8 || d->heads == 16 || d->heads == 32) || d->head_dim > 128)
    return LRKV_ERR_UNSUPPORTED;
  if (d->batch > kMaxBatch || static_cast<long long>(d->batch) * d->max_len > (1LL << 31) - 1)
    return LRKV_ERR_UNSUPPORTED;
  return LRKV_OK;
}

lrkv_status mla_make_plan(const lrkv_mla_dims& d, int num_sms, DecodePlan& P, size_t* ws_bytes) {
  std::memset(&P, 0, sizeof(P));
  P.B = d.batch; P.H = d.heads; P.dh = d.head_dim; P.r = d.latent_dim; P.max_len = d.max_len;
  P.map_len = d.max_len; P.map_seqs = d.batch;
  const float scale = d.scale > 0.f ? d.scale : 1.f / std::sqrt(static_cast<float>(d.head_dim));
  P.scale_log2 = scale * kLog2e;
  P.bf16 = 1; P.esz = 2; P.T = kDT; P.stream = 1;
  {
    const char* v = std::getenv("LRKV_WAIT_LIMIT_CYCLES");
    const long long x = (v && *v) ? std::atoll(v) : 0;
    P.wait_limit = x > 0 ? x : kWaitLimitCycles;
  }
  P.nthreads = 2 * (P.H / 8) * 32;
  P.mt = 1;
  P.grid = num_sms;
  P.ngw = 1;
  P.off_prefix = kDHeader;
  P.off_pq = round_up(kDHeader + (P.B + 1) * 4, 1024);
  P.pq_bytes = (P.H / 8) * (P.r / 16) * 32 * 16;  // the groups' q tables
  P.off_kv = round_up(P.off_pq + P.pq_bytes, 1024);
  P.stage_bytes = kDT * P.r * 2;
  const int budget = 226 * 1024;
  P.stages = std::min(kDMaxStages, (budget - P.off_kv - 1024) / P.stage_bytes);
  if (P.stages < 2) return LRKV_ERR_UNSUPPORTED;
  P.smem_bytes = P.off_kv + P.stages * P.stage_bytes + 1024;
  P.min_tokens = 8 * kDT;
  P.wide_merge = 1;
  P.wide_warps = 8;
  P.combine_ctas = static_cast<int>(std::min<long long>(static_cast<long long>(P.B) * P.H, 4ll * num_sms));
  *ws_bytes = decode_workspace_bytes(P);
  return LRKV_OK;
}

}  // namespace

}  // namespace lrkv

extern "C" {

lrkv_status lrkv_dense_decode_workspace_size(const lrkv_dense_dims* dims, size_t* bytes) {
  if (!bytes) return LRKV_ERR_INVALID_ARG;
  lrkv_status st = lrkv::dense_check(dims);
  if (st != LRKV_OK) return st;
  const int sms = lrkv::device_sm_count();
  if (sms < 1) return LRKV_ERR_CUDA;
  lrkv::DecodePlan P;
  return lrkv::dense_make_plan(*dims, sms, P, bytes);
}

lrkv_status lrkv_dense_decode(const lrkv_dense_dims* dims, const void* q, const void* k, const void* v,
                              const int32_t* seq_lens, float* out, float* lse, void* ws, size_t ws_bytes,
                              lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_dense_decode");
  lrkv_status st = lrkv::dense_check(dims);
  if (st != LRKV_OK) return st;
  if (!q || !k || !v || !seq_lens || !out) return LRKV_ERR_INVALID_ARG;
  if (!lrkv::d16(q) || !lrkv::d16(k) || !lrkv::d16(v)) return LRKV_ERR_INVALID_ARG;
  if (!ws) return LRKV_ERR_WORKSPACE;
  if (!lrkv::d16(ws)) return LRKV_ERR_INVALID_ARG;
  const int sms = lrkv::device_sm_count();
  if (sms < 1) return LRKV_ERR_CUDA;
  lrkv::DecodePlan P;
  size_t need = 0;
  if ((st = lrkv::dense_make_plan(*dims, sms, P, &need)) != LRKV_OK) return st;
  if (ws_bytes < need) return LRKV_ERR_WORKSPACE;
  lrkv::decode_bind_workspace(P, ws);
  P.q = q; P.k_s = k; P.v_s = v; P.seq_lens = seq_lens; P.out = out; P.lse = lse;
  const int kvg = P.nthreads / 32;
  // K, V [B][L][H_kv][d] seen as {d, L, H_kv, B}: a box {64, 16, kvg, 1} lands
  // as [head][token][64 columns], 128-byte swizzle
  CUtensorMap tm_k, tm_v;
  std::memset(&tm_k, 0, sizeof(tm_k));
  std::memset(&tm_v, 0, sizeof(tm_v));
  const uint64_t dd = static_cast<uint64_t>(dims->head_dim), hkv = static_cast<uint64_t>(dims->kv_heads);
  const uint64_t dm[4] = {dd, static_cast<uint64_t>(P.max_len), hkv, static_cast<uint64_t>(P.B)};
  const uint64_t strides[3] = {hkv * dd * 2, dd * 2, static_cast<uint64_t>(P.max_len) * hkv * dd * 2};
  const uint32_t box[4] = {64u, static_cast<uint32_t>(lrkv::kDT), static_cast<uint32_t>(kvg), 1u};
  if (!lrkv::make_tmap_4d_bf16_swizzled(&tm_k, k, dm, strides, box) ||
      !lrkv::make_tmap_4d_bf16_swizzled(&tm_v, v, dm, strides, box))
    return LRKV_ERR_CUDA;
  const lrkv::DenseFn kern = lrkv::dense_fn(dims->head_dim, dims->heads / dims->kv_heads);
  if (lrkv::ensure_kernel_smem(reinterpret_cast<const void*>(kern), P.smem_bytes, true) != cudaSuccess)
    return LRKV_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid, P.mt);
  cfg.blockDim = dim3(P.nthreads);
  cfg.dynamicSmemBytes = P.smem_bytes;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, P, tm_k, tm_v) != cudaSuccess) return LRKV_ERR_CUDA;
  return lrkv::decode_merge_launch(P, stream, true);
}

lrkv_status lrkv_mla_decode_workspace_size(const lrkv_mla_dims* dims, size_t* bytes) {
  if (!bytes) return LRKV_ERR_INVALID_ARG;
  lrkv_status st = lrkv::mla_check(dims);
  if (st != LRKV_OK) return st;
  const int sms = lrkv::device_sm_count();
  if (sms < 1) return LRKV_ERR_CUDA;
  lrkv::DecodePlan P;
  return lrkv::mla_make_plan(*dims, sms, P, bytes);
}

lrkv_status lrkv_mla_decode(const lrkv_mla_dims* dims, const void* q, const void* c, const void* w_uk,
                            const void* w_uv, const int32_t* seq_lens, float* out, float* lse, void* ws,
                            size_t ws_bytes, lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_mla_decode");
  lrkv_status st = lrkv::mla_check(dims);
  if (st != LRKV_OK) return st;
  if (!q || !c || !w_uk || !w_uv || !seq_lens || !out) return LRKV_ERR_INVALID_ARG;
  if (!lrkv::d16(c)) return LRKV_ERR_INVALID_ARG;
  if (!ws) return LRKV_ERR_WORKSPACE;
  if (!lrkv::d16(ws)) return LRKV_ERR_INVALID_ARG;
  const int sms = lrkv::device_sm_count();
  if (sms < 1) return LRKV_ERR_CUDA;
  lrkv::DecodePlan P;
  size_t need = 0;
  if ((st = lrkv::mla_make_plan(*dims, sms, P, &need)) != LRKV_OK) return st;
  if (ws_bytes < need) return LRKV_ERR_WORKSPACE;
  lrkv::decode_bind_workspace(P, ws);
  P.q = q; P.k_s = c; P.b_v = w_uv; P.seq_lens = seq_lens; P.out = out; P.lse = lse;
  CUtensorMap tm_c;
  std::memset(&tm_c, 0, sizeof(tm_c));
  if (!lrkv::make_tmap_3d_bf16(&tm_c, c, P.r, P.max_len, P.B, 64, lrkv::kDT, CU_TENSOR_MAP_SWIZZLE_128B))
    return LRKV_ERR_CUDA;
  const lrkv::MlaFn kern = lrkv::mla_fn(P.r);
  if (lrkv::ensure_kernel_smem(reinterpret_cast<const void*>(kern), P.smem_bytes, true) != cudaSuccess)
    return LRKV_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // q_c = q W_uk[h] into the workspace (stream-ordered after the launch
  // before, which may still read it)
  lrkv::lrkv_mla_absorb_kernel<<<dim3(P.H, P.B), 256, P.dh * 4, s>>>(P,
                                                                     static_cast<const __nv_bfloat16*>(w_uk));
  if (cudaGetLastError() != cudaSuccess) return LRKV_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid);
  cfg.blockDim = dim3(P.nthreads);
  cfg.dynamicSmemBytes = P.smem_bytes;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, P, tm_c) != cudaSuccess) return LRKV_ERR_CUDA;
  return lrkv::decode_merge_launch(P, stream, true);
}

}  // extern "C"
