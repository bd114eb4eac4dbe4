// decode_rope.cu — decode with full rotary position embedding of the keys on
// the factored cache ("Low-Rank Key Value Attention | What a shared cache can
// preserve", §8, "Full RoPE needs a stronger identity"; "Low-Rank Key Value
// Attention：中文研读笔记", §2.7).
//
// The rotation D_j of key position j cannot be moved into the rank-r latent
// for a generic basis B_h (the review's Figure 9), so the cache keeps
// unrotated rows and the exact score is a position-dependent contraction:
// q~ . (k_j D_j) with k_j = s_j + z_j B_h^T.  This kernel rebuilds the keys
// tile by tile on the tensor cores (K = Z_h B_h^T, mma.sync, exact bf16
// products, fp32 accumulation), adds the shared row, turns every pair
// (2k, 2k+1) by the table's (cos, sin) of (j, k) and takes the dot product
// with the rotated query; one online softmax per head.  The values are not
// rotated, so O_s and O_z accumulate as in the plain decode and the same
// merge lifts O_z through (B_h^V)^T.  The rebuild costs d_h r multiply-adds
// per (token, head) beyond the plain decode: the computational cost the
// review names for the exact option.
//
// Grid (range CTAs, groups of 8 heads).  Each of the 8 warps owns one head
// (B_h's MMA fragments live in its registers).  A ring of shared-memory stages
// is filled by TMA: per 16-token tile the shared rows k_s and v_s
// (128-byte-swizzled boxes), the group's latents z_k and z_v (segment rows
// padded to an odd number of 16-byte chunks) and the tile's 16 table rows;
// every warp walks the tiles in order and the last of the 8 warps to finish
// a stage refills it with the tile `stages` ahead.  Every wait is bounded.
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

constexpr int kRT = 16;                      // tokens per tile
constexpr int kRHeads = 8;                   // heads per CTA, one consumer warp each
constexpr int kRThreads = 32 * kRHeads;
constexpr int kRHeader = 1024;               // barriers and stage records
constexpr int kRMaxStages = 16;

}  // namespace

// Table of the rotation: cos_sin[j][2k] = cos(j theta_k),
// cos_sin[j][2k + 1] = sin(j theta_k), theta_k = base^(-2k / d_h); the angle
// and both functions in fp64, rounded once to fp32.
__global__ void lrkv_rope_table_kernel(int max_pos, int dh, double base, float* table) {
  const long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int half = dh / 2;
  if (i >= static_cast<long long>(max_pos) * half) return;
  const int j = static_cast<int>(i / half), k = static_cast<int>(i % half);
  const double theta = pow(base, -2.0 * k / dh);
  double sn, cs;
  sincos(static_cast<double>(j) * theta, &sn, &cs);
  table[static_cast<size_t>(j) * dh + 2 * k] = static_cast<float>(cs);
  table[static_cast<size_t>(j) * dh + 2 * k + 1] = static_cast<float>(sn);
}

template <int DH, int R>
__global__ void __launch_bounds__(kRThreads, 1)
    lrkv_decode_rope_kernel(const __grid_constant__ DecodePlan P, const __grid_constant__ CUtensorMap tm_k,
                            const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_zk,
                            const __grid_constant__ CUtensorMap tm_zv, const __grid_constant__ CUtensorMap tm_cs) {
  constexpr int NT = DH / 8;   // 8-column tiles of the rebuilt key
  constexpr int KS = R / 16;   // 16-wide steps over a head's latents
  constexpr int CW = DH / 32;  // shared value columns per lane
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_timeout;
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  pdl_trigger();  // the merge may launch: it waits for this grid before it reads
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, q4 = lane & 3;
  const int B = P.B, H = P.H;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  int* cons = reinterpret_cast<int*>(smem + 128);    // [16] warps done with each stage (all uses)
  int* issued = reinterpret_cast<int*>(smem + 256);  // [16] last tile issued into each stage
  int* pre = reinterpret_cast<int*>(smem + kRHeader);

  // ---- 1. barriers, sequence starts (clamped lengths) ----------------------
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
  const int segrow = P.segp * 2;  // bytes per latent segment row

  const int zseg0 = blockIdx.y * P.nsb;
  const uint32_t tx = static_cast<uint32_t>(2 * (DH / 64) * kRT * 128 + 2 * P.zt_bytes + P.cs_bytes);
  // the copies of tile (sequence b, rows t0 ..) into stage s (one thread)
  auto issue = [&](int s, int j, const TileWalk& t) {
    unsigned char* ks = smem + P.off_kv + static_cast<size_t>(s) * P.stage_bytes;
    unsigned char* vs = ks + P.kv_bytes;
    unsigned char* zk = vs + P.kv_bytes;
    unsigned char* zv = zk + P.zt_bytes;
    unsigned char* cs = zv + P.zt_bytes;
    mbar_arrive_expect_tx(&full[s], tx);
#pragma unroll
    for (int cb = 0; cb < DH / 64; ++cb) {
      tma_load_3d(ks + cb * kRT * 128, &tm_k, cb * 64, t.t0, t.b, &full[s]);
      tma_load_3d(vs + cb * kRT * 128, &tm_v, cb * 64, t.t0, t.b, &full[s]);
    }
    tma_load_4d(zk, &tm_zk, 0, t.t0, zseg0, t.b, &full[s]);
    tma_load_4d(zv, &tm_zv, 0, t.t0, zseg0, t.b, &full[s]);
    tma_load_2d(cs, &tm_cs, 0, t.t0, &full[s]);
    *reinterpret_cast<volatile int*>(&issued[s]) = j;
  };
  // the walk `stages` tiles ahead: the first stages' tiles go out now
  TileWalk ahead;
  bool ahead_more = walk_first(ahead, pre, B, g0, g1);
  for (int j = 0; j < P.stages && ahead_more; ++j) {
    if (tid == 0) issue(j, j, ahead);
    ahead_more = walk_next(ahead, pre, B, g1, kRT);
  }
  {
    // ================================================ consumers: head h ====
    const int h = blockIdx.y * kRHeads + warp;
    // B_h^K as the B operand of K = Z_h B_h^T (k = latent column, n = head
    // dim): lane (g, q4) holds B_h[8 n + g][16 kk + 2 q4 (+1)] and [.. + 8 (+9)]
    uint32_t bf[NT][KS][2];
    {
      const __nv_bfloat16* bk = static_cast<const __nv_bfloat16*>(P.b_k) + static_cast<size_t>(h) * DH * R;
#pragma unroll
      for (int n = 0; n < NT; ++n)
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          const __nv_bfloat16* row = bk + (8 * n + g) * R + 16 * kk + 2 * q4;
          bf[n][kk][0] = *reinterpret_cast<const uint32_t*>(row);
          bf[n][kk][1] = *reinterpret_cast<const uint32_t*>(row + 8);
        }
    }
    const int zoff = (warp / P.hs) * (kRT * segrow) + (warp % P.hs) * R * 2;  // this head in a latent tile
    // value columns of this lane: shared d0 .. d0 + CW - 1, private lane (+ 32)
    const int d0 = CW * lane;
    const int vcb = d0 >> 6, vch = (d0 & 63) >> 3, voff = (d0 & 7) * 2;

    TileWalk w;
    bool more = walk_first(w, pre, B, g0, g1);
    bool ok = true, waited = false;
    int cur_b = -1;
    float m = -INFINITY, l = 0.f;
    float os[CW], oz[2] = {0.f, 0.f};
#pragma unroll
    for (int e = 0; e < CW; ++e) os[e] = 0.f;
    uint32_t qv[NT];  // q~ of head h: columns 8 n + 2 q4, + 1 (bf16 pairs)

    // this head's partial of sequence b: (m, l) and the unnormalised
    // [O_s | O_z] at slot b + c (the merge takes every CTA's)
    auto write_partial = [&](int b) {
      if (!waited) {
        pdl_wait();  // the launch before may still read the workspace
        waited = true;
      }
      const size_t slot = static_cast<size_t>(b + c);
      if (lane == 0) {
        float* pml = P.part_ml + (slot * H + h) * 2;
        pml[0] = m;
        pml[1] = l;
      }
      float* o = P.part_acc + (slot * H + h) * (DH + R);
#pragma unroll
      for (int e = 0; e < CW; ++e) o[d0 + e] = os[e];
      if (lane < R) o[DH + lane] = oz[0];
      if (lane + 32 < R) o[DH + lane + 32] = oz[1];
    };

    for (int j = 0; more; ++j) {
      if (w.b != cur_b) {
        if (cur_b >= 0) write_partial(cur_b);
        cur_b = w.b;
        m = -INFINITY;
        l = 0.f;
#pragma unroll
        for (int e = 0; e < CW; ++e) os[e] = 0.f;
        oz[0] = oz[1] = 0.f;
        const __nv_bfloat16* qh = static_cast<const __nv_bfloat16*>(P.q) + (static_cast<size_t>(w.b) * H + h) * DH;
#pragma unroll
        for (int n = 0; n < NT; ++n) qv[n] = *reinterpret_cast<const uint32_t*>(qh + 8 * n + 2 * q4);
      }
      const int s = j % P.stages;
      const int nvalid = min(kRT, w.t_end - w.t0);
      if (ok && *reinterpret_cast<volatile int*>(&s_timeout)) ok = false;  // another warp gave up
      if (ok) {
        ok = mbar_wait_bounded(&full[s], static_cast<uint32_t>(j / P.stages) & 1u, P.wait_limit);
        if (!ok) *reinterpret_cast<volatile int*>(&s_timeout) = 1;
      }
      if (ok) {
        const unsigned char* ks = smem + P.off_kv + static_cast<size_t>(s) * P.stage_bytes;
        const unsigned char* vs = ks + P.kv_bytes;
        const unsigned char* zk = vs + P.kv_bytes;
        const unsigned char* zv = zk + P.zt_bytes;
        const float* cs = reinterpret_cast<const float*>(zv + P.zt_bytes);
        // ---- rebuilt, rotated key . q~ : tokens g (part0) and g + 8 (part1) ----
        uint32_t a[KS][4];
#pragma unroll
        for (int kk = 0; kk < KS; ++kk)
          ldsm_x4(a[kk][0], a[kk][1], a[kk][2], a[kk][3],
                  zk + zoff + (lane & 15) * segrow + (16 * kk + 8 * (lane >> 4)) * 2);
        const float* cs0 = cs + g * P.cs_row;
        const float* cs1 = cs0 + 8 * P.cs_row;
        float part0 = 0.f, part1 = 0.f;
#pragma unroll
        for (int n0 = 0; n0 < NT; n0 += 4) {
          float acc[4][4];
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            acc[u][0] = acc[u][1] = acc[u][2] = acc[u][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < KS; ++kk)
              mma_bf16_16816(acc[u], a[kk][0], a[kk][1], a[kk][2], a[kk][3], bf[n0 + u][kk][0], bf[n0 + u][kk][1]);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int n = n0 + u, d = 8 * n + 2 * q4;
            const unsigned char* kb = ks + (d >> 6) * (kRT * 128);
            const uint32_t s0 = *reinterpret_cast<const uint32_t*>(kb + swz_off(g, (d & 63) >> 3, 128) + 4 * q4);
            const uint32_t s1 = *reinterpret_cast<const uint32_t*>(kb + swz_off(g + 8, (d & 63) >> 3, 128) + 4 * q4);
            const float2 c0 = *reinterpret_cast<const float2*>(cs0 + d);  // (cos, sin) of pair d / 2
            const float2 c1 = *reinterpret_cast<const float2*>(cs1 + d);
            const float x0 = acc[u][0] + bf_lo(s0), x1 = acc[u][1] + bf_hi(s0);
            const float y0 = acc[u][2] + bf_lo(s1), y1 = acc[u][3] + bf_hi(s1);
            const float qa = bf_lo(qv[n]), qb = bf_hi(qv[n]);
            part0 = fmaf(qa, fmaf(x0, c0.x, -x1 * c0.y), fmaf(qb, fmaf(x0, c0.y, x1 * c0.x), part0));
            part1 = fmaf(qa, fmaf(y0, c1.x, -y1 * c1.y), fmaf(qb, fmaf(y0, c1.y, y1 * c1.x), part1));
          }
        }
        part0 += __shfl_xor_sync(0xffffffffu, part0, 1);
        part0 += __shfl_xor_sync(0xffffffffu, part0, 2);
        part1 += __shfl_xor_sync(0xffffffffu, part1, 1);
        part1 += __shfl_xor_sync(0xffffffffu, part1, 2);
        // ---- one online softmax over the tile (log2 domain) ----
        const float sc0 = g < nvalid ? part0 * P.scale_log2 : -INFINITY;
        const float sc1 = g + 8 < nvalid ? part1 * P.scale_log2 : -INFINITY;
        float mx = fmaxf(sc0, sc1);
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o2));
        const float mn = fmaxf(m, mx);
        const float alpha = m == -INFINITY ? 0.f : exp2f(m - mn);
        const float p0 = exp2f(sc0 - mn), p1 = exp2f(sc1 - mn);
        float ps = p0 + p1;
#pragma unroll
        for (int o2 = 4; o2 < 32; o2 <<= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o2);
        l = fmaf(l, alpha, ps);
        m = mn;
#pragma unroll
        for (int e = 0; e < CW; ++e) os[e] *= alpha;
        oz[0] *= alpha;
        oz[1] *= alpha;
        // ---- values, unrotated: rows of the history only (rows past it may hold anything) ----
        const unsigned char* vb = vs + vcb * (kRT * 128);
        const unsigned char* zvh = zv + zoff;
        for (int t = 0; t < nvalid; ++t) {
          const float pt = __shfl_sync(0xffffffffu, t < 8 ? p0 : p1, (t & 7) * 4);
          const unsigned char* vrow = vb + swz_off(t, vch, 128) + voff;
          if constexpr (CW == 4) {
            const uint2 v = *reinterpret_cast<const uint2*>(vrow);
            os[0] = fmaf(pt, bf_lo(v.x), os[0]);
            os[1] = fmaf(pt, bf_hi(v.x), os[1]);
            os[2] = fmaf(pt, bf_lo(v.y), os[2]);
            os[3] = fmaf(pt, bf_hi(v.y), os[3]);
          } else {
            const uint32_t v = *reinterpret_cast<const uint32_t*>(vrow);
            os[0] = fmaf(pt, bf_lo(v), os[0]);
            os[1] = fmaf(pt, bf_hi(v), os[1]);
          }
          const __nv_bfloat16* zr = reinterpret_cast<const __nv_bfloat16*>(zvh + t * segrow);
          if (lane < R) oz[0] = fmaf(pt, __bfloat162float(zr[lane]), oz[0]);
          if (lane + 32 < R) oz[1] = fmaf(pt, __bfloat162float(zr[lane + 32]), oz[1]);
        }
        // the stage is free once all eight heads are done with it: the last
        // warp to finish refills it with the tile `stages` ahead (a warp
        // counts only after it saw the stage's copy land, so a refill never
        // joins a pending phase)
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          __threadfence_block();
          const bool last = (atomicAdd(&cons[s], 1) % kRHeads) == kRHeads - 1;
          __threadfence_block();
          if (last && ahead_more && !*reinterpret_cast<volatile int*>(&s_timeout)) {
            fence_proxy_async_smem();
            issue(s, j + P.stages, ahead);
          }
        }
        __syncwarp();
      }
      more = walk_next(w, pre, B, g1, kRT);
      if (ahead_more) ahead_more = walk_next(ahead, pre, B, g1, kRT);
    }
    if (cur_b >= 0) write_partial(cur_b);
  }

  // ---- every copy this CTA issued has landed before it exits ----
  __syncthreads();
  if (tid == 0) {
    pdl_wait();
    bool drained = true;
    for (int st = 0; st < P.stages; ++st) {
      const int j = *reinterpret_cast<volatile int*>(&issued[st]);
      if (j >= 0) drained = mbar_wait_bounded(&full[st], static_cast<uint32_t>(j / P.stages) & 1u) && drained;
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

// ======================================================================= host
namespace {

using RopeFn = void (*)(const DecodePlan, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                        const CUtensorMap, const CUtensorMap);

template <int DH>
RopeFn rope_fn_r(int r) {
  switch (r) {
    case 16: return lrkv_decode_rope_kernel<DH, 16>;
    case 32: return lrkv_decode_rope_kernel<DH, 32>;
    case 48: return lrkv_decode_rope_kernel<DH, 48>;
    case 64: return lrkv_decode_rope_kernel<DH, 64>;
    default: return nullptr;
  }
}

RopeFn rope_fn(int dh, int r) {
  if (dh == 64) return rope_fn_r<64>(r);
  if (dh == 128) return rope_fn_r<128>(r);
  return nullptr;
}

lrkv_status rope_check(const lrkv_dims* d) {
  if (!d) return LRKV_ERR_INVALID_ARG;
  if (d->batch < 1 || d->heads < 1 || d->head_dim < 1 || d->rank < 0 || d->max_len < 1) return LRKV_ERR_INVALID_ARG;
  if (d->dtype != LRKV_BF16 && d->dtype != LRKV_F32) return LRKV_ERR_INVALID_ARG;
  if (!(d->scale == d->scale)) return LRKV_ERR_INVALID_ARG;
  if (d->dtype != LRKV_BF16 || !rope_fn(d->head_dim, d->rank) || d->heads % kRHeads != 0) return LRKV_ERR_UNSUPPORTED;
  if (d->batch > kMaxBatch || static_cast<long long>(d->batch) * d->max_len > (1LL << 31) - 1)
    return LRKV_ERR_UNSUPPORTED;
  return LRKV_OK;
}

lrkv_status rope_make_plan(const lrkv_dims& d, int num_sms, DecodePlan& P, size_t* ws_bytes) {
  std::memset(&P, 0, sizeof(P));
  P.B = d.batch; P.H = d.heads; P.dh = d.head_dim; P.r = d.rank; P.max_len = d.max_len;
  P.map_len = d.max_len; P.map_seqs = d.batch;
  const float scale = d.scale > 0.f ? d.scale : 1.f / std::sqrt(static_cast<float>(d.head_dim));
  P.scale_log2 = scale * kLog2e;
  P.bf16 = 1; P.esz = 2; P.T = kRT; P.stream = 1;
  {
    const char* v = std::getenv("LRKV_WAIT_LIMIT_CYCLES");
    const long long x = (v && *v) ? std::atoll(v) : 0;
    P.wait_limit = x > 0 ? x : kWaitLimitCycles;
  }
  P.mt = P.H / kRHeads;
  P.grid = std::max(1, num_sms / P.mt);
  P.ngw = 1;
  P.hs = 0;
  for (int hs = kRHeads; hs >= 1; hs >>= 1)
    if (P.H % hs == 0 && (hs * P.r) % 16 == 0 && hs * P.r + 8 <= 256) { P.hs = hs; break; }
  if (P.hs == 0) return LRKV_ERR_UNSUPPORTED;
  P.segw = P.hs * P.r;
  P.segp = P.segw + 8;
  P.nsb = kRHeads / P.hs;
  P.zt_bytes = P.nsb * kRT * P.segp * 2;
  P.kv_bytes = round_up(kRT * P.dh * 2, 1024);
  P.cs_row = P.dh + 4;  // table rows padded in shared memory (zeros from the box)
  P.cs_bytes = kRT * P.cs_row * 4;
  P.stage_bytes = round_up(2 * P.kv_bytes + 2 * P.zt_bytes + P.cs_bytes, 1024);
  P.off_prefix = kRHeader;
  P.off_kv = round_up(kRHeader + (P.B + 1) * 4, 1024);
  const int budget = 226 * 1024;
  P.stages = std::min(kRMaxStages, (budget - P.off_kv - 1024) / P.stage_bytes);
  if (P.stages < 2) return LRKV_ERR_UNSUPPORTED;
  P.smem_bytes = P.off_kv + P.stages * P.stage_bytes + 1024;
  P.min_tokens = 8 * kRT;
  P.wide_merge = 1;
  P.wide_warps = 8;
  P.combine_ctas = static_cast<int>(std::min<long long>(static_cast<long long>(P.B) * P.H, 4ll * num_sms));
  P.combine_smem = 0;
  *ws_bytes = decode_workspace_bytes(P);
  return LRKV_OK;
}

bool a16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

}  // namespace lrkv

extern "C" {

lrkv_status lrkv_rope_table(int max_pos, int head_dim, float base, float* cos_sin, lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_rope_table");
  if (max_pos < 1 || head_dim < 2 || head_dim % 2 != 0 || !(base > 1.f) || !cos_sin) return LRKV_ERR_INVALID_ARG;
  const long long n = static_cast<long long>(max_pos) * (head_dim / 2);
  if (n > (1ll << 40)) return LRKV_ERR_UNSUPPORTED;
  const int threads = 256;
  const long long blocks = (n + threads - 1) / threads;
  if (blocks > 0x7fffffffll) return LRKV_ERR_UNSUPPORTED;
  lrkv::lrkv_rope_table_kernel<<<static_cast<unsigned>(blocks), threads, 0, static_cast<cudaStream_t>(stream)>>>(
      max_pos, head_dim, static_cast<double>(base), cos_sin);
  return cudaGetLastError() == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

lrkv_status lrkv_decode_rope_workspace_size(const lrkv_dims* dims, size_t* bytes) {
  if (!bytes) return LRKV_ERR_INVALID_ARG;
  lrkv_status st = lrkv::rope_check(dims);
  if (st != LRKV_OK) return st;
  const int sms = lrkv::device_sm_count();
  if (sms < 1) return LRKV_ERR_CUDA;
  lrkv::DecodePlan P;
  return lrkv::rope_make_plan(*dims, sms, P, bytes);
}

lrkv_status lrkv_decode_rope(const lrkv_dims* dims, const void* q_rot, const void* k_s, const void* v_s,
                             const void* z_k, const void* z_v, const void* b_k, const void* b_v,
                             const float* cos_sin, int max_pos, const int32_t* seq_lens, float* out, float* lse,
                             void* ws, size_t ws_bytes, lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_decode_rope");
  lrkv_status st = lrkv::rope_check(dims);
  if (st != LRKV_OK) return st;
  if (!q_rot || !k_s || !v_s || !z_k || !z_v || !b_k || !b_v || !cos_sin || !seq_lens || !out)
    return LRKV_ERR_INVALID_ARG;
  if (!lrkv::a16(q_rot) || !lrkv::a16(k_s) || !lrkv::a16(v_s) || !lrkv::a16(z_k) || !lrkv::a16(z_v) ||
      !lrkv::a16(b_k) || !lrkv::a16(cos_sin) || !lrkv::a16(out))
    return LRKV_ERR_INVALID_ARG;
  if (max_pos < dims->max_len) return LRKV_ERR_INVALID_ARG;  // every cache row needs its table row
  if (!ws) return LRKV_ERR_WORKSPACE;
  if (!lrkv::a16(ws)) return LRKV_ERR_INVALID_ARG;
  const int sms = lrkv::device_sm_count();
  if (sms < 1) return LRKV_ERR_CUDA;
  lrkv::DecodePlan P;
  size_t need = 0;
  if ((st = lrkv::rope_make_plan(*dims, sms, P, &need)) != LRKV_OK) return st;
  if (ws_bytes < need) return LRKV_ERR_WORKSPACE;
  lrkv::decode_bind_workspace(P, ws);
  P.q = q_rot; P.k_s = k_s; P.v_s = v_s; P.z_k = z_k; P.z_v = z_v; P.b_k = b_k; P.b_v = b_v;
  P.seq_lens = seq_lens; P.out = out; P.lse = lse;
  P.rope_cs = cos_sin; P.rope_max_pos = max_pos;

  CUtensorMap tm_k, tm_v, tm_zk, tm_zv, tm_cs;
  std::memset(&tm_k, 0, sizeof(tm_k)); std::memset(&tm_v, 0, sizeof(tm_v));
  std::memset(&tm_zk, 0, sizeof(tm_zk)); std::memset(&tm_zv, 0, sizeof(tm_zv));
  std::memset(&tm_cs, 0, sizeof(tm_cs));
  const uint64_t row = static_cast<uint64_t>(P.H) * P.r * 2;
  const uint64_t zdims[4] = {static_cast<uint64_t>(P.segw), static_cast<uint64_t>(P.max_len),
                             static_cast<uint64_t>(P.H / P.hs), static_cast<uint64_t>(P.B)};
  const uint64_t zstr[3] = {row, static_cast<uint64_t>(P.segw) * 2, row * P.max_len};
  const uint32_t zbox[4] = {static_cast<uint32_t>(P.segp), static_cast<uint32_t>(lrkv::kRT),
                            static_cast<uint32_t>(P.nsb), 1u};
  if (!lrkv::make_tmap_3d_bf16(&tm_k, k_s, P.dh, P.max_len, P.B, 64, lrkv::kRT, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !lrkv::make_tmap_3d_bf16(&tm_v, v_s, P.dh, P.max_len, P.B, 64, lrkv::kRT, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !lrkv::make_tmap_4d_bf16_strided(&tm_zk, z_k, zdims, zstr, zbox) ||
      !lrkv::make_tmap_4d_bf16_strided(&tm_zv, z_v, zdims, zstr, zbox) ||
      !lrkv::make_tmap_2d_f32(&tm_cs, cos_sin, P.dh, static_cast<uint64_t>(max_pos), P.cs_row, lrkv::kRT))
    return LRKV_ERR_CUDA;
  const lrkv::RopeFn kern = lrkv::rope_fn(P.dh, P.r);
  if (lrkv::ensure_kernel_smem(reinterpret_cast<const void*>(kern), P.smem_bytes, true) != cudaSuccess)
    return LRKV_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid, P.mt);
  cfg.blockDim = dim3(lrkv::kRThreads);
  cfg.dynamicSmemBytes = P.smem_bytes;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, P, tm_k, tm_v, tm_zk, tm_zv, tm_cs) != cudaSuccess) return LRKV_ERR_CUDA;
  return lrkv::decode_merge_launch(P, stream, true);
}

}  // extern "C"
