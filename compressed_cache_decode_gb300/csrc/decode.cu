// decode.cu — split-KV decode against the factored LRKV cache (sm_103a).
//
// One decode step computes, for every sequence b and head h,
//   s_j = scale * (q_h . k_s,j + p_h . z_k,h,j),   p_h = q_h B_h^K
//   o_h = sum_j a_j v_s,j + (sum_j a_j z_v,h,j) (B_h^V)^T,  a = softmax(s)
// ("Low-Rank Key Value Attention | What a shared cache can preserve", §3,
// Algorithm 2 and the fused online-softmax paragraph; "Low-Rank Key Value
// Attention：中文研读笔记", §2.4, Eqs. (6)-(7)).  Three kernels:
//
//  absorb   p_h = q_h B_h^K in fp32 (Algorithm 2 step 02); resets the status.
//  split    the HBM-bound scan.  The concatenated histories of all sequences
//           are cut into `grid` equal token ranges, one per CTA, so any mix of
//           lengths keeps every SM busy.  A CTA streams its rows through a
//           ring of shared-memory stages filled by TMA: the shared rows k_s,
//           v_s as swizzled tensor tiles (read from HBM once for all H heads,
//           the reuse the review's roofline paragraph asks for) and the
//           latent rows as one bulk copy per tile.  Per tile:
//             A  shared scores on the tensor cores (bf16 mma.sync, heads are
//                the M dimension) and private scores p_h . z_k (fp32 FMA, one
//                thread per head and token group);
//             B  ONE online-softmax update per head over the summed scores,
//                and the private value sum, each value column owned by one
//                thread (no cross-thread merge);
//             C  shared values on the tensor cores, the accumulators rescaled
//                by the same factor as the private ones.
//           At the end of each (sequence, range) piece it writes the
//           unnormalised partial (m, l, acc_s, acc_z).
//  combine  merges the pieces of a sequence with the log-sum-exp rule, divides
//           by the denominator and maps the private sum through (B_h^V)^T
//           once (Algorithm 2 steps 06-09).
//
// The launches are chained with programmatic dependent launch, so the split
// kernel starts streaming the cache while absorb still runs.
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "decode_common.cuh"
#include "decode_plan.h"
#include "host_cache.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lrkv {

using namespace dec;

lrkv_status stream_plan(DecodePlan& P);
lrkv_status stream_prepare(const DecodePlan& P, CUtensorMap* tm_zk, CUtensorMap* tm_zv, CUtensorMap* tm_ks);
lrkv_status stream_launch(const DecodePlan& P, cudaStream_t stream, bool pdl, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, const CUtensorMap& tm_zk, const CUtensorMap& tm_zv,
                          const CUtensorMap& tm_ks);

namespace {

// Producer (one thread): the copies of one tile into stage `st`.
template <bool BF16>
__device__ __forceinline__ void issue_tile(const DecodePlan& P, const CUtensorMap* tm_k,
                                           const CUtensorMap* tm_v, unsigned char* st, uint64_t* bar,
                                           const TileWalk& w) {
  const int nvalid = min(P.T, w.t_end - w.t0);
  unsigned char* ks = st;
  unsigned char* vs = ks + P.kv_bytes;
  unsigned char* zk = vs + P.kv_bytes;
  unsigned char* zv = zk + P.z_bytes;
  const size_t row0 = static_cast<size_t>(w.b) * P.max_len + w.t0;
  const uint32_t zbytes = P.r > 0 ? static_cast<uint32_t>(nvalid) * P.z_row : 0u;
  fence_proxy_async_smem();
  if constexpr (BF16) {
    // full boxes (rows past the tensor end arrive as zeros)
    mbar_arrive_expect_tx(bar, 2u * P.T * P.dh * 2u + 2u * zbytes);
    for (int bx = 0; bx < P.nbox; ++bx) {
      tma_load_3d(ks + bx * P.T * P.span, tm_k, bx * P.box_cols, w.t0, w.b, bar);
      tma_load_3d(vs + bx * P.T * P.span, tm_v, bx * P.box_cols, w.t0, w.b, bar);
    }
  } else {
    const uint32_t kvb = static_cast<uint32_t>(nvalid) * P.dh * 4u;
    mbar_arrive_expect_tx(bar, 2u * kvb + 2u * zbytes);
    tma_load_1d(ks, static_cast<const unsigned char*>(P.k_s) + row0 * P.dh * 4, kvb, bar);
    tma_load_1d(vs, static_cast<const unsigned char*>(P.v_s) + row0 * P.dh * 4, kvb, bar);
  }
  if (zbytes) {
    tma_load_1d(zk, static_cast<const unsigned char*>(P.z_k) + row0 * P.z_row, zbytes, bar);
    tma_load_1d(zv, static_cast<const unsigned char*>(P.z_v) + row0 * P.z_row, zbytes, bar);
  }
}

}  // namespace

// ===================================================================== absorb
// grid = (H, ceil(B / kAbsorbSeq)), block = 256: B_h^K and the q rows of up
// to kAbsorbSeq sequences staged in shared memory, then one output
// p_{b,h,c} = q_{b,h} . B_h^K[:, c] per thread.
constexpr int kAbsorbSeq = 8;
constexpr int kCombineCtas = 16;  // SMs the streaming scan leaves to the merge
constexpr long long kLargeCacheBytes = 256ll << 20;  // see decode_make_plan

template <bool BF16>
__global__ void __launch_bounds__(256) lrkv_decode_absorb_kernel(const DecodePlan P) {
  extern __shared__ __align__(16) float absm[];  // B_h^K [dh][r] | q rows [kAbsorbSeq][dh]
  pdl_trigger();
  const int h = blockIdx.x, b0 = blockIdx.y * kAbsorbSeq, tid = threadIdx.x;
  if (h == 0 && blockIdx.y == 0 && tid == 0) *P.status = 0u;
  const int dh = P.dh, r = P.r, H = P.H;
  const int nb = min(kAbsorbSeq, P.B - b0);
  if (r == 0) return;
  float* bks = absm;
  float* qs = absm + dh * r;
  const size_t base = static_cast<size_t>(h) * dh * r;
  for (int i = tid; i < dh * r; i += blockDim.x) bks[i] = load_elem(P.b_k, base + i, BF16);
  for (int i = tid; i < nb * dh; i += blockDim.x) {
    const int bb = i / dh, k = i % dh;
    qs[i] = load_elem(P.q, (static_cast<size_t>(b0 + bb) * H + h) * dh + k, BF16);
  }
  __syncthreads();
  for (int idx = tid; idx < nb * r; idx += blockDim.x) {
    const int bb = idx / r, c = idx % r;
    const float* qr = qs + bb * dh;
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
    int k = 0;
    for (; k + 3 < dh; k += 4) {
      a0 = fmaf(qr[k], bks[k * r + c], a0);
      a1 = fmaf(qr[k + 1], bks[(k + 1) * r + c], a1);
      a2 = fmaf(qr[k + 2], bks[(k + 2) * r + c], a2);
      a3 = fmaf(qr[k + 3], bks[(k + 3) * r + c], a3);
    }
    for (; k < dh; ++k) a0 = fmaf(qr[k], bks[k * r + c], a0);
    P.p_abs[(static_cast<size_t>(b0 + bb) * H + h) * r + c] = (a0 + a1) + (a2 + a3);
  }
}

// ====================================================================== split
// Thread roles (H heads, 256 threads):
//   score role   (ha, tg) = (tid % H, tid / H), tg < ntg: the private score
//                p_h . z_k of tokens tg, tg + ntg, ... and (fp32) the shared
//                score, the softmax weights of those tokens, and a partial
//                denominator;
//   value role   (hb, rg) = (tid % H, tid / H), rg < nrg: value columns
//                [rg*cw, rg*cw + cw) of the private sum (fp32: of [shared |
//                private]) over every token of the tile;
//   MMA role     warps: shared scores and shared values on the tensor cores.
// Weights are taken against a per-head reference max m_ref.  A tile whose
// scores all stay below m_ref + 8 (log2 domain, weights <= 256) needs no
// rescale; otherwise (always on a piece's first tile) the tile max is reduced
// across the head's threads and every accumulator is rescaled once.  This is
// the online softmax of the review's fused variant with the rescale taken
// only when it is needed.
template <bool BF16, int RMAX, int NE>
__global__ void __launch_bounds__(kThreads, 1)
    lrkv_decode_split_kernel(const DecodePlan P, const __grid_constant__ CUtensorMap tm_k,
                             const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_bad;
  __shared__ int s_timeout;
  // the swizzled TMA boxes need 1024-byte-aligned destinations
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int B = P.B, H = P.H, dh = P.dh, r = P.r, T = P.T;
  constexpr int ESZ = BF16 ? 2 : 4;
  constexpr float kHeadroom = 8.f;  // log2 units

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  int* pre = reinterpret_cast<int*>(smem + P.off_prefix);
  unsigned char* q_sh = smem + P.off_q;
  float* s_sh = reinterpret_cast<float*>(smem + P.off_ssh);   // shared scores [T][s_stride]
  float* wf_sh = reinterpret_cast<float*>(smem + P.off_sp);   // fp32 weights [T][s_stride]
  __nv_bfloat16* w_sh = reinterpret_cast<__nv_bfloat16*>(smem + P.off_w);  // bf16 weights [Hp][w_stride]
  float* alpha_sh = reinterpret_cast<float*>(smem + P.off_alpha);  // [Hp]
  float* red_sh = reinterpret_cast<float*>(smem + P.off_red);      // [ntg][H]
  unsigned char* stages = smem + P.off_stage;

  // ---- 1. sequence starts (clamped lengths) --------------------------------
  if (tid == 0) { s_bad = 0; s_timeout = 0; }
  __syncthreads();
  for (int b = tid; b < B; b += blockDim.x) {
    int L = P.seq_lens[b];
    if (L < 0 || L > P.max_len) {
      s_bad = 1;
      L = min(max(L, 0), P.max_len);
    }
    pre[b + 1] = L;
  }
  if (tid == 0) pre[0] = 0;
  __syncthreads();
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
  if (blockIdx.x == 0) {
    for (int b = tid; b <= B; b += blockDim.x) P.prefix[b] = pre[b];
    if (tid == 0) { P.meta[0] = N; P.meta[1] = G; }
  }
  if (N == 0 || static_cast<int>(blockIdx.x) >= G) {
    if (s_bad && tid == 0) { pdl_wait(); record_status(P.status, kDevBounds); }
    return;
  }
  const int c = blockIdx.x;
  const int g0 = static_cast<int>(static_cast<long long>(c) * N / G);
  const int g1 = static_cast<int>(static_cast<long long>(c + 1) * N / G);

  // ---- 2. barriers, constant tiles, first copies ---------------------------
  if (tid == 0) {
    for (int s = 0; s < P.stages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  if constexpr (BF16) {
    for (int i = tid; i < P.Hp; i += blockDim.x) alpha_sh[i] = 1.f;
    for (int i = tid; i < P.Hp * P.w_stride; i += blockDim.x) w_sh[i] = __float2bfloat16(0.f);
  }
  __syncthreads();

  TileWalk pw;  // producer walk (thread 0)
  bool p_more = walk_first(pw, pre, B, g0, g1);
  int issued = 0;
  if (tid == 0) {
    for (int s = 0; s < P.stages && p_more; ++s) {
      issue_tile<BF16>(P, &tm_k, &tm_v, stages + static_cast<size_t>(s) * P.stage_bytes, &bars[s], pw);
      ++issued;
      p_more = walk_next(pw, pre, B, g1, T);
    }
  }

  // the absorb kernel's output (p) is read only after this point
  pdl_wait();
  if (s_bad && tid == 0) record_status(P.status, kDevBounds);

  // ---- 3. thread roles -----------------------------------------------------
  const int ha = tid % H, tg = tid / H;
  const bool a_active = tg < P.ntg;
  const int hb = ha, rg = tg;
  const bool b_active = rg < P.nrg;
  const int g = lane >> 2, q4 = lane & 3;  // MMA fragment coordinates
  const int mt = P.Hp / 16;
  const int n_vtiles = BF16 ? mt * (dh / 8) : 0;
  const int ltiles = BF16 ? mt * (T / 8) : 0;
  const int vw = BF16 ? r : dh + r;  // width of the per-thread value space
  const int col0 = rg * P.cw;

  float p_reg[RMAX];     // q_h B_h^K of head ha (this piece's sequence)
  float acc_c[kMaxCW];   // value columns owned by (hb, rg)
  float acc_v[kMaxValueTiles][4];  // shared-value MMA fragments (bf16)
  float m_ref = -INFINITY;  // reference max of head ha (identical in all its threads)
  float l_part = 0.f;       // denominator over this thread's tokens
#pragma unroll
  for (int i = 0; i < RMAX; ++i) p_reg[i] = 0.f;
#pragma unroll
  for (int i = 0; i < kMaxCW; ++i) acc_c[i] = 0.f;
#pragma unroll
  for (int j = 0; j < kMaxValueTiles; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc_v[j][k] = 0.f;

  TileWalk cw;
  walk_first(cw, pre, B, g0, g1);
  bool seg_start = true;
  int it = 0;
  bool ok = true;

  while (true) {
    const int s = it % P.stages;
    const uint32_t parity = static_cast<uint32_t>(it / P.stages) & 1u;
    unsigned char* ks = stages + static_cast<size_t>(s) * P.stage_bytes;
    unsigned char* vs = ks + P.kv_bytes;
    unsigned char* zk = vs + P.kv_bytes;
    unsigned char* zv = zk + P.z_bytes;
    const int nvalid = min(T, cw.t_end - cw.t0);
    // this thread's tokens in the score role: tg, tg + ntg, ... (< nvalid)
    const int nmine = (a_active && nvalid > tg) ? (nvalid - tg + P.ntg - 1) / P.ntg : 0;

    // ---- piece set-up: q (shared scores) and p (private scores) -----------
    if (seg_start) {
      const int b = cw.b;
      if constexpr (BF16) {
        const uint4* gq = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(P.q) +
                                                         static_cast<size_t>(b) * H * dh);
        const int cpr = dh / 8;
        for (int i = tid; i < P.Hp * cpr; i += blockDim.x) {
          const int hh = i / cpr, k8 = i % cpr;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (hh < H) v = gq[hh * cpr + k8];
          *reinterpret_cast<uint4*>(q_sh + (hh * P.q_stride + k8 * 8) * 2) = v;
        }
      } else {
        const float* gq = static_cast<const float*>(P.q) + static_cast<size_t>(b) * H * dh;
        float* qf = reinterpret_cast<float*>(q_sh);
        for (int i = tid; i < H * dh; i += blockDim.x) qf[(i / dh) * P.q_stride + (i % dh)] = gq[i];
      }
      if (a_active && r > 0) {
        const float* gp = P.p_abs + (static_cast<size_t>(b) * H + ha) * r;
#pragma unroll
        for (int c4 = 0; c4 < RMAX; c4 += 4) {
          if (c4 < r) {
            const float4 v = *reinterpret_cast<const float4*>(gp + c4);
            p_reg[c4] = v.x; p_reg[c4 + 1] = v.y; p_reg[c4 + 2] = v.z; p_reg[c4 + 3] = v.w;
          }
        }
      }
      __syncthreads();
      seg_start = false;
    }

    // ---- wait for the tile (bounded; every thread observes the barrier) ----
    const bool got = mbar_wait_bounded(&bars[s], parity);
    if (!got) s_timeout = 1;

    // ---- phase A: scores ----------------------------------------------------
    float sc[kMaxPPT];  // this thread's summed, scaled scores (log2 domain)
#pragma unroll
    for (int i = 0; i < kMaxPPT; ++i) sc[i] = 0.f;
    if (got) {
      if constexpr (BF16) {
        // rows past the piece's end must hold zeros before the value MMA
        if (nvalid < T) {
          const int cpr = P.span / 16;  // 16-byte chunks per box row
          const int per = (T - nvalid) * cpr;
          for (int i = tid; i < P.nbox * per; i += blockDim.x) {
            const int bx = i / per, rem = i % per;
            const int row = nvalid + rem / cpr, ch = rem % cpr;
            *reinterpret_cast<uint4*>(vs + bx * T * P.span + row * P.span + ch * 16) = make_uint4(0, 0, 0, 0);
          }
          fence_proxy_async_smem();
        }
        for (int item = warp; item < ltiles; item += nwarps) {
          const int mi = item / (T / 8), nj = item % (T / 8);
          float d[4] = {0.f, 0.f, 0.f, 0.f};
          const int trow = nj * 8 + (lane & 7);
          for (int kk = 0; kk < dh / 16; ++kk) {
            uint32_t a0, a1, a2, a3, b0, b1;
            ldsm_x4(a0, a1, a2, a3, q_sh + ((mi * 16 + (lane & 15)) * P.q_stride + kk * 16 + (lane >> 4) * 8) * 2);
            const int k0 = kk * 16 + ((lane >> 3) & 1) * 8;
            const int bx = k0 / P.box_cols, ch = (k0 % P.box_cols) / 8;
            ldsm_x2(b0, b1, ks + bx * T * P.span + swz_off(trow, ch, P.span));
            mma_bf16_16816(d, a0, a1, a2, a3, b0, b1);
          }
          const int h0 = mi * 16 + g, t0 = nj * 8 + 2 * q4;
          s_sh[t0 * P.s_stride + h0] = d[0];
          s_sh[(t0 + 1) * P.s_stride + h0] = d[1];
          s_sh[t0 * P.s_stride + h0 + 8] = d[2];
          s_sh[(t0 + 1) * P.s_stride + h0 + 8] = d[3];
        }
      }
      if (nmine > 0) {
        const unsigned char* zrow = zk + ha * r * ESZ;
#pragma unroll
        for (int i = 0; i < kMaxPPT; ++i) {
          if (i < nmine) {
            const int t = tg + i * P.ntg;
            float part[4] = {0.f, 0.f, 0.f, 0.f};
            if (r > 0) {
              const unsigned char* zt = zrow + static_cast<size_t>(t) * P.z_row;
#pragma unroll
              for (int c0 = 0; c0 < RMAX; c0 += NE) {
                if (c0 < r) {
                  float zv4[NE];
                  load_vec<BF16, NE>(zt + c0 * ESZ, zv4);
#pragma unroll
                  for (int e = 0; e < NE; ++e) part[e & 3] = fmaf(zv4[e], p_reg[c0 + e], part[e & 3]);
                }
              }
            }
            if constexpr (!BF16) {
              const float* qh = reinterpret_cast<const float*>(q_sh) + ha * P.q_stride;
              const float* kt = reinterpret_cast<const float*>(ks) + t * dh;
              for (int k = 0; k < dh; k += 4) {
                const float4 x = *reinterpret_cast<const float4*>(qh + k);
                const float4 y = *reinterpret_cast<const float4*>(kt + k);
                part[0] = fmaf(x.x, y.x, part[0]); part[1] = fmaf(x.y, y.y, part[1]);
                part[2] = fmaf(x.z, y.z, part[2]); part[3] = fmaf(x.w, y.w, part[3]);
              }
            }
            sc[i] = (part[0] + part[1]) + (part[2] + part[3]);
          }
        }
      }
    }
    __syncthreads();  // (#1) shared scores in shared memory; everyone left the previous tile
    if (s_timeout) { ok = false; break; }
    if (tid == 0 && it > 0 && p_more) {  // refill the stage the previous tile used
      const int sp = (it - 1) % P.stages;
      issue_tile<BF16>(P, &tm_k, &tm_v, stages + static_cast<size_t>(sp) * P.stage_bytes, &bars[sp], pw);
      ++issued;
      p_more = walk_next(pw, pre, B, g1, T);
    }

    // ---- phase B: weights against the reference max --------------------------
    bool need = false;
    float mloc = -INFINITY;
#pragma unroll
    for (int i = 0; i < kMaxPPT; ++i) {
      if (i < nmine) {
        const int t = tg + i * P.ntg;
        float v = sc[i];
        if constexpr (BF16) v += s_sh[t * P.s_stride + ha];
        v *= P.scale_log2;
        sc[i] = v;
        mloc = fmaxf(mloc, v);
      }
    }
    need = mloc > m_ref + kHeadroom;
    auto write_weights = [&](float mref) {
      float lsum = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPPT; ++i) {
        if (i < nmine) {
          const int t = tg + i * P.ntg;
          const float w = exp2f(sc[i] - mref);
          lsum += w;
          wf_sh[t * P.s_stride + ha] = w;
          if constexpr (BF16) w_sh[ha * P.w_stride + t] = __float2bfloat16(w);
        }
      }
      return lsum;
    };
    float lsum = 0.f;
    if (!need) lsum = write_weights(m_ref);
    // rows past the piece's end carry zero weight
    if (a_active) {
      for (int t = nvalid + tg; t < T; t += P.ntg) {
        wf_sh[t * P.s_stride + ha] = 0.f;
        if constexpr (BF16) w_sh[ha * P.w_stride + t] = __float2bfloat16(0.f);
      }
    }
    if (__syncthreads_or(need)) {  // (#2) rare: some head's max moved up
      if (a_active) red_sh[tg * H + ha] = mloc;
      __syncthreads();
      float alpha = 1.f;
      if (a_active || b_active) {
        float mt_ = -INFINITY;
        for (int k = 0; k < P.ntg; ++k) mt_ = fmaxf(mt_, red_sh[k * H + ha]);
        const float m_new = fmaxf(m_ref, mt_);
        alpha = exp2f(m_ref - m_new);  // 0 on a piece's first tile
        m_ref = m_new;
      }
      if (a_active) {
        l_part *= alpha;
        lsum = write_weights(m_ref);
        if (BF16 && tg == 0) alpha_sh[ha] = alpha;
      }
      if (b_active) {
#pragma unroll
        for (int i = 0; i < kMaxCW; ++i) acc_c[i] *= alpha;
      }
      __syncthreads();
      if constexpr (BF16) {
#pragma unroll
        for (int j = 0; j < kMaxValueTiles; ++j) {
          const int vt = warp + j * nwarps;
          if (vt < n_vtiles) {
            const int mi = vt / (dh / 8);
            const float a_lo = alpha_sh[mi * 16 + g], a_hi = alpha_sh[mi * 16 + g + 8];
            acc_v[j][0] *= a_lo; acc_v[j][1] *= a_lo; acc_v[j][2] *= a_hi; acc_v[j][3] *= a_hi;
          }
        }
      }
    }
    l_part += lsum;

    // ---- phase C: values ----------------------------------------------------
    if constexpr (BF16) {
#pragma unroll
      for (int j = 0; j < kMaxValueTiles; ++j) {
        const int vt = warp + j * nwarps;
        if (vt < n_vtiles) {
          const int mi = vt / (dh / 8), nt = vt % (dh / 8);
          const unsigned char* wrow = reinterpret_cast<const unsigned char*>(w_sh) +
                                      (mi * 16 + (lane & 15)) * P.w_stride * 2;
          const int n0 = nt * 8;
          const unsigned char* vbox = vs + (n0 / P.box_cols) * T * P.span;
          const int ch = (n0 % P.box_cols) / 8;
          if ((T & 15) == 0) {
            for (int kk = 0; kk < T / 16; ++kk) {
              uint32_t a0, a1, a2, a3, b0, b1;
              ldsm_x4(a0, a1, a2, a3, wrow + (kk * 16 + (lane >> 4) * 8) * 2);
              ldsm_x2_trans(b0, b1, vbox + swz_off(kk * 16 + (lane & 15), ch, P.span));
              mma_bf16_16816(acc_v[j], a0, a1, a2, a3, b0, b1);
            }
          } else {
            uint32_t a0, a1, b0;
            ldsm_x2(a0, a1, wrow);
            ldsm_x1_trans(b0, vbox + swz_off(lane & 7, ch, P.span));
            mma_bf16_1688(acc_v[j], a0, a1, b0);
          }
        }
      }
    }
    if (b_active && vw > 0) {
      for (int t = 0; t < nvalid; ++t) {
        const float w = wf_sh[t * P.s_stride + hb];
        if constexpr (BF16) {
          const unsigned char* zt = zv + static_cast<size_t>(t) * P.z_row + (hb * r + col0) * ESZ;
#pragma unroll
          for (int c0 = 0; c0 < kMaxCW; c0 += NE) {
            if (c0 < P.cw && col0 + c0 < r) {
              float zv4[NE];
              load_vec<BF16, NE>(zt + c0 * ESZ, zv4);
#pragma unroll
              for (int e = 0; e < NE; ++e) acc_c[c0 + e] = fmaf(w, zv4[e], acc_c[c0 + e]);
            }
          }
        } else {
#pragma unroll
          for (int c0 = 0; c0 < kMaxCW; c0 += 4) {
            const int col = col0 + c0;
            if (c0 < P.cw && col < vw) {
              const unsigned char* src = col < dh
                  ? vs + (static_cast<size_t>(t) * dh + col) * 4
                  : zv + static_cast<size_t>(t) * P.z_row + (hb * r + col - dh) * 4;
              float x4[4];
              load_vec<false, 4>(src, x4);
#pragma unroll
              for (int e = 0; e < 4; ++e) acc_c[c0 + e] = fmaf(w, x4[e], acc_c[c0 + e]);
            }
          }
        }
      }
    }

    // ---- end of a (sequence, range) piece: write the partial ---------------
    const bool last_of_piece = cw.t0 + T >= cw.t_end;
    if (last_of_piece) {
      const int slot = cw.b + c;
      float* pacc = P.part_acc + static_cast<size_t>(slot) * H * (dh + r);
      __syncthreads();  // red_sh may still be read by the rescale above
      if (a_active) red_sh[tg * H + ha] = l_part;
      __syncthreads();
      if (a_active && tg == 0) {
        float l_tot = 0.f;
        for (int k = 0; k < P.ntg; ++k) l_tot += red_sh[k * H + ha];
        P.part_ml[(static_cast<size_t>(slot) * H + ha) * 2 + 0] = m_ref;
        P.part_ml[(static_cast<size_t>(slot) * H + ha) * 2 + 1] = l_tot;
      }
      if (b_active) {
        const int off = BF16 ? dh : 0;  // bf16: the columns are private ones
#pragma unroll
        for (int i = 0; i < kMaxCW; ++i)
          if (i < P.cw && col0 + i < vw) pacc[hb * (dh + r) + off + col0 + i] = acc_c[i];
      }
      if constexpr (BF16) {
#pragma unroll
        for (int j = 0; j < kMaxValueTiles; ++j) {
          const int vt = warp + j * nwarps;
          if (vt < n_vtiles) {
            const int mi = vt / (dh / 8), nt = vt % (dh / 8);
            const int h0 = mi * 16 + g, col = nt * 8 + 2 * q4;
            if (h0 < H) { pacc[h0 * (dh + r) + col] = acc_v[j][0]; pacc[h0 * (dh + r) + col + 1] = acc_v[j][1]; }
            if (h0 + 8 < H) { pacc[(h0 + 8) * (dh + r) + col] = acc_v[j][2]; pacc[(h0 + 8) * (dh + r) + col + 1] = acc_v[j][3]; }
          }
        }
      }
      m_ref = -INFINITY;
      l_part = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxCW; ++i) acc_c[i] = 0.f;
#pragma unroll
      for (int j = 0; j < kMaxValueTiles; ++j)
#pragma unroll
        for (int k = 0; k < 4; ++k) acc_v[j][k] = 0.f;
      seg_start = true;
    }

    ++it;
    if (!walk_next(cw, pre, B, g1, T)) break;
    if (seg_start) __syncthreads();  // q/p of the next piece overwrite the old ones
  }

  pdl_trigger();
  if (!ok) {
    // a tile never arrived: report, drain what is still in flight, return
    if (tid == 0) {
      record_status(P.status, kDevTimeout);
      for (int j = it; j < issued; ++j)
        mbar_wait_bounded(&bars[j % P.stages], static_cast<uint32_t>(j / P.stages) & 1u, kWaitLimitCycles / 8);
    }
    __syncthreads();
  }
}

// ==================================================================== combine
// One warp per (sequence b, head h), grid-stride over the pairs (the grid
// is kept small, so that the streaming scan can leave it a few SMs of its
// own and the next step's scan starts beside it): the pieces
// (m_i, l_i, acc_i) merged with the log-sum-exp rule, then the lift
// o = acc_s / L + (acc_z / L) (B_h^V)^T and lse = (M + log2 L) ln 2
// (Algorithm 2 steps 06-09).  Lane j owns columns j + 32 k of
// [acc_s | acc_z] and merges them over every piece in one pass (8-32 pieces
// of loads in flight, the running maximum raised as it goes; m_i, l_i are read
// by every lane of the warp at once).  The first pair's B_h^V rows are an
// input, loaded before the wait on the scan kernel when they fit in
// registers.
constexpr int kCombineWarps = 8;
constexpr int kCombineLocalB = 256;  // up to this batch, a warp finds its sequence's pieces from seq_lens
constexpr int kCombinePre = 32;  // B^V words a lane may hold (2 rows of r <= 32)

template <bool BF16, int KC>  // KC: columns per lane, ceil((dh + r) / 32)
__global__ void __launch_bounds__(32 * kCombineWarps) lrkv_decode_combine_kernel(const DecodePlan P) {
  extern __shared__ __align__(16) unsigned char csmem[];
  constexpr int kCombinePieces = KC <= 3 ? 32 : KC <= 6 ? 16 : 8;  // pieces of loads in flight
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = P.H, dh = P.dh, r = P.r, W = dh + r;
  float* zbar = reinterpret_cast<float*>(csmem) + warp * max(r, 1);  // [r] per warp
  const int nmax = P.grid * P.ngw;                                     // partials of one sequence, at most
  float* wts = reinterpret_cast<float*>(csmem) + kCombineWarps * max(r, 1) + warp * 2 * nmax;  // [nmax] per warp
  float* lsm = wts + nmax;                                                                     // [nmax] per warp
  const long long npairs = static_cast<long long>(P.B) * H;
  const long long wstride = static_cast<long long>(gridDim.x) * kCombineWarps;
  long long bh = static_cast<long long>(blockIdx.x) * kCombineWarps + warp;
  const int nd = (dh + 31) / 32;  // output rows d = lane + 32 k of this lane
  const bool pre_bv = BF16 && nd <= 2 && r <= 32;
  uint32_t bvp[kCombinePre];
  auto load_bv = [&](int h) {
#pragma unroll
    for (int i = 0; i < kCombinePre; ++i) {
      const int k = i / 16, c2 = i % 16, d = lane + 32 * k;
      bvp[i] = (k < nd && d < dh && 2 * c2 < r)
                   ? reinterpret_cast<const uint32_t*>(static_cast<const __nv_bfloat16*>(P.b_v) +
                                                       (static_cast<size_t>(h) * dh + d) * r)[c2]
                   : 0u;
    }
  };
  if (pre_bv && bh < npairs) load_bv(static_cast<int>(bh % H));
  // the first pair's sequence range and the scan's CTA count, from seq_lens
  // (an input) the way the scan derives them, before the wait
  const bool local = P.stream && P.B <= kCombineLocalB;
  int l_start = 0, l_end = 0;
  long long l_N = 0;
  auto locate = [&](int b) {
    int before = 0, mine = 0, total = 0;
    for (int b0 = 0; b0 < P.B; b0 += 32) {
      const int bb = b0 + lane;
      const int L = bb < P.B ? min(max(P.seq_lens[bb], 0), P.max_len) : 0;
      int x = bb < b ? L : 0, y = bb == b ? L : 0, z = L;
      for (int o2 = 16; o2 > 0; o2 >>= 1) {
        x += __shfl_xor_sync(0xffffffffu, x, o2);
        y += __shfl_xor_sync(0xffffffffu, y, o2);
        z += __shfl_xor_sync(0xffffffffu, z, o2);
      }
      before += x; mine += y; total += z;
    }
    l_start = before; l_end = before + mine; l_N = total;
  };
  if (local && bh < npairs) locate(static_cast<int>(bh / H));
  pdl_trigger();  // the next step's scan may launch (it waits before it writes)
  pdl_wait();
  const long long N = local ? l_N : P.meta[0];
  const long long G = local ? max(1ll, min(static_cast<long long>(P.grid), (N + P.min_tokens - 1) / max(P.min_tokens, 1)))
                            : P.meta[1];
  for (bool first = true; bh < npairs; bh += wstride, first = false) {
    const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
    if (!first) {
      if (pre_bv) load_bv(h);
      if (local) locate(b);
    }
    float* o = P.out + (static_cast<size_t>(b) * H + h) * dh;
    const int start = local ? l_start : P.prefix[b], end = local ? l_end : P.prefix[b + 1];
    if (end <= start) {
      for (int k = lane; k < dh; k += 32) o[k] = 0.f;
      if (lane == 0 && P.lse) P.lse[static_cast<size_t>(b) * H + h] = -INFINITY;
      continue;
    }
    const int c0 = cta_of_token(start, N, G), c1 = cta_of_token(end - 1, N, G);
    const int n = (c1 - c0 + 1) * P.ngw;                    // partials of this sequence
    const size_t s0 = static_cast<size_t>(b + c0) * P.ngw;  // first of them
    const float* ml = P.part_ml + (s0 * H + h) * 2;
    const float* acc0 = P.part_acc + (s0 * H + h) * W;
    const size_t mstep = static_cast<size_t>(H) * 2, astep = static_cast<size_t>(H) * W;
    // 1. the partials' weights 2^(m_i - M) against the largest maximum M,
    //    the lanes taking the partials in turn (kept in shared memory)
    __syncwarp();  // the previous pair's weight reads are done
    float M = -INFINITY;
#pragma unroll 4
    for (int i = lane; i < n; i += 32) {
      const float m = ml[i * mstep];
      wts[i] = m;
      lsm[i] = ml[i * mstep + 1];
      M = fmaxf(M, m);
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o2));
    float L = 0.f;
    for (int i = lane; i < n; i += 32) {
      const float m = wts[i];
      const float w = m == -INFINITY ? 0.f : exp2f(m - M);
      wts[i] = w;
      L = fmaf(w, lsm[i], L);
    }
#pragma unroll
    for (int o2 = 16; o2 > 0; o2 >>= 1) L += __shfl_xor_sync(0xffffffffu, L, o2);
    __syncwarp();
    // 2. the weighted sum of the partials' rows (lanes own columns)
    float a[KC];
#pragma unroll
    for (int k = 0; k < KC; ++k) a[k] = 0.f;
    for (int i0 = 0; i0 < n; i0 += kCombinePieces) {
      float vi[kCombinePieces][KC];
#pragma unroll
      for (int u = 0; u < kCombinePieces; ++u) {
        const bool ok = i0 + u < n;
#pragma unroll
        for (int k = 0; k < KC; ++k) {
          const int j = lane + 32 * k;
          vi[u][k] = (ok && j < W) ? acc0[(i0 + u) * astep + j] : 0.f;
        }
      }
#pragma unroll
      for (int u = 0; u < kCombinePieces; ++u) {
        const float w = i0 + u < n ? wts[i0 + u] : 0.f;
#pragma unroll
        for (int k = 0; k < KC; ++k) a[k] = fmaf(w, vi[u][k], a[k]);
      }
    }
    const float inv_l = 1.f / L;
    __syncwarp();  // the previous pair's zbar reads are done
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const int j = lane + 32 * k;
      if (j >= dh && j < W) zbar[j - dh] = a[k] * inv_l;
    }
    __syncwarp();
#pragma unroll
    for (int k = 0; k < KC; ++k) {
      const int d = lane + 32 * k;
      if (d >= dh) continue;
      float v = a[k] * inv_l;
      if (pre_bv) {
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) {
          const int i = k * 16 + c2;
          if (i < kCombinePre && 2 * c2 < r) {
            v = fmaf(bf_lo(bvp[i]), zbar[2 * c2], v);
            v = fmaf(bf_hi(bvp[i]), zbar[2 * c2 + 1], v);
          }
        }
      } else {
        const size_t base = (static_cast<size_t>(h) * dh + d) * r;
        for (int cc = 0; cc < r; ++cc) v = fmaf(load_elem(P.b_v, base + cc, BF16), zbar[cc], v);
      }
      o[d] = v;
    }
    if (lane == 0 && P.lse) P.lse[static_cast<size_t>(b) * H + h] = (M + log2f(L)) * kLn2;
  }
  if (P.stream && blockIdx.x == 0 && warp == 0) {
    // the device status of this call: the bits every scan CTA wrote
    uint32_t bits = 0u;
    for (int i = lane; i < P.grid * P.mt; i += 32) bits |= P.cta_status[i];
    for (int o2 = 16; o2 > 0; o2 >>= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, o2);
    if (lane == 0) *P.status = bits;
  }
}

// ================================================================ wide merge
// The merge of the bf16 streaming decode: one CTA per (sequence b, head h),
// grid-stride.  The partials of the sequence's pieces are split over the NW
// warps (warp w takes partials w, w + NW, ...); each warp merges its share in
// one pass against a running maximum, a batch of partials in flight at a time
// (lanes own columns of [acc_s | acc_z]); the CTA merges the warp results
// through shared memory with the same log-sum-exp rule, then lifts the
// private sum: o = acc_s / L + (acc_z / L) (B_h^V)^T (each output column's
// B^V row read with 8-byte loads all in flight) and lse = (M + log2 L) ln 2
// (Algorithm 2 steps 06-09).
constexpr int kWideWarps = 8;  // warps per (sequence, head); 16 for at most 64 pairs

template <bool BF16, int KC, int NW>  // KC: columns per lane, ceil((dh + r) / 32); NW: warps
__global__ void __launch_bounds__(32 * NW) lrkv_decode_merge_wide_kernel(const DecodePlan P) {
  __shared__ float s_m[NW], s_l[NW];
  __shared__ float s_acc[NW][32 * KC];
  __shared__ float s_z[KC * 32];   // acc_z / L (private width <= 32 KC)
  __shared__ float s_os[KC * 32];  // acc_s / L
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int H = P.H, dh = P.dh, r = P.r, W = dh + r;
  pdl_trigger();  // the next step's scan may launch (it waits before it writes)
  pdl_wait();
  const long long N = P.meta[0], G = P.meta[1];
  const long long npairs = static_cast<long long>(P.B) * H;
  const size_t mstep = static_cast<size_t>(H) * 2, astep = static_cast<size_t>(H) * W;
  for (long long bh = blockIdx.x; bh < npairs; bh += gridDim.x) {
    const int b = static_cast<int>(bh / H), h = static_cast<int>(bh % H);
    float* o = P.out + (static_cast<size_t>(b) * H + h) * dh;
    const int start = P.prefix[b], end = P.prefix[b + 1];
    if (end <= start) {
      for (int k = threadIdx.x; k < dh; k += blockDim.x) o[k] = 0.f;
      if (threadIdx.x == 0 && P.lse) P.lse[static_cast<size_t>(b) * H + h] = -INFINITY;
      continue;
    }
    const int c0 = cta_of_token(start, N, G), c1 = cta_of_token(end - 1, N, G);
    const int n = (c1 - c0 + 1) * P.ngw;
    const size_t s0 = static_cast<size_t>(b + c0) * P.ngw;
    const float* ml = P.part_ml + (s0 * H + h) * 2;
    const float* acc0 = P.part_acc + (s0 * H + h) * W;
    // 1. this warp's share in one pass, eight partials' (m, l) and rows in
    //    flight at a time (fewer for wide rows), against a running maximum (raised per batch: the
    //    sums so far are rescaled, the same for every lane)
    float mw = -INFINITY, lw = 0.f;
    float a[KC];
#pragma unroll
    for (int k = 0; k < KC; ++k) a[k] = 0.f;
    constexpr int kBatch = KC <= 3 ? 8 : KC <= 6 ? 6 : KC <= 10 ? 4 : 2;  // registers: kBatch x KC row values
    for (int i0 = warp; i0 < n; i0 += kBatch * NW) {
      float v[kBatch][KC], mv[kBatch], lv[kBatch];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const int i = i0 + u * NW;
        const bool ok = i < n;
        mv[u] = ok ? ml[i * mstep] : -INFINITY;
        lv[u] = ok ? ml[i * mstep + 1] : 0.f;
#pragma unroll
        for (int k = 0; k < KC; ++k) {
          const int j = lane + 32 * k;
          v[u][k] = (ok && j < W) ? acc0[i * astep + j] : 0.f;
        }
      }
      float bm = mv[0];
#pragma unroll
      for (int u = 1; u < kBatch; ++u) bm = fmaxf(bm, mv[u]);
      if (bm > mw) {
        const float sc = mw == -INFINITY ? 0.f : exp2f(mw - bm);
        lw *= sc;
#pragma unroll
        for (int k = 0; k < KC; ++k) a[k] *= sc;
        mw = bm;
      }
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const float wt = mv[u] == -INFINITY ? 0.f : exp2f(mv[u] - mw);
        lw = fmaf(wt, lv[u], lw);
#pragma unroll
        for (int k = 0; k < KC; ++k) a[k] = fmaf(wt, v[u][k], a[k]);
      }
    }
    __syncthreads();  // the previous pair's reads of the shared arrays are done
    if (lane == 0) {
      s_m[warp] = mw;
      s_l[warp] = lw;
    }
#pragma unroll
    for (int k = 0; k < KC; ++k) s_acc[warp][lane + 32 * k] = a[k];
    __syncthreads();
    // 2. the CTA's merge of the warp shares (threads own columns)
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, s_m[w]);
    float sw[NW], L = 0.f;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      sw[w] = s_m[w] == -INFINITY ? 0.f : exp2f(s_m[w] - M);
      L = fmaf(sw[w], s_l[w], L);
    }
    const float inv_l = 1.f / L;
    for (int t = threadIdx.x; t < W; t += blockDim.x) {
      float acc = 0.f;
#pragma unroll
      for (int w = 0; w < NW; ++w) acc = fmaf(sw[w], s_acc[w][t], acc);
      if (t < dh) s_os[t] = acc * inv_l; else s_z[t - dh] = acc * inv_l;
    }
    __syncthreads();
    // 3. the lift through (B_h^V)^T and the outputs: a thread's B^V row read
    //    with 8-byte loads, all in flight at once, where r and the base allow
    const bool vec = BF16 && r % 4 == 0 && r <= 64 && (reinterpret_cast<uintptr_t>(P.b_v) & 7u) == 0;
    for (int t = threadIdx.x; t < dh; t += blockDim.x) {
      float v = s_os[t];
      const size_t base = (static_cast<size_t>(h) * dh + t) * r;
      if (vec) {
        const uint2* row = reinterpret_cast<const uint2*>(static_cast<const __nv_bfloat16*>(P.b_v) + base);
        uint2 w[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) w[q] = 4 * q < r ? row[q] : make_uint2(0u, 0u);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
          if (4 * q < r) {
            v = fmaf(bf_lo(w[q].x), s_z[4 * q], v);
            v = fmaf(bf_hi(w[q].x), s_z[4 * q + 1], v);
            v = fmaf(bf_lo(w[q].y), s_z[4 * q + 2], v);
            v = fmaf(bf_hi(w[q].y), s_z[4 * q + 3], v);
          }
        }
      } else {
        for (int cc = 0; cc < r; ++cc) v = fmaf(load_elem(P.b_v, base + cc, BF16), s_z[cc], v);
      }
      o[t] = v;
    }
    if (threadIdx.x == 0 && P.lse) P.lse[static_cast<size_t>(b) * H + h] = (M + log2f(L)) * kLn2;
  }
  if (blockIdx.x == 0 && warp == 0) {
    // the device status of this call: the bits every scan CTA wrote
    uint32_t bits = 0u;
    for (int i = lane; i < P.grid * P.mt; i += 32) bits |= P.cta_status[i];
    for (int o2 = 16; o2 > 0; o2 >>= 1) bits |= __shfl_xor_sync(0xffffffffu, bits, o2);
    if (lane == 0) *P.status = bits;
  }
}

// ======================================================================= host
namespace {

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  return (v && *v) ? std::atoi(v) : dflt;
}

// The bound of the decode's waits for its copies (SM cycles): the
// environment variable LRKV_WAIT_LIMIT_CYCLES when it holds a positive
// number (for tests of the timeout path), else kWaitLimitCycles.
long long wait_limit_cycles() {
  const char* v = std::getenv("LRKV_WAIT_LIMIT_CYCLES");
  const long long x = (v && *v) ? std::atoll(v) : 0;
  return x > 0 ? x : kWaitLimitCycles;
}

using SplitFn = void (*)(const DecodePlan, const CUtensorMap, const CUtensorMap);
using CombineFn = void (*)(const DecodePlan);

template <bool BF16>
CombineFn combine_fn(const DecodePlan& P) {
  const int cols = (P.dh + P.r + 31) / 32;
  if (P.wide_merge) {
    if (P.wide_warps == 16) {
      if (cols <= 3) return lrkv_decode_merge_wide_kernel<BF16, 3, 16>;
      if (cols <= 6) return lrkv_decode_merge_wide_kernel<BF16, 6, 16>;
      if (cols <= 10) return lrkv_decode_merge_wide_kernel<BF16, 10, 16>;
      return lrkv_decode_merge_wide_kernel<BF16, 20, 16>;
    }
    if (cols <= 3) return lrkv_decode_merge_wide_kernel<BF16, 3, kWideWarps>;
    if (cols <= 6) return lrkv_decode_merge_wide_kernel<BF16, 6, kWideWarps>;
    if (cols <= 10) return lrkv_decode_merge_wide_kernel<BF16, 10, kWideWarps>;
    return lrkv_decode_merge_wide_kernel<BF16, 20, kWideWarps>;
  }
  if (cols <= 3) return lrkv_decode_combine_kernel<BF16, 3>;
  if (cols <= 6) return lrkv_decode_combine_kernel<BF16, 6>;
  return lrkv_decode_combine_kernel<BF16, 10>;
}

SplitFn split_fn(const DecodePlan& P) {
  const int rmax = P.r <= 16 ? 16 : P.r <= 32 ? 32 : 64;
  if (P.bf16) {
    if (P.vec == 8) {
      if (rmax == 16) return lrkv_decode_split_kernel<true, 16, 8>;
      if (rmax == 32) return lrkv_decode_split_kernel<true, 32, 8>;
      return lrkv_decode_split_kernel<true, 64, 8>;
    }
    if (rmax == 16) return lrkv_decode_split_kernel<true, 16, 4>;
    if (rmax == 32) return lrkv_decode_split_kernel<true, 32, 4>;
    return lrkv_decode_split_kernel<true, 64, 4>;
  }
  if (rmax == 16) return lrkv_decode_split_kernel<false, 16, 4>;
  if (rmax == 32) return lrkv_decode_split_kernel<false, 32, 4>;
  return lrkv_decode_split_kernel<false, 64, 4>;
}

// An event recorded on `stream`; while the stream is being captured into a
// CUDA graph it becomes an external event-record node (a plain record would
// only mark a dependency), so that replays can be timed with it.
cudaError_t record_event(cudaEvent_t ev, cudaStream_t stream) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(stream, &cs) != cudaSuccess) return cudaErrorInvalidValue;
  return cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, stream, cudaEventRecordExternal)
                                             : cudaEventRecord(ev, stream);
}

template <bool BF16>
// Every host step (tensor maps, shared-memory attributes) comes before the
// first launch, so that the profiled interval [ev_begin, ev_end] holds the
// scan kernel alone.
lrkv_status launch_all(const DecodePlan& P, cudaStream_t stream, cudaEvent_t ev_begin, cudaEvent_t ev_end) {
  const bool pdl = ev_begin == nullptr && ev_end == nullptr;
  CUtensorMap tm_k, tm_v, tm_zk, tm_zv, tm_ks;
  std::memset(&tm_ks, 0, sizeof(tm_ks));
  std::memset(&tm_k, 0, sizeof(tm_k));
  std::memset(&tm_v, 0, sizeof(tm_v));
  std::memset(&tm_zk, 0, sizeof(tm_zk));
  std::memset(&tm_zv, 0, sizeof(tm_zv));
  if (BF16) {
    const CUtensorMapSwizzle sw = P.span == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : P.span == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                                 : CU_TENSOR_MAP_SWIZZLE_32B;
    if (!make_tmap_3d_bf16(&tm_k, P.k_s, P.dh, P.map_len, P.map_seqs, P.box_cols, P.T, sw) ||
        !make_tmap_3d_bf16(&tm_v, P.v_s, P.dh, P.map_len, P.map_seqs, P.box_cols, P.T, sw))
      return LRKV_ERR_CUDA;
  }
  const SplitFn split = P.stream ? nullptr : split_fn(P);
  if (P.stream) {
    const lrkv_status st = stream_prepare(P, &tm_zk, &tm_zv, &tm_ks);
    if (st != LRKV_OK) return st;
  } else if (cudaFuncSetAttribute(split, cudaFuncAttributeMaxDynamicSharedMemorySize, P.smem_bytes) != cudaSuccess) {
    return LRKV_ERR_CUDA;
  }
  const int absorb_smem = std::max((P.dh * P.r + kAbsorbSeq * P.dh) * 4, 16);
  if (P.stream) {
    // the small kernels around the scan ask for the same L1/shared split as
    // the scan, so the SMs need no reconfiguration between the launches
    if (ensure_kernel_smem(reinterpret_cast<const void*>(lrkv_decode_absorb_kernel<BF16>), 0, true) !=
            cudaSuccess ||
        ensure_kernel_smem(reinterpret_cast<const void*>(combine_fn<BF16>(P)), 0, true) != cudaSuccess)
      return LRKV_ERR_CUDA;
  }
  if (absorb_smem > 48 * 1024 &&
      cudaFuncSetAttribute(lrkv_decode_absorb_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           absorb_smem) != cudaSuccess)
    return LRKV_ERR_CUDA;
  const CombineFn combine = combine_fn<BF16>(P);
  if (!P.wide_merge && P.combine_smem > 48 * 1024 &&
      cudaFuncSetAttribute(combine, cudaFuncAttributeMaxDynamicSharedMemorySize, P.combine_smem) != cudaSuccess)
    return LRKV_ERR_CUDA;

  if (!P.stream) {  // the streaming kernel absorbs q itself
    lrkv_decode_absorb_kernel<BF16><<<dim3(P.H, (P.B + kAbsorbSeq - 1) / kAbsorbSeq), 256, absorb_smem, stream>>>(P);
    if (cudaGetLastError() != cudaSuccess) return LRKV_ERR_CUDA;
  }
  if (ev_begin && record_event(ev_begin, stream) != cudaSuccess) return LRKV_ERR_CUDA;

  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  if (P.stream) {
    const lrkv_status st = stream_launch(P, stream, pdl, tm_k, tm_v, tm_zk, tm_zv, tm_ks);
    if (st != LRKV_OK) return st;
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(P.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = P.smem_bytes;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    if (cudaLaunchKernelEx(&cfg, split, P, tm_k, tm_v) != cudaSuccess) return LRKV_ERR_CUDA;
  }
  if (ev_end && record_event(ev_end, stream) != cudaSuccess) return LRKV_ERR_CUDA;

  cudaLaunchConfig_t ccfg = {};
  ccfg.gridDim = dim3(P.combine_ctas);
  ccfg.blockDim = dim3(32 * (P.wide_merge ? (P.wide_warps == 16 ? 16 : kWideWarps) : kCombineWarps));
  ccfg.dynamicSmemBytes = P.wide_merge ? 0 : P.combine_smem;
  ccfg.stream = stream;
  ccfg.attrs = attr;
  ccfg.numAttrs = pdl ? 1 : 0;
  if (cudaLaunchKernelEx(&ccfg, combine, P) != cudaSuccess) return LRKV_ERR_CUDA;
  return LRKV_OK;
}

}  // namespace

lrkv_status decode_make_plan(const lrkv_dims& d, int num_sms, DecodePlan& P, size_t* ws_bytes) {
  std::memset(&P, 0, sizeof(P));
  P.B = d.batch; P.H = d.heads; P.dh = d.head_dim; P.r = d.rank; P.max_len = d.max_len;
  P.map_len = d.max_len; P.map_seqs = d.batch;  // contiguous cache (a paged call overrides)
  const float scale = d.scale > 0.f ? d.scale : 1.f / std::sqrt(static_cast<float>(d.head_dim));
  P.scale_log2 = scale * kLog2e;
  P.bf16 = d.dtype == LRKV_BF16;
  P.esz = P.bf16 ? 2 : 4;
  P.wait_limit = wait_limit_cycles();
  const int H = P.H, dh = P.dh, r = P.r;
  if (r % 4 != 0) return LRKV_ERR_UNSUPPORTED;
  if (H > kThreads) return LRKV_ERR_UNSUPPORTED;

  // value columns per thread: every (head, column group) pair owns cw columns
  const int vw = P.bf16 ? r : dh + r;
  P.vec = P.bf16 ? ((r % 8 == 0) ? 8 : 4) : 4;
  const int max_groups = kThreads / H;
  P.ntg = max_groups;
  if (vw == 0) {
    P.cw = P.vec;
    P.nrg = 1;
  } else {
    int cw = P.vec;
    while (cw <= kMaxCW && (vw + cw - 1) / cw > max_groups) cw += P.vec;
    if (cw > kMaxCW) return LRKV_ERR_UNSUPPORTED;
    P.cw = cw;
    P.nrg = (vw + cw - 1) / cw;
  }

  // tile: T tokens, a multiple of 8, at most kMaxTile, about `target` bytes
  const int z_row = H * r * P.esz;
  P.z_row = z_row;
  const int per_token = 2 * dh * P.esz + 2 * z_row;
  const int target = env_int("LRKV_DECODE_STAGE_KB", 56) * 1024;
  int T = 8;
  while (T * 2 <= kMaxTile && T * 2 * per_token <= target && T * 2 <= kMaxPPT * P.ntg) T *= 2;
  const int forced_T = env_int("LRKV_DECODE_TILE", 0);
  if (forced_T >= 8 && forced_T <= kMaxTile && forced_T % 8 == 0) T = forced_T;
  if (T > kMaxPPT * P.ntg) return LRKV_ERR_UNSUPPORTED;
  P.T = T;

  if (P.bf16) {
    if (dh % 16 != 0) return LRKV_ERR_UNSUPPORTED;
    P.Hp = round_up(H, 16);
    const int mt = P.Hp / 16;
    if (mt * (dh / 8) > kMaxValueTiles * (kThreads / 32)) return LRKV_ERR_UNSUPPORTED;
    const int row_bytes = dh * 2;
    P.span = row_bytes >= 128 ? 128 : row_bytes >= 64 ? 64 : 32;
    if (row_bytes % P.span != 0) return LRKV_ERR_UNSUPPORTED;
    P.box_cols = P.span / 2;
    P.nbox = dh / P.box_cols;
    P.kv_bytes = round_up(T * dh * 2, 1024);
    P.q_stride = dh + 8;
    P.w_stride = ((T / 8) & 1) ? T : T + 8;
  } else {
    P.Hp = H;
    P.kv_bytes = round_up(T * dh * 4, 1024);
    P.q_stride = ((dh / 4) & 1) ? dh : dh + 4;
    P.w_stride = T;
  }
  P.z_bytes = round_up(std::max(T * z_row, 16), 1024);
  P.s_stride = P.Hp + 1;

  // shared-memory carve-up
  int off = 64;  // mbarriers
  P.off_prefix = off; off = round_up(off + (P.B + 1) * 4, 16);
  P.off_q = off; off = round_up(off + P.Hp * P.q_stride * P.esz, 16);
  P.off_ssh = off; off = round_up(off + (P.bf16 ? T * P.s_stride * 4 : 0), 16);
  P.off_sp = off; off = round_up(off + T * P.s_stride * 4, 16);  // fp32 weights
  P.off_w = off; off = round_up(off + (P.bf16 ? P.Hp * P.w_stride * 2 : 0), 16);
  P.off_alpha = off; off = round_up(off + P.Hp * 4, 16);
  P.off_red = off; off = round_up(off + P.ntg * H * 4, 1024);
  P.off_stage = off;
  P.stage_bytes = 2 * P.kv_bytes + 2 * P.z_bytes;
  const int max_stages = std::min(8, env_int("LRKV_DECODE_STAGES", 6));
  const int stages = std::min(max_stages, (227 * 1024 - 1024 - off) / P.stage_bytes);
  if (stages < 2) return LRKV_ERR_UNSUPPORTED;
  P.stages = stages;
  P.smem_bytes = off + stages * P.stage_bytes + 1024;  // + alignment slack
  P.ngw = 1;
  // bf16 shapes the streaming kernel covers use it; the rest (and fp32) run
  // the tile-synchronous kernel planned above
  // CTAs of the narrow combine: one warp per (sequence, head)
  const long long pair_ctas = (static_cast<long long>(P.B) * H + kCombineWarps - 1) / kCombineWarps;
  // A large cache: at least kLargeCacheBytes of rows at capacity (its merge
  // is never the narrow one).
  const long long cap_bytes = static_cast<long long>(P.B) * P.max_len * per_token;
  const bool large = P.bf16 && cap_bytes >= kLargeCacheBytes;
  // The bf16 scan's merge runs wide: one CTA per (sequence, head), 8 or 16
  // warps splitting its partials, after the scan, which takes every SM.
  // Tuning: LRKV_DECODE_WIDE_MERGE=0 keeps a small cache's merge narrow (one
  // warp per pair on SMs the scan leaves free, beside the next call's scan):
  // faster for independent back-to-back calls (8 x 4K rows: 21.0 against
  // 24.7 us a call), slower wherever a call waits for the one before it
  // (latency p50 38.8 against 32.7 us; dependent decode steps 35.6 against
  // 30.4 us), and far slower with many pairs (16 x 1K rows of 32 heads: 62 us
  // for its 512 pairs).
  const bool many_pairs = static_cast<long long>(P.B) * H > static_cast<long long>(kCombineWarps) * kCombineCtas;
  const bool narrow = P.bf16 && !large && !many_pairs && env_int("LRKV_DECODE_WIDE_MERGE", 1) == 0;
  const int reserve = narrow ? static_cast<int>(std::min<long long>(pair_ctas, kCombineCtas)) : 0;
  P.grid = env_int("LRKV_DECODE_GRID", std::max(1, num_sms - reserve));
  // the streaming kernel's grid is (range CTAs, row tiles of 16 heads): it
  // divides P.grid by the row tiles
  if (P.bf16 && env_int("LRKV_DECODE_TILE_SYNC", 0) == 0) stream_plan(P);
  if (!P.stream) P.grid = env_int("LRKV_DECODE_GRID", num_sms);
  P.wide_merge = (P.stream && !narrow) ? 1 : 0;
  // with at most 64 (sequence, head) pairs each pair's merge gets 16 warps
  // (one 64K-row sequence of 32 heads, 304 partials a pair: 14.8 -> 14.2 us;
  // four sequences, 128 pairs of 76: 8.4 us with 8 warps, 9.1 with 16)
  P.wide_warps = static_cast<long long>(P.B) * H <= 64 ? 16 : kWideWarps;
  if (P.wide_merge)
    P.combine_ctas = static_cast<int>(std::min<long long>(static_cast<long long>(P.B) * H, 4ll * num_sms));
  else
    P.combine_ctas = P.stream ? std::max(reserve, 1)
                              : static_cast<int>(std::min<long long>(pair_ctas, large ? num_sms : 65535));
  P.min_tokens = env_int("LRKV_DECODE_MIN_TOKENS", P.stream ? 8 * P.T : 2 * P.T);
  if (P.stream) {
    // L2 prefetch window beyond the ring (tiles per CTA): none.  Tuning:
    // LRKV_DECODE_PREFETCH_TILES=n has thread 0 prefetch each CTA's n tiles
    // after the ring into L2 once it has absorbed.  Measured slower
    // everywhere: on 4 x 64K rows of 32 heads 0.69 -> 0.51 of the HBM peak
    // (two row tiles prefetched the same rows; the ring alone keeps HBM
    // busier); on 8 x 4K rows of 16 heads 25.4 us a launch without, 26.6
    // with 9 tiles, 27.3 with 4: the prefetch traffic delays the block's
    // instruction fetches, which miss to HBM once the caches are cold (the
    // loop's first code then arrives ~8K cycles later than without).
    const int pfw = 0;
    P.pfw = env_int("LRKV_DECODE_PREFETCH_TILES", pfw);
  }
  // per warp: the lift's z row, and the weights and denominators of one sequence's partials
  P.combine_smem = kCombineWarps * (std::max(r, 1) + 2 * P.grid * P.ngw) * 4;
  *ws_bytes = decode_workspace_bytes(P);
  return LRKV_OK;
}

size_t decode_workspace_bytes(const DecodePlan& P) {
  // workspace: status | meta | prefix | p | part_ml | part_acc | CTA status
  const size_t slots = static_cast<size_t>(P.B + P.grid) * P.ngw;
  size_t w = 256;
  w += static_cast<size_t>(round_up(P.B + 1, 64)) * 4;
  w += static_cast<size_t>(P.B) * P.H * std::max(P.r, 1) * 4;
  w = (w + 255) / 256 * 256;
  w += slots * P.H * 2 * 4;
  w = (w + 255) / 256 * 256;
  w += slots * P.H * (P.dh + P.r) * 4;
  w = (w + 255) / 256 * 256;
  w += static_cast<size_t>(P.grid) * std::max(P.mt, 1) * 4;
  return w;
}

lrkv_status decode_merge_launch(const DecodePlan& P, void* stream, bool pdl) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const CombineFn combine = P.bf16 ? combine_fn<true>(P) : combine_fn<false>(P);
  if (ensure_kernel_smem(reinterpret_cast<const void*>(combine), P.wide_merge ? 0 : P.combine_smem, true) !=
      cudaSuccess)
    return LRKV_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t ccfg = {};
  ccfg.gridDim = dim3(P.combine_ctas);
  ccfg.blockDim = dim3(32 * (P.wide_merge ? (P.wide_warps == 16 ? 16 : kWideWarps) : kCombineWarps));
  ccfg.dynamicSmemBytes = P.wide_merge ? 0 : P.combine_smem;
  ccfg.stream = s;
  ccfg.attrs = attr;
  ccfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&ccfg, combine, P) == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

void decode_bind_workspace(DecodePlan& P, void* ws) {
  unsigned char* base = static_cast<unsigned char*>(ws);
  P.status = reinterpret_cast<uint32_t*>(base);
  P.meta = reinterpret_cast<int*>(base + 16);
  size_t off = 256;
  P.prefix = reinterpret_cast<int*>(base + off);
  off += static_cast<size_t>(round_up(P.B + 1, 64)) * 4;
  P.p_abs = reinterpret_cast<float*>(base + off);
  off += static_cast<size_t>(P.B) * P.H * std::max(P.r, 1) * 4;
  off = (off + 255) / 256 * 256;
  P.part_ml = reinterpret_cast<float*>(base + off);
  off += static_cast<size_t>(P.B + P.grid) * P.ngw * P.H * 2 * 4;
  off = (off + 255) / 256 * 256;
  P.part_acc = reinterpret_cast<float*>(base + off);
  off += static_cast<size_t>(P.B + P.grid) * P.ngw * P.H * (P.dh + P.r) * 4;
  off = (off + 255) / 256 * 256;
  P.cta_status = reinterpret_cast<uint32_t*>(base + off);
}

lrkv_status decode_launch(const DecodePlan& P, void* stream, void* ev_begin, void* ev_end) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaEvent_t e0 = static_cast<cudaEvent_t>(ev_begin), e1 = static_cast<cudaEvent_t>(ev_end);
  return P.bf16 ? launch_all<true>(P, s, e0, e1) : launch_all<false>(P, s, e0, e1);
}

}  // namespace lrkv
