// decode_stream.cu — the bf16 split-KV scan as independent warp streams.
//
// One CTA owns a range of the concatenated histories (see decode.cu).  8-token
// tiles stream through a ring of shared-memory stages filled by TMA (shared
// rows k_s, v_s as swizzled tensor boxes, read once for all heads; latent rows
// as per-token bulk copies into padded rows).  Warps work independently: warp
// (group, m) takes every ng-th tile and handles the 16 heads of MMA row tile
// m; the group that finishes a tile refills its stage with the tile `stages`
// ahead, so there is no separate producer.  Per tile, FlashAttention-2 style:
//   * shared scores q_h . k_s on the tensor cores (bf16 mma.sync, heads are
//     the rows, q kept in registers as A fragments for the whole piece);
//   * private scores p_h . z_k,h in fp32 (p_h = q_h B_h^K from the absorb
//     kernel), added before the softmax;
//   * ONE online softmax per head (row max over the quad of lanes holding the
//     row) over the summed scores ("Low-Rank Key Value Attention | What a
//     shared cache can preserve", §3, fused online-softmax paragraph);
//   * shared values on the tensor cores with the probabilities reused from
//     the score fragments as the A operand; private values sum_j a_j z_v,h,j
//     in fp32 with the same rescale factor.
// No CTA-wide barrier is taken per tile.  At the end of each (sequence,
// range) piece the groups' partial states are merged on chip (tree through
// shared memory) or written per group for the combine kernel.
#include <cmath>
#include <algorithm>
#include <cstring>

#include <cuda.h>

#include "decode_common.cuh"
#include "decode_plan.h"
#include "ptx.cuh"

namespace lrkv {

using namespace dec;

namespace {

constexpr int kT = 8;                 // tokens per tile (one MMA n-tile)
constexpr int kScratch = 16 * 8 + 32;  // floats of per-warp scratch

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

// Pieces of this CTA's token range: (sequence b, rows [t_beg, t_end)).
struct Piece {
  int b, t_beg, t_end, ntiles;
};

__device__ __forceinline__ bool piece_first(Piece& p, const int* pre, int B, int g0, int g1) {
  TileWalk w;
  if (!walk_first(w, pre, B, g0, g1)) return false;
  p.b = w.b; p.t_beg = w.t0; p.t_end = w.t_end;
  p.ntiles = (p.t_end - p.t_beg + kT - 1) / kT;
  return true;
}

__device__ __forceinline__ bool piece_next(Piece& p, const int* pre, int B, int g1) {
  int b = p.b + 1;
  while (b < B && pre[b] < g1 && pre[b + 1] == pre[b]) ++b;
  if (b >= B || pre[b] >= g1) return false;
  p.b = b; p.t_beg = 0; p.t_end = min(pre[b + 1], g1) - pre[b];
  p.ntiles = (p.t_end + kT - 1) / kT;
  return true;
}

// Producer warp: the copies of tile (piece p, row t0) into stage s.
__device__ __forceinline__ void stream_issue(const DecodePlan& P, const CUtensorMap* tm_k,
                                             const CUtensorMap* tm_v, unsigned char* smem, uint64_t* full,
                                             int s, int b, int t0, int nvalid, int lane) {
  unsigned char* ks = smem + P.off_kv + static_cast<size_t>(s) * 2 * P.kv_bytes;
  unsigned char* vs = ks + P.kv_bytes;
  unsigned char* zk = smem + P.off_z + static_cast<size_t>(s) * 2 * kT * P.zs_stride;
  unsigned char* zv = zk + kT * P.zs_stride;
  fence_proxy_async_smem();  // earlier generic reads of the stage before the async writes
  if (lane == 0) {
    mbar_arrive_expect_tx(&full[s], 2u * kT * P.dh * 2u + 2u * static_cast<uint32_t>(nvalid) * P.z_row);
  }
  __syncwarp();
  if (lane < P.nbox) {
    tma_load_3d(ks + lane * kT * P.span, tm_k, lane * P.box_cols, t0, b, &full[s]);
    tma_load_3d(vs + lane * kT * P.span, tm_v, lane * P.box_cols, t0, b, &full[s]);
  }
  if (P.r > 0 && lane < 2 * nvalid) {
    const int row = lane >> 1;
    const size_t g = (static_cast<size_t>(b) * P.max_len + t0 + row) * P.z_row;
    if (lane & 1)
      tma_load_1d(zv + row * P.zs_stride, static_cast<const unsigned char*>(P.z_v) + g, P.z_row, &full[s]);
    else
      tma_load_1d(zk + row * P.zs_stride, static_cast<const unsigned char*>(P.z_k) + g, P.z_row, &full[s]);
  }
}

// Per-warp partial state of 16 heads, moved through shared memory or global.
// Row layout (width W = dh + r + 2): [m, l, acc_s[dh], acc_z[r]].
template <int DHT, int RMAX>
struct WarpState {
  float m0, m1, l0, l1;           // rows g and g+8 of the MMA tile
  float acc_v[2 * DHT][4];        // shared-value fragments
  float acc_z[RMAX];              // private sum of head hh = lane & 15
};

}  // namespace

// Walks the tile sequence forward (monotone), giving the coordinates of tile j.
struct TileCursor {
  Piece pc;
  int ibase;
  bool more;
  __device__ __forceinline__ bool seek(int j, const int* pre, int B, int g1) {
    while (more && j >= ibase + pc.ntiles) {
      ibase += pc.ntiles;
      more = piece_next(pc, pre, B, g1);
    }
    return more;
  }
};

template <int DHT, int RMAX, int NE>
__global__ void __launch_bounds__(32 * kStreamConsumers, 1)
    lrkv_decode_stream_kernel(const DecodePlan P, const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_bad;
  __shared__ int s_timeout;
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int B = P.B, H = P.H, dh = P.dh, r = P.r;
  const int n_cons = P.ng * P.mt;  // warps
  const int W = dh + r + 2;

  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  uint64_t* empty = full + P.stages;
  int* pre = reinterpret_cast<int*>(smem + P.off_prefix);
  float* p_sh = reinterpret_cast<float*>(smem + P.off_p);

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

  if (tid == 0) {
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 32 * P.mt);
    }
    fence_barrier_init();
  }
  __syncthreads();

  // ---- first `stages` tiles: each group issues the ones it will consume ----
  {
    const int gi0 = warp / P.mt;
    if (warp % P.mt == 0) {
      TileCursor cur;
      cur.more = piece_first(cur.pc, pre, B, g0, g1);
      cur.ibase = 0;
      for (int j = gi0; j < P.stages && cur.seek(j, pre, B, g1); j += P.ng) {
        const int t0 = cur.pc.t_beg + (j - cur.ibase) * kT;
        stream_issue(P, &tm_k, &tm_v, smem, full, j, cur.pc.b, t0, min(kT, cur.pc.t_end - t0), lane);
      }
    }
  }

  // ============================================================ warps ====
  pdl_wait();  // p = q B^K from the absorb kernel
  if (s_bad && tid == 0) record_status(P.status, kDevBounds);

  const int gi = warp / P.mt, mi = warp % P.mt;
  const int g = lane >> 2, q4 = lane & 3;
  const int hh = lane & 15, tp = lane >> 4;  // private-value role: head, token parity
  float* scr = reinterpret_cast<float*>(smem + P.off_scr) + warp * kScratch;
  float* mbuf = reinterpret_cast<float*>(smem + P.off_merge);
  const int nct = n_cons * 32;

  WarpState<DHT, RMAX> st;
  uint32_t qa[DHT][4];

  Piece pc;
  bool more = piece_first(pc, pre, B, g0, g1);
  int ibase = 0;      // global tile index of the piece's first tile
  bool ok = true;
  TileCursor refill;  // tiles this warp issues (index of its tile + stages)
  refill.more = piece_first(refill.pc, pre, B, g0, g1);
  refill.ibase = 0;
  while (more) {
    // ---- piece set-up: p_h for the heads, q fragments of this warp's tile --
    named_sync(1, nct);  // the previous piece's merge is finished
    {
      const float* gp = P.p_abs + static_cast<size_t>(pc.b) * H * r;
      for (int i = tid; i < H * r; i += nct) p_sh[(i / r) * P.p_stride + (i % r)] = gp[i];
      const __nv_bfloat16* gq = static_cast<const __nv_bfloat16*>(P.q) + static_cast<size_t>(pc.b) * H * dh;
      const int h0 = mi * 16 + g, h1 = h0 + 8;
#pragma unroll
      for (int kk = 0; kk < DHT; ++kk) {
        const int k = kk * 16 + 2 * q4;
        qa[kk][0] = h0 < H ? *reinterpret_cast<const uint32_t*>(gq + h0 * dh + k) : 0u;
        qa[kk][1] = h1 < H ? *reinterpret_cast<const uint32_t*>(gq + h1 * dh + k) : 0u;
        qa[kk][2] = h0 < H ? *reinterpret_cast<const uint32_t*>(gq + h0 * dh + k + 8) : 0u;
        qa[kk][3] = h1 < H ? *reinterpret_cast<const uint32_t*>(gq + h1 * dh + k + 8) : 0u;
      }
    }
    st.m0 = st.m1 = -INFINITY;
    st.l0 = st.l1 = 0.f;
#pragma unroll
    for (int n = 0; n < 2 * DHT; ++n)
#pragma unroll
      for (int k = 0; k < 4; ++k) st.acc_v[n][k] = 0.f;
#pragma unroll
    for (int k = 0; k < RMAX; ++k) st.acc_z[k] = 0.f;
    named_sync(1, nct);  // p_sh ready

    // ---- this group's tiles of the piece ------------------------------------
    const int first = ibase + ((gi - ibase) % P.ng + P.ng) % P.ng;
    for (int i = first; i < ibase + pc.ntiles; i += P.ng) {
      const int s = i % P.stages;
      const int t0 = pc.t_beg + (i - ibase) * kT;
      const int nvalid = min(kT, pc.t_end - t0);
      if (ok) {
        ok = mbar_wait_bounded(&full[s], static_cast<uint32_t>(i / P.stages) & 1u);
        if (!ok) *reinterpret_cast<volatile int*>(&s_timeout) = 1;
      }
      if (ok && !*reinterpret_cast<volatile int*>(&s_timeout)) {
        const unsigned char* ks = smem + P.off_kv + static_cast<size_t>(s) * 2 * P.kv_bytes;
        const unsigned char* vs = ks + P.kv_bytes;
        const unsigned char* zk = smem + P.off_z + static_cast<size_t>(s) * 2 * kT * P.zs_stride;
        const unsigned char* zv = zk + kT * P.zs_stride;

        // shared scores: rows = heads of tile mi, columns = the 8 tokens
        float sv[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int kk = 0; kk < DHT; ++kk) {
          const int k0 = kk * 16 + ((lane >> 3) & 1) * 8;
          uint32_t b0, b1;
          ldsm_x2(b0, b1, ks + (k0 / P.box_cols) * kT * P.span + swz_off(lane & 7, (k0 % P.box_cols) / 8, P.span));
          mma_bf16_16816(sv, qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b0, b1);
        }
        // private scores of (head g / g+8, token 2q4 / 2q4+1)
        if (r > 0) {
#pragma unroll
          for (int hs = 0; hs < 2; ++hs) {
            const int h = mi * 16 + g + 8 * hs;
            if (h < H) {
              const float* ph = p_sh + h * P.p_stride;
              const unsigned char* z0 = zk + (2 * q4) * P.zs_stride + h * r * 2;
              float a0[4] = {0.f, 0.f, 0.f, 0.f}, a1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
              for (int c0 = 0; c0 < RMAX; c0 += NE) {
                if (c0 < r) {
                  float pv[NE], x0[NE], x1[NE];
#pragma unroll
                  for (int e = 0; e < NE; e += 4) {
                    const float4 v = *reinterpret_cast<const float4*>(ph + c0 + e);
                    pv[e] = v.x; pv[e + 1] = v.y; pv[e + 2] = v.z; pv[e + 3] = v.w;
                  }
                  load_vec<true, NE>(z0 + c0 * 2, x0);
                  load_vec<true, NE>(z0 + P.zs_stride + c0 * 2, x1);
#pragma unroll
                  for (int e = 0; e < NE; ++e) {
                    a0[e & 3] = fmaf(x0[e], pv[e], a0[e & 3]);
                    a1[e & 3] = fmaf(x1[e], pv[e], a1[e & 3]);
                  }
                }
              }
              sv[2 * hs] += (a0[0] + a0[1]) + (a0[2] + a0[3]);
              sv[2 * hs + 1] += (a1[0] + a1[1]) + (a1[2] + a1[3]);
            }
          }
        }
        // scale, mask rows past the piece's end, one online softmax per head
        const bool v0 = 2 * q4 < nvalid, v1 = 2 * q4 + 1 < nvalid;
        sv[0] = v0 ? sv[0] * P.scale_log2 : -INFINITY;
        sv[1] = v1 ? sv[1] * P.scale_log2 : -INFINITY;
        sv[2] = v0 ? sv[2] * P.scale_log2 : -INFINITY;
        sv[3] = v1 ? sv[3] * P.scale_log2 : -INFINITY;
        float mx0 = fmaxf(sv[0], sv[1]), mx1 = fmaxf(sv[2], sv[3]);
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(st.m0, mx0), mn1 = fmaxf(st.m1, mx1);
        const float al0 = exp2f(st.m0 - mn0), al1 = exp2f(st.m1 - mn1);  // mn is finite
        st.m0 = mn0;
        st.m1 = mn1;
        const float p0 = exp2f(sv[0] - mn0), p1 = exp2f(sv[1] - mn0);
        const float p2 = exp2f(sv[2] - mn1), p3 = exp2f(sv[3] - mn1);
        st.l0 = st.l0 * al0 + (p0 + p1);
        st.l1 = st.l1 * al1 + (p2 + p3);
        if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
          for (int n = 0; n < 2 * DHT; ++n) {
            st.acc_v[n][0] *= al0; st.acc_v[n][1] *= al0;
            st.acc_v[n][2] *= al1; st.acc_v[n][3] *= al1;
          }
        }
        // shared values: the probabilities are the A fragment of m16n8k8
        const uint32_t pa0 = pack_bf16(p0, p1), pa1 = pack_bf16(p2, p3);
        const uint32_t keep = (v0 ? 0x0000ffffu : 0u) | (v1 ? 0xffff0000u : 0u);
#pragma unroll
        for (int n = 0; n < 2 * DHT; ++n) {
          const int n0 = n * 8;
          uint32_t b0;
          ldsm_x1_trans(b0, vs + (n0 / P.box_cols) * kT * P.span + swz_off(lane & 7, (n0 % P.box_cols) / 8, P.span));
          mma_bf16_1688(st.acc_v[n], pa0, pa1, b0 & keep);
        }
        // private values: lane (head hh, token parity tp)
        if (r > 0) {
          scr[g * 8 + 2 * q4] = p0;
          scr[g * 8 + 2 * q4 + 1] = p1;
          scr[(g + 8) * 8 + 2 * q4] = p2;
          scr[(g + 8) * 8 + 2 * q4 + 1] = p3;
          if (q4 == 0) { scr[128 + g] = al0; scr[128 + g + 8] = al1; }
          __syncwarp();
          const int h = mi * 16 + hh;
          if (h < H) {
            const float a = scr[128 + hh];
            if (a != 1.f) {
#pragma unroll
              for (int k = 0; k < RMAX; ++k) st.acc_z[k] *= a;
            }
#pragma unroll
            for (int k = 0; k < kT / 2; ++k) {
              const int t = tp + 2 * k;
              if (t < nvalid) {
                const float w = scr[hh * 8 + t];
                const unsigned char* zt = zv + t * P.zs_stride + h * r * 2;
#pragma unroll
                for (int c0 = 0; c0 < RMAX; c0 += NE) {
                  if (c0 < r) {
                    float x[NE];
                    load_vec<true, NE>(zt + c0 * 2, x);
#pragma unroll
                    for (int e = 0; e < NE; ++e) st.acc_z[c0 + e] = fmaf(w, x[e], st.acc_z[c0 + e]);
                  }
                }
              }
            }
          }
          __syncwarp();
        }
      }
      // done with the stage: refill it with tile i + stages
      const int j = i + P.stages;
      if (P.mt > 1) mbar_arrive(&empty[s]);
      if (mi == 0 && refill.seek(j, pre, B, g1)) {
        if (P.mt > 1 && ok) {
          int got = 0;
          if (lane == 0) got = mbar_wait_bounded(&empty[s], static_cast<uint32_t>(i / P.stages) & 1u) ? 1 : 0;
          got = __shfl_sync(0xffffffffu, got, 0);
          if (!got) { ok = false; *reinterpret_cast<volatile int*>(&s_timeout) = 1; }
        }
        __syncwarp();
        if (ok) {
          const int jt0 = refill.pc.t_beg + (j - refill.ibase) * kT;
          stream_issue(P, &tm_k, &tm_v, smem, full, s, refill.pc.b, jt0, min(kT, refill.pc.t_end - jt0), lane);
        }
      }
    }

    // ---- end of the piece: reduce within the warp ------------------------------
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 1);
    st.l0 += __shfl_xor_sync(0xffffffffu, st.l0, 2);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 1);
    st.l1 += __shfl_xor_sync(0xffffffffu, st.l1, 2);
#pragma unroll
    for (int k = 0; k < RMAX; ++k) st.acc_z[k] += __shfl_xor_sync(0xffffffffu, st.acc_z[k], 16);

    // write this warp's state into a row block of width W (16 head rows)
    auto put = [&](float* dst) {
      if (q4 == 0) {
        dst[g * W] = st.m0; dst[g * W + 1] = st.l0;
        dst[(g + 8) * W] = st.m1; dst[(g + 8) * W + 1] = st.l1;
      }
#pragma unroll
      for (int n = 0; n < 2 * DHT; ++n) {
        const int col = 2 + n * 8 + 2 * q4;
        dst[g * W + col] = st.acc_v[n][0]; dst[g * W + col + 1] = st.acc_v[n][1];
        dst[(g + 8) * W + col] = st.acc_v[n][2]; dst[(g + 8) * W + col + 1] = st.acc_v[n][3];
      }
      if (tp == 0) {
#pragma unroll
        for (int k = 0; k < RMAX; ++k)
          if (k < r) dst[hh * W + 2 + dh + k] = st.acc_z[k];
      }
    };

    if (P.merge_smem) {
      // tree merge of the groups' states of the same row tile: at step s,
      // group gi = 2sk + s hands its state to group 2sk
      for (int step = 1; step < P.ng; step <<= 1) {
        const int k = gi / (2 * step), rem = gi % (2 * step);
        float* slot = mbuf + static_cast<size_t>((k * P.mt + mi)) * 16 * W;
        if (rem == step) put(slot);
        named_sync(1, nct);
        if (rem == 0 && gi + step < P.ng) {
          const float* src = slot;
          const float mb0 = src[g * W], lb0 = src[g * W + 1];
          const float mb1 = src[(g + 8) * W], lb1 = src[(g + 8) * W + 1];
          const float M0 = fmaxf(st.m0, mb0), M1 = fmaxf(st.m1, mb1);
          const float fa0 = M0 == -INFINITY ? 0.f : exp2f(st.m0 - M0);
          const float fb0 = M0 == -INFINITY ? 0.f : exp2f(mb0 - M0);
          const float fa1 = M1 == -INFINITY ? 0.f : exp2f(st.m1 - M1);
          const float fb1 = M1 == -INFINITY ? 0.f : exp2f(mb1 - M1);
          st.m0 = M0; st.m1 = M1;
          st.l0 = st.l0 * fa0 + lb0 * fb0;
          st.l1 = st.l1 * fa1 + lb1 * fb1;
#pragma unroll
          for (int n = 0; n < 2 * DHT; ++n) {
            const int col = 2 + n * 8 + 2 * q4;
            st.acc_v[n][0] = st.acc_v[n][0] * fa0 + src[g * W + col] * fb0;
            st.acc_v[n][1] = st.acc_v[n][1] * fa0 + src[g * W + col + 1] * fb0;
            st.acc_v[n][2] = st.acc_v[n][2] * fa1 + src[(g + 8) * W + col] * fb1;
            st.acc_v[n][3] = st.acc_v[n][3] * fa1 + src[(g + 8) * W + col + 1] * fb1;
          }
          // factors of head hh for the private sums
          if (q4 == 0) {
            scr[128 + g] = fa0; scr[128 + g + 8] = fa1;
            scr[144 + g] = fb0; scr[144 + g + 8] = fb1;
          }
          __syncwarp();
          const float fa = scr[128 + hh], fb = scr[144 + hh];
#pragma unroll
          for (int k = 0; k < RMAX; ++k)
            if (k < r) st.acc_z[k] = st.acc_z[k] * fa + src[hh * W + 2 + dh + k] * fb;
          __syncwarp();
        }
        named_sync(1, nct);
      }
    }
    if (!P.merge_smem || gi == 0) {
      // write the (merged) state as this piece's partial
      const int slot = (pc.b + c) * P.ngw + (P.merge_smem ? 0 : gi);
      float* pacc = P.part_acc + static_cast<size_t>(slot) * H * (dh + r);
      float* pml = P.part_ml + static_cast<size_t>(slot) * H * 2;
      const int h0 = mi * 16 + g, h1 = h0 + 8;
      if (q4 == 0) {
        if (h0 < H) { pml[h0 * 2] = st.m0; pml[h0 * 2 + 1] = st.l0; }
        if (h1 < H) { pml[h1 * 2] = st.m1; pml[h1 * 2 + 1] = st.l1; }
      }
#pragma unroll
      for (int n = 0; n < 2 * DHT; ++n) {
        const int col = n * 8 + 2 * q4;
        if (h0 < H) { pacc[h0 * (dh + r) + col] = st.acc_v[n][0]; pacc[h0 * (dh + r) + col + 1] = st.acc_v[n][1]; }
        if (h1 < H) { pacc[h1 * (dh + r) + col] = st.acc_v[n][2]; pacc[h1 * (dh + r) + col + 1] = st.acc_v[n][3]; }
      }
      const int h = mi * 16 + hh;
      if (tp == 0 && h < H) {
#pragma unroll
        for (int k = 0; k < RMAX; ++k)
          if (k < r) pacc[h * (dh + r) + dh + k] = st.acc_z[k];
      }
    }
    ibase += pc.ntiles;
    more = piece_next(pc, pre, B, g1);
  }
  if (!ok && lane == 0) record_status(P.status, kDevTimeout);
  pdl_trigger();
}

// ======================================================================= host
namespace {

using StreamFn = void (*)(const DecodePlan, const CUtensorMap, const CUtensorMap);

template <int DHT>
StreamFn pick_r(const DecodePlan& P) {
  if (P.r <= 16) return P.vec == 8 ? lrkv_decode_stream_kernel<DHT, 16, 8> : lrkv_decode_stream_kernel<DHT, 16, 4>;
  if (P.r <= 32) return P.vec == 8 ? lrkv_decode_stream_kernel<DHT, 32, 8> : lrkv_decode_stream_kernel<DHT, 32, 4>;
  return P.vec == 8 ? lrkv_decode_stream_kernel<DHT, 64, 8> : lrkv_decode_stream_kernel<DHT, 64, 4>;
}

StreamFn stream_fn(const DecodePlan& P) {
  switch (P.dh / 16) {
    case 4: return pick_r<4>(P);
    case 8: return pick_r<8>(P);
    default: return nullptr;
  }
}

}  // namespace

// Fills the streaming-kernel fields of an already sized plan.
static lrkv_status stream_plan_impl(DecodePlan& P);

lrkv_status stream_plan(DecodePlan& P_out) {
  DecodePlan P = P_out;
  const lrkv_status st = stream_plan_impl(P);
  if (st == LRKV_OK) P_out = P;
  return st;
}

static lrkv_status stream_plan_impl(DecodePlan& P) {
  const int dh = P.dh, r = P.r, H = P.H;
  if (!(dh == 64 || dh == 128)) return LRKV_ERR_UNSUPPORTED;
  if (r > 0 && r % 4 != 0) return LRKV_ERR_UNSUPPORTED;
  P.stream = 1;
  P.T = kT;
  P.Hp = round_up(H, 16);
  P.mt = P.Hp / 16;
  if (P.mt > kStreamConsumers) return LRKV_ERR_UNSUPPORTED;
  const int row_bytes = dh * 2;
  P.span = row_bytes >= 128 ? 128 : 64;
  P.box_cols = P.span / 2;
  P.nbox = dh / P.box_cols;
  P.kv_bytes = round_up(kT * dh * 2, 1024);
  P.vec = (r % 8 == 0) ? 8 : 4;
  P.z_row = H * r * 2;
  {
    int zs = round_up(std::max(P.z_row, 16), 16);
    if (((zs / 16) & 1) == 0) zs += 16;
    P.zs_stride = zs;
  }
  {
    const int r4 = round_up(std::max(r, 1), 4);
    P.p_stride = ((r4 / 4) & 1) ? r4 : r4 + 4;
  }
  const int ng_max = kStreamConsumers / P.mt;
  const int W = dh + r + 2;
  const int stage_bytes = 2 * P.kv_bytes + round_up(2 * kT * P.zs_stride, 16);

  // shared memory: barriers | prefix | p | scratch | merge buffer | kv ring | z ring
  auto layout = [&](int stages, int merge, int ng) {
    int off = 256;
    P.off_prefix = off; off = round_up(off + (P.B + 1) * 4, 16);
    P.off_p = off; off = round_up(off + H * P.p_stride * 4, 16);
    P.off_scr = off; off = round_up(off + (ng * P.mt) * kScratch * 4, 16);
    P.off_merge = off; off = round_up(off + (merge ? ((ng + 1) / 2) * P.mt * 16 * W * 4 : 0), 1024);
    P.off_kv = off; off += stages * 2 * P.kv_bytes;
    P.off_z = off; off += stages * round_up(2 * kT * P.zs_stride, 16);
    return off + 1024;  // alignment slack
  };
  const int budget = 226 * 1024;  // opt-in limit (227 KB) less static shared memory
  // most groups whose ring holds a tile for each; merge on chip if it fits
  int best_stages = 0, best_merge = 0, best_ng = 0;
  for (int ng = ng_max; ng >= 1 && best_stages == 0; --ng) {
    for (int merge = 1; merge >= 0; --merge) {
      int stages = 0;
      while (stages < 16 && layout(stages + 1, merge, ng) <= budget) ++stages;
      if (stages >= ng && stages >= 2) {
        best_stages = std::min(stages, 2 * ng);
        best_merge = merge;
        best_ng = ng;
        break;
      }
    }
  }
  if (best_stages == 0) return LRKV_ERR_UNSUPPORTED;
  P.ng = best_ng;
  P.merge_smem = best_merge;
  P.ngw = best_merge ? 1 : best_ng;
  P.stages = best_stages;
  P.smem_bytes = layout(P.stages, P.merge_smem, P.ng);
  P.stage_bytes = stage_bytes;
  P.nthreads = 32 * (P.ng * P.mt);
  (void)stage_bytes;
  return stream_fn(P) ? LRKV_OK : LRKV_ERR_UNSUPPORTED;
}

lrkv_status stream_launch(const DecodePlan& P, cudaStream_t stream, bool pdl, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v) {
  const StreamFn kern = stream_fn(P);
  if (!kern) return LRKV_ERR_UNSUPPORTED;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P.smem_bytes) != cudaSuccess)
    return LRKV_ERR_CUDA;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid);
  cfg.blockDim = dim3(P.nthreads);
  cfg.dynamicSmemBytes = P.smem_bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, P, tm_k, tm_v) == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

}  // namespace lrkv
