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
//           ring of shared-memory stages filled by 1-D TMA bulk copies: each
//           shared row k_s/v_s is read from HBM once and serves all H heads
//           (the reuse the review's roofline paragraph asks for), each latent
//           row once for its head.  Per tile it forms the summed score
//           (shared part on the tensor cores with bf16 mma.sync, private part
//           as fp32 dot products), runs ONE online softmax per head, and
//           updates two accumulators per head: d_h-wide shared and r-wide
//           private.  At the end of each (sequence, range) piece it writes
//           the unnormalised partial (m, l, acc_s, acc_z).
//  combine  merges the pieces of a sequence with the log-sum-exp rule, divides
//           by the denominator and maps the private sum through (B_h^V)^T
//           once (Algorithm 2 steps 06-09).
//
// The three launches are chained with programmatic dependent launch, so the
// split kernel starts streaming the cache while absorb still runs.
#include <cmath>
#include <cstdlib>
#include <cstring>

#include "decode_plan.h"
#include "ptx.cuh"

namespace lrkv {

namespace {

constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

__host__ __device__ inline int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Padded shared-memory row stride: a multiple of 16 bytes holding an odd
// number of 16-byte chunks, so consecutive rows start in different bank
// groups (conflict-free ldmatrix and per-row vector loads).
inline int odd_chunk_stride(int bytes) {
  int s = round_up(bytes > 0 ? bytes : 16, 16);
  if (((s / 16) & 1) == 0) s += 16;
  return s;
}

// CTA that owns global token g when N tokens are cut into G ranges
// [floor(c N / G), floor((c+1) N / G)).
__device__ __forceinline__ int cta_of_token(long long g, long long N, long long G) {
  return static_cast<int>(((g + 1) * G - 1) / N);
}

// ---------------------------------------------------------- element loads --
template <bool BF16, int NE>
__device__ __forceinline__ void load_vec(const unsigned char* p, float* f) {
  if constexpr (BF16) {
    if constexpr (NE == 8) {
      const uint4 u = *reinterpret_cast<const uint4*>(p);
      f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
      f[4] = bf_lo(u.z); f[5] = bf_hi(u.z); f[6] = bf_lo(u.w); f[7] = bf_hi(u.w);
    } else if constexpr (NE == 4) {
      const uint2 u = *reinterpret_cast<const uint2*>(p);
      f[0] = bf_lo(u.x); f[1] = bf_hi(u.x); f[2] = bf_lo(u.y); f[3] = bf_hi(u.y);
    } else if constexpr (NE == 2) {
      const uint32_t u = *reinterpret_cast<const uint32_t*>(p);
      f[0] = bf_lo(u); f[1] = bf_hi(u);
    } else {
      const uint32_t u = *reinterpret_cast<const unsigned short*>(p);
      f[0] = __uint_as_float(u << 16);
    }
  } else {
    if constexpr (NE == 4) {
      const float4 v = *reinterpret_cast<const float4*>(p);
      f[0] = v.x; f[1] = v.y; f[2] = v.z; f[3] = v.w;
    } else if constexpr (NE == 2) {
      const float2 v = *reinterpret_cast<const float2*>(p);
      f[0] = v.x; f[1] = v.y;
    } else {
      f[0] = *reinterpret_cast<const float*>(p);
    }
  }
}

template <int NE>
__device__ __forceinline__ void load_f32(const float* p, float* f) {
  if constexpr (NE % 4 == 0) {
#pragma unroll
    for (int e = 0; e < NE; e += 4) {
      const float4 v = *reinterpret_cast<const float4*>(p + e);
      f[e] = v.x; f[e + 1] = v.y; f[e + 2] = v.z; f[e + 3] = v.w;
    }
  } else if constexpr (NE == 2) {
    const float2 v = *reinterpret_cast<const float2*>(p);
    f[0] = v.x; f[1] = v.y;
  } else {
    f[0] = p[0];
  }
}

__device__ __forceinline__ float load_elem(const void* base, size_t i, bool bf16) {
  if (bf16) return __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[i]);
  return reinterpret_cast<const float*>(base)[i];
}

// --------------------------------------------------- private-branch pieces --
// Private logits p_h . z_k,h,t for this lane's tokens (four partial sums per
// token to shorten the dependent FMA chain).
template <bool BF16, int NE, int RMAX>
__device__ __forceinline__ void private_logits(const unsigned char* zrow0, int tok_stride_bytes,
                                               int ppt, const float* ph, int r,
                                               float (&res)[kMaxPPT]) {
  constexpr int ESZ = BF16 ? 2 : 4;
  float part[kMaxPPT][4];
#pragma unroll
  for (int i = 0; i < kMaxPPT; ++i)
#pragma unroll
    for (int k = 0; k < 4; ++k) part[i][k] = 0.f;
#pragma unroll
  for (int c = 0; c < RMAX; c += NE) {
    if (c < r) {
      float pv[NE];
      load_f32<NE>(ph + c, pv);
#pragma unroll
      for (int i = 0; i < kMaxPPT; ++i) {
        if (i < ppt) {
          float zv[NE];
          load_vec<BF16, NE>(zrow0 + static_cast<size_t>(i) * tok_stride_bytes + c * ESZ, zv);
#pragma unroll
          for (int e = 0; e < NE; ++e) part[i][e & 3] = fmaf(zv[e], pv[e], part[i][e & 3]);
        }
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kMaxPPT; ++i) res[i] = (part[i][0] + part[i][1]) + (part[i][2] + part[i][3]);
}

// acc_z = alpha * acc_z + sum_i w_i z_v,h,t_i
template <bool BF16, int NE, int RMAX>
__device__ __forceinline__ void private_values(const unsigned char* zrow0, int tok_stride_bytes,
                                               int ppt, const float (&w)[kMaxPPT], float alpha,
                                               int r, float (&acc)[RMAX]) {
  constexpr int ESZ = BF16 ? 2 : 4;
#pragma unroll
  for (int c = 0; c < RMAX; ++c) acc[c] *= alpha;
#pragma unroll
  for (int i = 0; i < kMaxPPT; ++i) {
    if (i < ppt) {
#pragma unroll
      for (int c = 0; c < RMAX; c += NE) {
        if (c < r) {
          float zv[NE];
          load_vec<BF16, NE>(zrow0 + static_cast<size_t>(i) * tok_stride_bytes + c * ESZ, zv);
#pragma unroll
          for (int e = 0; e < NE; ++e) acc[c + e] = fmaf(w[i], zv[e], acc[c + e]);
        }
      }
    }
  }
}

// Dot product of two staged rows of length n (fp32 path, shared logits).
__device__ __forceinline__ float dot_f32(const float* a, const float* b, int n) {
  float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
  for (int k = 0; k < n; k += 4) {
    const float4 x = *reinterpret_cast<const float4*>(a + k);
    const float4 y = *reinterpret_cast<const float4*>(b + k);
    s0 = fmaf(x.x, y.x, s0); s1 = fmaf(x.y, y.y, s1); s2 = fmaf(x.z, y.z, s2); s3 = fmaf(x.w, y.w, s3);
  }
  return (s0 + s1) + (s2 + s3);
}

// ------------------------------------------------------ token-range walk --
// A CTA's token range [g0, g1) of the concatenated histories, visited tile by
// tile; tiles never straddle two sequences.
struct TileWalk {
  int b;       // sequence
  int t0;      // first row of the tile within the sequence
  int t_beg;   // first row of this CTA's piece of the sequence
  int t_end;   // one past its last row
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
  w.t_beg = g0 - pre[b];
  w.t0 = w.t_beg;
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
  w.t_beg = 0;
  w.t0 = 0;
  w.t_end = min(pre[b + 1], g1) - pre[b];
  return true;
}

// Producer: warp 0 issues the row copies of one tile into stage `s`.
__device__ __forceinline__ void issue_tile(const DecodePlan& P, unsigned char* stage, uint64_t* bar,
                                           const TileWalk& w, int lane) {
  const int nvalid = min(P.T, w.t_end - w.t0);
  const uint32_t bytes =
      static_cast<uint32_t>(nvalid) * static_cast<uint32_t>(2 * P.ks_row + (P.r > 0 ? 2 * P.z_row : 0));
  if (lane == 0) mbar_arrive_expect_tx(bar, bytes);
  __syncwarp();
  unsigned char* ks = stage;
  unsigned char* vs = ks + P.T * P.ks_stride;
  unsigned char* zk = vs + P.T * P.ks_stride;
  unsigned char* zv = zk + P.T * P.z_stride;
  const size_t row0 = static_cast<size_t>(w.b) * P.max_len + w.t0;
  const unsigned char* gks = static_cast<const unsigned char*>(P.k_s) + row0 * P.ks_row;
  const unsigned char* gvs = static_cast<const unsigned char*>(P.v_s) + row0 * P.ks_row;
  for (int i = lane; i < nvalid; i += 32) {
    tma_load_1d(ks + i * P.ks_stride, gks + static_cast<size_t>(i) * P.ks_row, P.ks_row, bar);
    tma_load_1d(vs + i * P.ks_stride, gvs + static_cast<size_t>(i) * P.ks_row, P.ks_row, bar);
  }
  if (P.r > 0) {
    const unsigned char* gzk = static_cast<const unsigned char*>(P.z_k) + row0 * P.z_row;
    const unsigned char* gzv = static_cast<const unsigned char*>(P.z_v) + row0 * P.z_row;
    for (int i = lane; i < nvalid; i += 32) {
      tma_load_1d(zk + i * P.z_stride, gzk + static_cast<size_t>(i) * P.z_row, P.z_row, bar);
      tma_load_1d(zv + i * P.z_stride, gzv + static_cast<size_t>(i) * P.z_row, P.z_row, bar);
    }
  }
}

}  // namespace

// ===================================================================== absorb
template <bool BF16>
__global__ void __launch_bounds__(128) lrkv_decode_absorb_kernel(const DecodePlan P) {
  pdl_trigger();
  const int h = blockIdx.x, b = blockIdx.y;
  if (h == 0 && b == 0 && threadIdx.x == 0) *P.status = 0u;
  if (P.r == 0) return;
  __shared__ float qs[256];
  for (int k = threadIdx.x; k < P.dh; k += blockDim.x)
    qs[k] = load_elem(P.q, (static_cast<size_t>(b) * P.H + h) * P.dh + k, BF16);
  __syncthreads();
  for (int c = threadIdx.x; c < P.r; c += blockDim.x) {
    float acc = 0.f;
    const size_t base = static_cast<size_t>(h) * P.dh * P.r + c;
    for (int k = 0; k < P.dh; ++k) acc = fmaf(qs[k], load_elem(P.b_k, base + static_cast<size_t>(k) * P.r, BF16), acc);
    P.p_abs[(static_cast<size_t>(b) * P.H + h) * P.r + c] = acc;
  }
}

// ====================================================================== split
template <bool BF16, int RMAX>
__global__ void __launch_bounds__(kMaxThreads, 1) lrkv_decode_split_kernel(const DecodePlan P) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ int s_ok;
  __shared__ int s_bad;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nwarps = blockDim.x >> 5;
  const int B = P.B, H = P.H, dh = P.dh, r = P.r, T = P.T;
  constexpr int ESZ = BF16 ? 2 : 4;

  uint64_t* bars = reinterpret_cast<uint64_t*>(smem);
  int* pre = reinterpret_cast<int*>(smem + P.off_prefix);
  unsigned char* q_sh = smem + P.off_q;
  float* p_sh = reinterpret_cast<float*>(smem + P.off_p);
  float* s_sh = reinterpret_cast<float*>(smem + P.off_s);
  unsigned char* w_sh = smem + P.off_w;
  float* alpha_sh = reinterpret_cast<float*>(smem + P.off_alpha);
  unsigned char* stages = smem + P.off_stage;

  // ---- 1. sequence starts (clamped lengths) --------------------------------
  if (tid == 0) s_bad = 0;
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

  // ---- 2. barriers and the first tiles -------------------------------------
  if (tid == 0) {
    for (int s = 0; s < P.stages; ++s) mbar_init(&bars[s], 1);
    fence_barrier_init();
  }
  // constant parts of the MMA operand tiles
  if constexpr (BF16) {
    for (int i = tid; i < P.Hp; i += blockDim.x) alpha_sh[i] = 1.f;
    __nv_bfloat16* wt = reinterpret_cast<__nv_bfloat16*>(w_sh);
    for (int i = tid; i < P.Hp * P.w_stride; i += blockDim.x) wt[i] = __float2bfloat16(0.f);
  }
  __syncthreads();

  TileWalk pw;  // producer walk (warp 0)
  bool p_more = walk_first(pw, pre, B, g0, g1);
  int issued = 0;
  if (warp == 0) {
    for (int s = 0; s < P.stages && p_more; ++s) {
      issue_tile(P, stages + static_cast<size_t>(s) * P.stage_bytes, &bars[s], pw, lane);
      ++issued;
      p_more = walk_next(pw, pre, B, g1, T);
    }
  }

  // operands produced by the absorb kernel are read only after this point
  pdl_wait();
  if (s_bad && tid == 0) record_status(P.status, kDevBounds);

  // ---- 3. per-thread roles -------------------------------------------------
  const int h = tid / P.lph;          // head of this lane (private branch, softmax)
  const int lt = tid % P.lph;         // lane within the head group
  const bool active = h < H;
  const int ppt = P.ppt;
  const int g = lane >> 2, q4 = lane & 3;  // MMA fragment coordinates

  // online-softmax state of head h (identical across the group's lanes)
  float m_run = -INFINITY;
  float l_part = 0.f;
  float acc_z[RMAX];
#pragma unroll
  for (int i = 0; i < RMAX; ++i) acc_z[i] = 0.f;
  // shared-value accumulators: bf16 -> MMA fragments; f32 -> per-lane columns
  float acc_v[kMaxValueTiles][4];
#pragma unroll
  for (int j = 0; j < kMaxValueTiles; ++j)
#pragma unroll
    for (int k = 0; k < 4; ++k) acc_v[j][k] = 0.f;
  const int mt = P.Hp / 16;
  const int n_vtiles = BF16 ? mt * (dh / 8) : 0;
  const int ltiles = BF16 ? mt * (T / 8) : 0;
  const int kps = BF16 ? (dh / 16) / P.ksplit : 0;

  TileWalk cw;
  walk_first(cw, pre, B, g0, g1);
  bool seg_start = true;
  int it = 0;
  bool ok = true;

  while (true) {
    const int s = it % P.stages;
    const uint32_t parity = static_cast<uint32_t>(it / P.stages) & 1u;
    unsigned char* st = stages + static_cast<size_t>(s) * P.stage_bytes;
    unsigned char* ks = st;
    unsigned char* vs = ks + T * P.ks_stride;
    unsigned char* zk = vs + T * P.ks_stride;
    unsigned char* zv = zk + T * P.z_stride;
    const int nvalid = min(T, cw.t_end - cw.t0);

    // ---- wait for the tile (bounded), refill the stage freed last round ----
    if (tid == 0) s_ok = mbar_wait_bounded(&bars[s], parity) ? 1 : 0;
    __syncthreads();  // (#1) also: every thread finished the previous tile
    if (!s_ok) { ok = false; break; }
    mbar_try_wait(&bars[s], parity);  // acquire the TMA writes in every thread
    if (warp == 0 && it > 0 && p_more) {
      const int sp = (it - 1) % P.stages;
      issue_tile(P, stages + static_cast<size_t>(sp) * P.stage_bytes, &bars[sp], pw, lane);
      ++issued;
      p_more = walk_next(pw, pre, B, g1, T);
    }

    // ---- segment set-up: q and p of sequence cw.b --------------------------
    if (seg_start) {
      const int b = cw.b;
      if constexpr (BF16) {
        const uint4* gq = reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(P.q) +
                                                         static_cast<size_t>(b) * H * dh);
        const int cpr = dh / 8;  // 16-byte chunks per row
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
      const float* gp = P.p_abs + static_cast<size_t>(b) * H * r;
      for (int i = tid; i < H * r; i += blockDim.x) p_sh[(i / r) * P.p_stride + (i % r)] = gp[i];
      __syncthreads();
      seg_start = false;
    }

    // ---- zero the rows past the piece's end (values must not carry NaN) ---
    if constexpr (BF16) {
      if (nvalid < T) {
        const int cpr = P.ks_stride / 16;
        for (int i = tid; i < (T - nvalid) * cpr; i += blockDim.x) {
          const int row = nvalid + i / cpr;
          *reinterpret_cast<uint4*>(vs + row * P.ks_stride + (i % cpr) * 16) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
    }

    // ---- scores: shared part (MMA warps) and private part (head lanes) ------
    if constexpr (BF16) {
      for (int item = warp; item < ltiles * P.ksplit; item += nwarps) {
        const int tile = item % ltiles, kg = item / ltiles;
        const int mi = tile / (T / 8), nj = tile % (T / 8);
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        for (int kk = kg * kps; kk < (kg + 1) * kps; ++kk) {
          uint32_t a0, a1, a2, a3, b0, b1;
          ldsm_x4(a0, a1, a2, a3, q_sh + ((mi * 16 + (lane & 15)) * P.q_stride + kk * 16 + (lane >> 4) * 8) * 2);
          ldsm_x2(b0, b1, ks + (nj * 8 + (lane & 7)) * P.ks_stride + (kk * 16 + ((lane >> 3) & 1) * 8) * 2);
          mma_bf16_16816(d, a0, a1, a2, a3, b0, b1);
        }
        float* sk = s_sh + (kg * P.Hp) * T;
        const int row = mi * 16 + g, col = nj * 8 + 2 * q4;
        sk[row * T + col] = d[0];
        sk[row * T + col + 1] = d[1];
        sk[(row + 8) * T + col] = d[2];
        sk[(row + 8) * T + col + 1] = d[3];
      }
    }
    // this lane's tokens lt, lt + lph, ... ; only the first `nvi` hold rows
    const int nvi = (nvalid > lt) ? min(ppt, (nvalid - lt + P.lph - 1) / P.lph) : 0;
    float sc[kMaxPPT];
    {
      float pr[kMaxPPT] = {0.f, 0.f, 0.f, 0.f};
      if (active && r > 0) {
        const unsigned char* z0 = zk + lt * P.z_stride + h * r * ESZ;
        const float* ph = p_sh + h * P.p_stride;
        const int tstride = P.lph * P.z_stride;
        switch (P.vec) {
          case 8: if constexpr (BF16) private_logits<BF16, 8, RMAX>(z0, tstride, nvi, ph, r, pr); break;
          case 4: private_logits<BF16, 4, RMAX>(z0, tstride, nvi, ph, r, pr); break;
          case 2: private_logits<BF16, 2, RMAX>(z0, tstride, nvi, ph, r, pr); break;
          default: private_logits<BF16, 1, RMAX>(z0, tstride, nvi, ph, r, pr); break;
        }
      }
      if constexpr (!BF16) {
        if (active) {
          const float* qh = reinterpret_cast<const float*>(q_sh) + h * P.q_stride;
#pragma unroll
          for (int i = 0; i < kMaxPPT; ++i)
            if (i < nvi)
              pr[i] += dot_f32(qh, reinterpret_cast<const float*>(ks + (lt + i * P.lph) * P.ks_stride), dh);
        }
      }
#pragma unroll
      for (int i = 0; i < kMaxPPT; ++i) sc[i] = pr[i];
    }
    if constexpr (BF16) __syncthreads();  // (#2) shared-part scores are in s_sh

    // ---- one online softmax per head over the summed scores ---------------
    float w[kMaxPPT];
    float alpha = 1.f;
    {
      float mloc = -INFINITY;
#pragma unroll
      for (int i = 0; i < kMaxPPT; ++i) {
        float v = -INFINITY;
        const int t = lt + i * P.lph;
        if (i < ppt && active && t < nvalid) {
          float sum = sc[i];
          if constexpr (BF16) {
            for (int kg = 0; kg < P.ksplit; ++kg) sum += s_sh[(kg * P.Hp + h) * T + t];
          }
          v = sum * P.scale_log2;
        }
        sc[i] = v;
        mloc = fmaxf(mloc, v);
      }
      for (int o = P.lph >> 1; o > 0; o >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, o));
      const float m_new = fmaxf(m_run, mloc);
      alpha = (m_new == -INFINITY) ? 1.f : exp2f(m_run - m_new);
      float lsum = 0.f;
#pragma unroll
      for (int i = 0; i < kMaxPPT; ++i) {
        w[i] = (sc[i] == -INFINITY) ? 0.f : exp2f(sc[i] - m_new);
        lsum += w[i];
      }
      l_part = l_part * alpha + lsum;
      m_run = m_new;
      if (active) {
#pragma unroll
        for (int i = 0; i < kMaxPPT; ++i) {
          if (i < ppt) {
            const int t = lt + i * P.lph;
            if constexpr (BF16)
              reinterpret_cast<__nv_bfloat16*>(w_sh)[h * P.w_stride + t] = __float2bfloat16(w[i]);
            else
              reinterpret_cast<float*>(w_sh)[h * P.w_stride + t] = w[i];
          }
        }
        if (BF16 && lt == 0) alpha_sh[h] = alpha;
      }
      if (active && r > 0) {
        const unsigned char* z0 = zv + lt * P.z_stride + h * r * ESZ;
        const int tstride = P.lph * P.z_stride;
        switch (P.vec) {
          case 8: if constexpr (BF16) private_values<BF16, 8, RMAX>(z0, tstride, nvi, w, alpha, r, acc_z); break;
          case 4: private_values<BF16, 4, RMAX>(z0, tstride, nvi, w, alpha, r, acc_z); break;
          case 2: private_values<BF16, 2, RMAX>(z0, tstride, nvi, w, alpha, r, acc_z); break;
          default: private_values<BF16, 1, RMAX>(z0, tstride, nvi, w, alpha, r, acc_z); break;
        }
      }
    }

    // ---- shared values ------------------------------------------------------
    if constexpr (BF16) {
      __syncthreads();  // (#3) W and alpha of every head are in shared memory
#pragma unroll
      for (int j = 0; j < kMaxValueTiles; ++j) {
        const int vt = warp + j * nwarps;
        if (vt < n_vtiles) {
          const int mi = vt / (dh / 8), nt = vt % (dh / 8);
          const float a_lo = alpha_sh[mi * 16 + g], a_hi = alpha_sh[mi * 16 + g + 8];
          acc_v[j][0] *= a_lo; acc_v[j][1] *= a_lo; acc_v[j][2] *= a_hi; acc_v[j][3] *= a_hi;
          const unsigned char* wrow = w_sh + ((mi * 16 + (lane & 15)) * P.w_stride) * 2;
          if ((T & 15) == 0) {
            for (int kk = 0; kk < T / 16; ++kk) {
              uint32_t a0, a1, a2, a3, b0, b1;
              ldsm_x4(a0, a1, a2, a3, wrow + (kk * 16 + (lane >> 4) * 8) * 2);
              ldsm_x2_trans(b0, b1, vs + (kk * 16 + (lane & 15)) * P.ks_stride + nt * 16);
              mma_bf16_16816(acc_v[j], a0, a1, a2, a3, b0, b1);
            }
          } else {
            uint32_t a0, a1, b0;
            ldsm_x2(a0, a1, wrow);
            ldsm_x1_trans(b0, vs + (lane & 7) * P.ks_stride + nt * 16);
            mma_bf16_1688(acc_v[j], a0, a1, b0);
          }
        }
      }
    } else {
      __syncwarp();  // the head group's W are in shared memory
      if (active) {
        const float* wrow = reinterpret_cast<const float*>(w_sh) + h * P.w_stride;
#pragma unroll
        for (int j = 0; j < kMaxValueTiles * 4; ++j) {
          const int k = lt + j * P.lph;
          if (k < dh) {
            float a = acc_v[j >> 2][j & 3] * alpha;
            for (int t = 0; t < nvalid; ++t)
              a = fmaf(wrow[t], reinterpret_cast<const float*>(vs + t * P.ks_stride)[k], a);
            acc_v[j >> 2][j & 3] = a;
          }
        }
      }
    }

    // ---- end of a (sequence, range) piece: write the partial ---------------
    const bool last_of_piece = cw.t0 + T >= cw.t_end;
    if (last_of_piece) {
      const int slot = cw.b + c;
      float l_tot = l_part;
      for (int o = P.lph >> 1; o > 0; o >>= 1) l_tot += __shfl_xor_sync(0xffffffffu, l_tot, o);
#pragma unroll
      for (int i = 0; i < RMAX; ++i)
        for (int o = P.lph >> 1; o > 0; o >>= 1) acc_z[i] += __shfl_xor_sync(0xffffffffu, acc_z[i], o);
      float* pacc = P.part_acc + static_cast<size_t>(slot) * H * (dh + r);
      if (active) {
        if (lt == 0) {
          P.part_ml[(static_cast<size_t>(slot) * H + h) * 2 + 0] = m_run;
          P.part_ml[(static_cast<size_t>(slot) * H + h) * 2 + 1] = l_tot;
        }
#pragma unroll
        for (int i = 0; i < RMAX; ++i)
          if (i < r && (i % P.lph) == lt) pacc[h * (dh + r) + dh + i] = acc_z[i];
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
      } else {
        if (active) {
#pragma unroll
          for (int j = 0; j < kMaxValueTiles * 4; ++j) {
            const int k = lt + j * P.lph;
            if (k < dh) pacc[h * (dh + r) + k] = acc_v[j >> 2][j & 3];
          }
        }
      }
      // fresh state for the next piece
      m_run = -INFINITY;
      l_part = 0.f;
#pragma unroll
      for (int i = 0; i < RMAX; ++i) acc_z[i] = 0.f;
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
template <bool BF16>
__global__ void __launch_bounds__(128) lrkv_decode_combine_kernel(const DecodePlan P) {
  extern __shared__ __align__(16) unsigned char csmem[];
  pdl_wait();
  const int h = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
  const int H = P.H, dh = P.dh, r = P.r;
  float* o = P.out + (static_cast<size_t>(b) * H + h) * dh;
  const int start = P.prefix[b], end = P.prefix[b + 1];
  if (end <= start) {
    for (int k = tid; k < dh; k += blockDim.x) o[k] = 0.f;
    if (tid == 0 && P.lse) P.lse[static_cast<size_t>(b) * H + h] = -INFINITY;
    return;
  }
  const long long N = P.meta[0], G = P.meta[1];
  const int c0 = cta_of_token(start, N, G), c1 = cta_of_token(end - 1, N, G);
  const int n = c1 - c0 + 1;
  float* wsl = reinterpret_cast<float*>(csmem);   // [n] per-piece weights
  float* zbar = wsl + n;                          // [r]
  __shared__ float red[32];
  __shared__ float s_M, s_L;

  float mloc = -INFINITY;
  for (int i = tid; i < n; i += blockDim.x)
    mloc = fmaxf(mloc, P.part_ml[(static_cast<size_t>(b + c0 + i) * H + h) * 2]);
  for (int off = 16; off > 0; off >>= 1) mloc = fmaxf(mloc, __shfl_xor_sync(0xffffffffu, mloc, off));
  if ((tid & 31) == 0) red[tid >> 5] = mloc;
  __syncthreads();
  if (tid == 0) {
    float M = -INFINITY;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) M = fmaxf(M, red[i]);
    s_M = M;
  }
  __syncthreads();
  const float M = s_M;
  float lloc = 0.f;
  for (int i = tid; i < n; i += blockDim.x) {
    const size_t sl = (static_cast<size_t>(b + c0 + i) * H + h) * 2;
    const float wgt = exp2f(P.part_ml[sl] - M);
    wsl[i] = wgt;
    lloc += wgt * P.part_ml[sl + 1];
  }
  for (int off = 16; off > 0; off >>= 1) lloc += __shfl_xor_sync(0xffffffffu, lloc, off);
  __syncthreads();
  if ((tid & 31) == 0) red[tid >> 5] = lloc;
  __syncthreads();
  if (tid == 0) {
    float L = 0.f;
    for (int i = 0; i < (int)(blockDim.x >> 5); ++i) L += red[i];
    s_L = L;
  }
  __syncthreads();
  const float inv_l = 1.f / s_L;
  const int width = dh + r;
  float oshared[2] = {0.f, 0.f};
  for (int j = tid; j < width; j += blockDim.x) {
    float a = 0.f;
    for (int i = 0; i < n; ++i)
      a = fmaf(wsl[i], P.part_acc[(static_cast<size_t>(b + c0 + i) * H + h) * width + j], a);
    a *= inv_l;
    if (j < dh) oshared[j / blockDim.x] = a; else zbar[j - dh] = a;
  }
  __syncthreads();
  for (int k = tid, jj = 0; k < dh; k += blockDim.x, ++jj) {
    float a = oshared[jj];
    const size_t base = (static_cast<size_t>(h) * dh + k) * r;
    for (int cc = 0; cc < r; ++cc) a = fmaf(load_elem(P.b_v, base + cc, BF16), zbar[cc], a);
    o[k] = a;
  }
  if (tid == 0 && P.lse) P.lse[static_cast<size_t>(b) * H + h] = (M + log2f(s_L)) * kLn2;
}

// ======================================================================= host
namespace {

int env_int(const char* name, int dflt) {
  const char* v = std::getenv(name);
  return (v && *v) ? std::atoi(v) : dflt;
}

template <bool BF16, int RMAX>
lrkv_status launch_split(const DecodePlan& P, cudaStream_t stream) {
  auto kern = lrkv_decode_split_kernel<BF16, RMAX>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P.smem_bytes) != cudaSuccess)
    return LRKV_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid);
  cfg.blockDim = dim3(P.nthreads);
  cfg.dynamicSmemBytes = P.smem_bytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, P) == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

template <bool BF16>
lrkv_status launch_all(const DecodePlan& P, cudaStream_t stream) {
  lrkv_decode_absorb_kernel<BF16><<<dim3(P.H, P.B), 128, 0, stream>>>(P);
  if (cudaGetLastError() != cudaSuccess) return LRKV_ERR_CUDA;
  lrkv_status st;
  if (P.r <= 16) st = launch_split<BF16, 16>(P, stream);
  else if (P.r <= 32) st = launch_split<BF16, 32>(P, stream);
  else st = launch_split<BF16, 64>(P, stream);
  if (st != LRKV_OK) return st;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.H, P.B);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = P.combine_smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (P.combine_smem > 48 * 1024 &&
      cudaFuncSetAttribute(lrkv_decode_combine_kernel<BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           P.combine_smem) != cudaSuccess)
    return LRKV_ERR_CUDA;
  if (cudaLaunchKernelEx(&cfg, lrkv_decode_combine_kernel<BF16>, P) != cudaSuccess) return LRKV_ERR_CUDA;
  return LRKV_OK;
}

template <bool BF16, int RMAX>
lrkv_status occupancy_of(const DecodePlan& P, int* occ) {
  auto kern = lrkv_decode_split_kernel<BF16, RMAX>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P.smem_bytes) != cudaSuccess)
    return LRKV_ERR_CUDA;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occ, kern, P.nthreads, P.smem_bytes) == cudaSuccess
             ? LRKV_OK
             : LRKV_ERR_CUDA;
}

lrkv_status split_occupancy(const DecodePlan& P, int* occ) {
  if (P.bf16) {
    if (P.r <= 16) return occupancy_of<true, 16>(P, occ);
    if (P.r <= 32) return occupancy_of<true, 32>(P, occ);
    return occupancy_of<true, 64>(P, occ);
  }
  if (P.r <= 16) return occupancy_of<false, 16>(P, occ);
  if (P.r <= 32) return occupancy_of<false, 32>(P, occ);
  return occupancy_of<false, 64>(P, occ);
}

}  // namespace

lrkv_status decode_make_plan(const lrkv_dims& d, int num_sms, DecodePlan& P, size_t* ws_bytes) {
  std::memset(&P, 0, sizeof(P));
  P.B = d.batch; P.H = d.heads; P.dh = d.head_dim; P.r = d.rank; P.max_len = d.max_len;
  const float scale = d.scale > 0.f ? d.scale : 1.f / std::sqrt(static_cast<float>(d.head_dim));
  P.scale_log2 = scale * kLog2e;
  P.bf16 = d.dtype == LRKV_BF16;
  P.esz = P.bf16 ? 2 : 4;
  const int H = P.H, dh = P.dh, r = P.r;

  // lanes per head: as many as fit 256 threads, at most a warp
  int lph = 32;
  while (lph > 1 && H * lph > kMaxThreads) lph >>= 1;
  if (H * lph > kMaxThreads) return LRKV_ERR_UNSUPPORTED;
  P.lph = lph;
  P.nthreads = std::max(128, round_up(H * lph, 32));
  if (P.nthreads > kMaxThreads) return LRKV_ERR_UNSUPPORTED;
  const int nwarps = P.nthreads / 32;

  P.ks_row = dh * P.esz;
  P.z_row = H * r * P.esz;
  P.ks_stride = odd_chunk_stride(P.ks_row);
  P.z_stride = r > 0 ? odd_chunk_stride(P.z_row) : 0;
  const int per_token = 2 * (P.ks_stride + P.z_stride);

  if (P.bf16) {
    P.vec = (r % 8 == 0) ? 8 : (r % 4 == 0) ? 4 : (r % 2 == 0) ? 2 : 1;
    P.Hp = round_up(H, 16);
  } else {
    P.vec = (r % 4 == 0) ? 4 : (r % 2 == 0) ? 2 : 1;
    P.Hp = H;
  }
  if (r == 0) P.vec = 1;

  // tile: T = ppt * lph tokens, a multiple of 8, about 48 KB of rows per stage
  const int stage_target = env_int("LRKV_DECODE_STAGE_KB", 48) * 1024;
  int best = 0;
  for (int ppt = 1; ppt <= kMaxPPT; ppt *= 2) {
    const int T = ppt * lph;
    if (T % 8 != 0 || T > 64) continue;
    if (best == 0 || T * per_token <= stage_target) best = T;
  }
  const int forced_T = env_int("LRKV_DECODE_TILE", 0);
  if (forced_T > 0 && forced_T % lph == 0 && forced_T % 8 == 0 && forced_T / lph <= kMaxPPT) best = forced_T;
  if (best == 0) return LRKV_ERR_UNSUPPORTED;
  P.T = best;
  P.ppt = P.T / lph;

  if (P.bf16) {
    const int mt = P.Hp / 16;
    const int ltiles = mt * (P.T / 8);
    const int ksteps = dh / 16;
    P.ksplit = 1;
    for (int k = ksteps; k >= 1; --k)
      if (ksteps % k == 0 && ltiles * k <= nwarps) { P.ksplit = k; break; }
    if (mt * (dh / 8) > kMaxValueTiles * nwarps) return LRKV_ERR_UNSUPPORTED;
    P.q_stride = dh + 8;
    P.w_stride = ((P.T / 8) & 1) ? P.T : P.T + 8;
  } else {
    if (dh > kMaxValueTiles * 4 * lph) return LRKV_ERR_UNSUPPORTED;
    P.ksplit = 0;
    P.q_stride = ((dh / 4) & 1) ? dh : dh + 4;
    P.w_stride = P.T;
  }
  {
    const int r4 = round_up(std::max(r, 1), 4);
    P.p_stride = ((r4 / 4) & 1) ? r4 : r4 + 4;
  }

  // shared-memory carve-up
  int off = 64;  // mbarriers
  P.off_prefix = off; off = round_up(off + (P.B + 1) * 4, 16);
  P.off_q = off; off = round_up(off + P.Hp * P.q_stride * P.esz, 16);
  P.off_p = off; off = round_up(off + H * P.p_stride * 4, 16);
  P.off_s = off; off = round_up(off + (P.bf16 ? P.ksplit * P.Hp * P.T * 4 : 0), 16);
  P.off_w = off; off = round_up(off + P.Hp * P.w_stride * P.esz, 16);
  P.off_alpha = off; off = round_up(off + P.Hp * 4, 128);
  P.off_stage = off;
  P.stage_bytes = round_up(P.T * per_token, 128);
  // Two CTAs per SM when at least two stages fit in half the SM's shared
  // memory (independent CTAs overlap one another's barriers); else one CTA
  // with a deeper ring.
  const int max_stages = env_int("LRKV_DECODE_STAGES", 4);
  const int want_cps = env_int("LRKV_DECODE_CTAS_PER_SM", 0);
  int cps = 0, stages = 0;
  for (int try_cps = 2; try_cps >= 1; --try_cps) {
    if (want_cps > 0 && try_cps != want_cps) continue;
    const int budget = (try_cps == 2 ? 113 : 227) * 1024 - off;
    const int st = std::min(max_stages, budget / P.stage_bytes);
    if (st >= 2) { cps = try_cps; stages = st; break; }
  }
  if (stages < 2) return LRKV_ERR_UNSUPPORTED;
  P.stages = stages;
  P.smem_bytes = off + stages * P.stage_bytes;
  // resident CTAs per SM as the hardware will actually schedule them
  // (registers may allow fewer than shared memory does)
  int occ = cps;
  if (split_occupancy(P, &occ) != LRKV_OK) return LRKV_ERR_CUDA;
  P.grid = env_int("LRKV_DECODE_GRID", num_sms * std::max(1, std::min(occ, cps)));
  P.min_tokens = env_int("LRKV_DECODE_MIN_TOKENS", 2 * P.T);
  const int slots = P.B + P.grid;
  P.combine_smem = (P.grid + 1 + r) * 4;

  // workspace: status | meta | prefix | p | part_ml | part_acc
  size_t w = 256;
  w += static_cast<size_t>(round_up(P.B + 1, 64)) * 4;
  w += static_cast<size_t>(P.B) * H * std::max(r, 1) * 4;
  w = (w + 255) / 256 * 256;
  w += static_cast<size_t>(slots) * H * 2 * 4;
  w = (w + 255) / 256 * 256;
  w += static_cast<size_t>(slots) * H * (dh + r) * 4;
  *ws_bytes = w;
  return LRKV_OK;
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
  off += static_cast<size_t>(P.B + P.grid) * P.H * 2 * 4;
  off = (off + 255) / 256 * 256;
  P.part_acc = reinterpret_cast<float*>(base + off);
}

lrkv_status decode_launch(const DecodePlan& P, void* stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  return P.bf16 ? launch_all<true>(P, s) : launch_all<false>(P, s);
}

}  // namespace lrkv
