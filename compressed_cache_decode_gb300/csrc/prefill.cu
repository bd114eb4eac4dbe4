// prefill.cu — causal attention of a block of queries against the factored
// LRKV cache on the tensor cores (tcgen05 + TMEM + TMA, sm_103a).
//
// For a query row i of head h the logits are a dense contraction over the
// concatenated [q_h | q_h B_h^K] . [k_s | z_k,h] (K = d_h + r), one causal
// softmax, and the values [v_s | z_v,h] (N = d_h + r), finally lifted
//   o_h = O_s / l + (O_z / l) (B_h^V)^T
// ("Low-Rank Key Value Attention：中文研读笔记", §2.4, Eqs. (6)-(7); "Low-Rank
// Key Value Attention | What a shared cache can preserve", §3).
//
// Persistent: one CTA per SM works through items (sequence b, head h, 128
// query rows), heaviest first, dealt out in a snake; an item's copies, Pq and
// first scores overlap the previous item's last tiles and output.  Warps 0-7
// run the softmax and the epilogue (one query row per lane, each row split
// over two warps by key columns), warp 8 issues TMA, one thread of warp 9
// issues every MMA:
//   Pq   = Q B_h^K          (TMEM, then split in place into two bf16 parts,
//                           high and low, so the latent scores keep about 16
//                           significant bits; both are TMEM A operands)
//   S_j  = Q K_s,j^T + Pq Z_k,j^T        two TMEM buffers, S_{j+1} runs while
//                                        the softmax of tile j does; two key
//                                        and two value stages
//   [O_s | O_z] += P_j [V_s,j | Z_v,j]   one N = 192 MMA per 16 keys, P_j read
//                                        straight from TMEM (the softmax
//                                        overwrites S_j with bf16 P_j)
//   O_s += bf16(O_z) (B_h^V)^T           the lift, once
// Scores are taken against a per-row reference max; the accumulators are
// rescaled only when a row's max grows by more than 2^8 (then the row's own
// TMEM lane is read, scaled and written back).
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>

#include "host_cache.h"
#include "lrkv.h"
#include "trace.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lrkv {

namespace {

constexpr int kBQ = 128, kBK = 128, kDH = 128, kR = 64;
constexpr int kThreads = 320;  // warps 0-7 softmax, 8 TMA, 9 MMA
constexpr float kPfLog2e = 1.44269504088896340736f;
constexpr float kPfLn2 = 0.69314718055994530942f;
// shared-memory carve-up (bytes, 1024-aligned)
constexpr int kOffQ = 0;                          // Q: [2 halves][128][64]             32 KB
constexpr int kKStage = 49152;                    // K_s [2][128][64] 32 KB + Z_k [128][64] 16 KB
                                                  // (a value stage: V_s + Z_v, same shape)
constexpr int kOffK = kOffQ + 32768;              // 2 key stages; after the last scores the last
                                                  // tile's stage holds B^V and then bf16(O_z)
constexpr int kOffV = kOffK + 2 * kKStage;        // 2 value stages (B^K in stage 1 until Pq is done)
constexpr int kSmem = kOffV + 2 * kKStage + 1024; // + alignment slack
// TMEM columns
constexpr uint32_t kColS = 0;      // S_0 [0,128), S_1 [128,256)
constexpr uint32_t kColOs = 256;   // O_s [256,384)
constexpr uint32_t kColOz = 384;   // O_z [384,448)
constexpr uint32_t kColPq = 448;   // fp32 Q B^K [448,512), then bf16 high part [448,480), low [480,512)

struct PrefillParams {
  int B, H, Tq, max_len;
  int out_v8;  // out is 32-byte aligned: 256-bit stores
  float scale_log2;
  const int32_t* seq_lens;
  const float* key_scale;  // [B][H][max_len] reciprocal key RMS, or NULL
  // paged cache: row t of sequence b is row t & (2^page_shift - 1) of page
  // block_table[b][t >> page_shift] (page_size >= 128: a key tile never spans
  // two pages); NULL: [B][max_len]
  const int32_t* block_table;
  int max_blocks, page_shift, num_pages;
  float* out;
  float* lse;
  uint32_t* status;
};

struct PrefillMaps {
  CUtensorMap q;    // {64, Tq, 2, H, B}
  CUtensorMap ks;   // {64, rows, 2, seqs}: (rows, seqs) = (max_len, B), or (page_size, pages)
  CUtensorMap vs;   // {64, rows, 2, seqs}
  CUtensorMap zk;   // {r, H, rows, seqs}
  CUtensorMap zv;   // {r, H, rows, seqs}
  CUtensorMap bk;   // {r, dh, H}
  CUtensorMap bv;   // {r, dh, H}
};

// L2 prefetch of a 5-D tensor box (no destination, no completion)
__device__ __forceinline__ void tma_prefetch_5d(const void* tmap, int x, int y, int z, int w, int v) {
  asm volatile("cp.async.bulk.prefetch.tensor.5d.L2.global.tile [%0, {%1, %2, %3, %4, %5}];" ::"l"(tmap), "r"(x),
               "r"(y), "r"(z), "r"(w), "r"(v)
               : "memory");
}

// byte offset of element (row, col) in a [rows][64] bf16 tile written with
// the 128-byte swizzle
__device__ __forceinline__ uint32_t sw128(int row, int col) {
  const uint32_t chunk = static_cast<uint32_t>(col >> 3) ^ static_cast<uint32_t>(row & 7);
  return static_cast<uint32_t>(row) * 128u + chunk * 16u + static_cast<uint32_t>(col & 7) * 2u;
}

__device__ __forceinline__ void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// 2^x on the MUFU pipe (flush-to-zero; 2^-inf = +0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// max of three (sm_100 three-input max)
__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float y;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(y) : "f"(a), "f"(b), "f"(c));
  return y;
}

// 32 TMEM columns of this warp's 32 lanes, load and wait in one statement so
// that no use of the registers can be scheduled before the data arrived
__device__ __forceinline__ void tmem_ld32_wait(uint32_t taddr, uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
      : "r"(taddr)
      : "memory");
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&v)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

// 64 TMEM columns (two 32-column loads, one wait)
__device__ __forceinline__ void tmem_ld64_wait(uint32_t taddr, uint32_t (&v)[64]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]),
        "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]),
        "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]),
        "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]),
        "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]),
        "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]),
        "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]),
        "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
      : "r"(taddr), "r"(taddr + 32u)
      : "memory");
}

// A work item: (sequence b, head h, 128 query rows from q0) and its keys.
struct Item {
  int b, h, q0, L, off, nkt;
  bool valid, bad_len;
};

// Item k of CTA c among G: items ordered heaviest (latest query tile) first,
// dealt to the CTAs in a snake (c, then G - 1 - c on the next round), which
// evens out the CTAs' totals.
__device__ __forceinline__ Item item_of(const PrefillParams& p, int c, int G, int k) {
  Item it;
  const int X = (p.Tq + kBQ - 1) / kBQ, HB = p.H * p.B;
  const int idx = k * G + ((k & 1) ? G - 1 - c : c);
  it.valid = idx < X * HB;
  it.bad_len = false;
  it.b = it.h = it.q0 = it.L = it.off = 0;
  it.nkt = 1;
  if (!it.valid) return it;
  const int qtr = idx / HB, hb = idx - qtr * HB;
  it.h = hb % p.H;
  it.b = hb / p.H;
  it.q0 = (X - 1 - qtr) * kBQ;
  int L = p.seq_lens[it.b];
  if (L < p.Tq || L > p.max_len) {
    it.bad_len = true;
    L = min(max(L, p.Tq), p.max_len);
  }
  it.L = L;
  it.off = L - p.Tq;  // absolute position of query 0
  const int last_key = min(L - 1, it.off + it.q0 + kBQ - 1);
  it.nkt = last_key / kBK + 1;
  return it;
}

// Bounded wait that also gives up as soon as another thread of the CTA
// recorded a failure (so that a failed CTA leaves its item loop quickly).
__device__ __forceinline__ bool pwait(uint64_t* bar, uint32_t parity, volatile int* fail) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (*fail) return false;
    if (clock64() - t0 > kWaitLimitCycles) {
      *fail = 1;
      return false;
    }
  }
  return true;
}

__device__ __forceinline__ void st_global_v8(float* dst, const float (&v)[8]) {
  asm volatile("st.global.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dst), "f"(v[0]), "f"(v[1]), "f"(v[2]),
               "f"(v[3]), "f"(v[4]), "f"(v[5]), "f"(v[6]), "f"(v[7])
               : "memory");
}

}  // namespace

// Tensor-map (sequence or page, row) of key tile row `row` of sequence b; a
// page outside the pool is recorded (its copy reads zeros).
__device__ __forceinline__ int kv_seq(const PrefillParams& p, int b, int row, int& r_out) {
  if (!p.block_table) {
    r_out = row;
    return b;
  }
  const int pg = __ldg(p.block_table + static_cast<size_t>(b) * p.max_blocks + (row >> p.page_shift));
  r_out = row & ((1 << p.page_shift) - 1);
  if (pg < 0 || pg >= p.num_pages) atomicOr(p.status, 2u);
  return pg;
}

// KS: the scores are multiplied by the keys' cached RMSNorm scales
template <bool KS>
__global__ void __launch_bounds__(kThreads, 1)
    lrkv_prefill_kernel(const PrefillParams p, const __grid_constant__ PrefillMaps maps) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ uint64_t bar_q, bar_pq, bar_pqs, bar_ozs, bar_bv, bar_pv, bar_all, bar_lift, bar_ofree;
  __shared__ uint64_t bar_k0, bar_g[2], bar_ve[2], bar_sf[2], bar_pf[2];
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;
  __shared__ float xchg[2][kBQ];  // the two halves of a row swap their maxima, at the end their sums
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  volatile int* fail = &s_fail;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cta = blockIdx.x, G = gridDim.x;

  if (threadIdx.x == 0) {
    mbar_init(&bar_q, 1); mbar_init(&bar_pq, 1); mbar_init(&bar_pqs, 256); mbar_init(&bar_bv, 1);
    mbar_init(&bar_pv, 1); mbar_init(&bar_all, 1); mbar_init(&bar_lift, 1); mbar_init(&bar_ofree, 256);
    mbar_init(&bar_ozs, 256);
    mbar_init(&bar_k0, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&bar_g[i], 1); mbar_init(&bar_ve[i], 1);
      mbar_init(&bar_sf[i], 1); mbar_init(&bar_pf[i], 256);
    }
    s_fail = 0;
    fence_barrier_init();
    // the first item's copies go out before anything else: Q and B^K (the
    // first MMA's operands; B^K sits in value stage 1 until Pq is done) and K_0
    const Item it = item_of(p, cta, G, 0);
    if (it.valid) {
      mbar_arrive_expect_tx(&bar_q, 32768 + 16384);
      tma_load_5d(smem + kOffQ, &maps.q, 0, it.q0, 0, it.h, it.b, &bar_q);
      tma_load_3d(smem + kOffV + kKStage, &maps.bk, 0, 0, it.h, &bar_q);
      mbar_arrive_expect_tx(&bar_k0, kKStage);
      int r0;
      const int s0 = kv_seq(p, it.b, 0, r0);
      tma_load_4d(smem + kOffK, &maps.ks, 0, r0, 0, s0, &bar_k0);
      tma_load_4d(smem + kOffK + 32768, &maps.zk, 0, it.h, r0, s0, &bar_k0);
    }
  }
  if (warp == 0) tmem_alloc(&tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_base;
  const uint32_t sQ = smem_u32(smem + kOffQ), sK = smem_u32(smem + kOffK), sV = smem_u32(smem + kOffV);

  if (warp == 8) {
    // ================================================================ TMA ====
    // One box per operand tile: the two 64-column halves of a 128-row tile
    // of Q, k_s or v_s come in one copy (the halves are a tensor-map
    // dimension).  Tiles are numbered J over all of this CTA's items; group
    // J = {V_J, K_{J+1}} (four copies, 96 KB, one barrier; K_{J+1} may be the
    // next item's first key tile) goes out once P_{J-2} V_{J-2} is done, which
    // frees value stage J % 2 and, the MMAs completing in issue order, the key
    // stage of S_{J-1}.  When J - 1 ended an item, that key stage held the
    // item's lift operands (B^V, bf16(O_z)) and the next item's B^K, so the
    // group also waits for that lift and for the next Q B^K.  The TMA unit
    // serves copies that complete on one barrier faster than copies spread
    // over several.
    if (lane == 0) {
      auto load_k = [&](int j, const Item& w, int kt, uint64_t* bar) {
        unsigned char* dst = smem + kOffK + (j & 1) * kKStage;
        int rw;
        const int sq = kv_seq(p, w.b, kt * kBK, rw);
        tma_load_4d(dst, &maps.ks, 0, rw, 0, sq, bar);
        tma_load_4d(dst + 32768, &maps.zk, 0, w.h, rw, sq, bar);
      };
      auto load_v = [&](int j, const Item& w, int kt, uint64_t* bar) {
        unsigned char* dst = smem + kOffV + (j & 1) * kKStage;
        int rw;
        const int sq = kv_seq(p, w.b, kt * kBK, rw);
        tma_load_4d(dst, &maps.vs, 0, rw, 0, sq, bar);
        tma_load_4d(dst + 32768, &maps.zv, 0, w.h, rw, sq, bar);
      };
      bool ok = true;
      int J = 0;  // this item's first tile
      Item it = item_of(p, cta, G, 0);
      for (int k = 0; ok && it.valid; ++k) {
        const Item nx = item_of(p, cta, G, k + 1);
        if (nx.valid) tma_prefetch_5d(&maps.q, 0, nx.q0, 0, nx.h, nx.b);  // its queries start moving into L2
        for (int t = 0; ok && t < it.nkt; ++t) {
          const int Jt = J + t;
          if (Jt == 1)  // value stage 1 held the first B^K, key stage 0 held K_0
            ok = pwait(&bar_pq, 0, fail) && pwait(&bar_sf[0], 0, fail);
          else if (Jt >= 2)
            ok = pwait(&bar_ve[Jt & 1], static_cast<uint32_t>((Jt - 2) >> 1) & 1u, fail);
          // an item's first scores are issued after the previous item's last
          // P V, so for its second group that P V does not vouch for them
          if (ok && t == 1 && k > 0) ok = pwait(&bar_sf[J & 1], static_cast<uint32_t>(J >> 1) & 1u, fail);
          const bool more_k = t + 1 < it.nkt || nx.valid;
          if (ok && t == 0 && k > 0 && more_k)
            ok = pwait(&bar_lift, static_cast<uint32_t>(k - 1) & 1u, fail) &&
                 pwait(&bar_pq, static_cast<uint32_t>(k) & 1u, fail);
          if (!ok) break;
          uint64_t* gb = &bar_g[Jt & 1];
          mbar_arrive_expect_tx(gb, more_k ? 2 * kKStage : kKStage);
          load_v(Jt, it, t, gb);
          if (t + 1 < it.nkt)
            load_k(Jt + 1, it, t + 1, gb);
          else if (nx.valid)
            load_k(Jt + 1, nx, 0, gb);
        }
        if (!ok) break;
        // the item's last scores done: its key stage takes B^V (lift) and the
        // next item's B^K; the next item's Q replaces this one's
        const int Jl = J + it.nkt - 1;
        ok = pwait(&bar_sf[Jl & 1], static_cast<uint32_t>(Jl >> 1) & 1u, fail);
        if (!ok) break;
        unsigned char* stg = smem + kOffK + (Jl & 1) * kKStage;
        mbar_arrive_expect_tx(&bar_bv, 16384);
        tma_load_3d(stg, &maps.bv, 0, 0, it.h, &bar_bv);
        if (nx.valid) {
          mbar_arrive_expect_tx(&bar_q, 32768 + 16384);
          tma_load_5d(smem + kOffQ, &maps.q, 0, nx.q0, 0, nx.h, nx.b, &bar_q);
          tma_load_3d(stg + 32768, &maps.bk, 0, 0, nx.h, &bar_q);
        }
        J += it.nkt;
        it = nx;
      }
    }
  } else if (warp == 9) {
    // =============================================================== MMA ====
    if (lane == 0) {
      const uint32_t id_pq = idesc_bf16(kBQ, kR, 0, 1), id_s = idesc_bf16(kBQ, kBK, 0, 0);
      // values: one N = d_h + r = 192 MMA per 16 keys; a value stage's v_s
      // halves and z_v are three 64-column blocks 16 KB apart, O_s and O_z
      // adjacent TMEM columns
      const uint32_t id_v = idesc_bf16(kBQ, kDH + kR, 0, 1), id_l = idesc_bf16(kBQ, kDH, 0, 0);
      auto issue_s = [&](int j) {
        const uint32_t kbase = sK + (j & 1) * kKStage;
        const uint32_t d = tmem + kColS + (j & 1) * 128;
        for (int kk = 0; kk < kDH / 16; ++kk) {
          const uint32_t o = (kk >> 2) * 16384 + (kk & 3) * 32;
          tc_mma_ss(d, smem_desc(sQ + o, 16, 1024, 2), smem_desc(kbase + o, 16, 1024, 2), id_s, kk > 0);
        }
        for (int kk = 0; kk < kR / 16; ++kk) {  // A = Pq parts from TMEM, 8 columns per 16 values
          const uint64_t zd = smem_desc(kbase + 32768 + kk * 32, 16, 1024, 2);
          tc_mma_ts(d, tmem + kColPq + kk * 8, zd, id_s, 1);
          tc_mma_ts(d, tmem + kColPq + 32 + kk * 8, zd, id_s, 1);
        }
        tc_commit(&bar_sf[j & 1]);
      };
      // Pq = Q B^K : M=128, N=64, K=128; B^K tile is [dh][r], r contiguous (MN-major)
      auto issue_pq = [&](int k, uint32_t sBk) {
        bool good = pwait(&bar_q, static_cast<uint32_t>(k) & 1u, fail);
        tc_fence_after();
        if (!good) return false;
        for (int kk = 0; kk < kDH / 16; ++kk) {
          const uint64_t ad = smem_desc(sQ + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024, 2);
          tc_mma_ss(tmem + kColPq, ad, smem_desc(sBk + kk * 2048, 16384, 1024, 2), id_pq, kk > 0);
        }
        tc_commit(&bar_pq);
        return true;
      };
      int J = 0;
      Item it = item_of(p, cta, G, 0);
      bool ok = true;
      for (int k = 0; ok && it.valid; ++k) {
        if (it.bad_len) atomicOr(p.status, 2u);
        // the first item's B^K sits in value stage 1, a later one's in the key
        // stage of the previous item's last tile (after that item's lift)
        if (!issue_pq(k, k == 0 ? sV + kKStage : sK + ((J - 1) & 1) * kKStage + 32768)) { ok = false; break; }
        ok = pwait(&bar_pqs, static_cast<uint32_t>(k) & 1u, fail);  // bf16 Pq (high, low) is in TMEM
        // K_J: the first item's came with the set-up; a later item's came in
        // the previous item's last group, waited for before its last P V
        if (ok && k == 0) ok = pwait(&bar_k0, 0u, fail);
        tc_fence_after();
        if (!ok) break;
        issue_s(J);
        for (int t = 0; t < it.nkt; ++t) {
          const int Jt = J + t;
          const uint32_t gpar = static_cast<uint32_t>(Jt >> 1) & 1u;  // group Jt = {V_Jt, K_Jt+1}
          if (t + 1 < it.nkt) {
            if (!pwait(&bar_g[Jt & 1], gpar, fail)) { ok = false; break; }
            tc_fence_after();
            issue_s(Jt + 1);
          }
          if (!pwait(&bar_pf[Jt & 1], static_cast<uint32_t>(Jt >> 1) & 1u, fail) ||
              !pwait(&bar_g[Jt & 1], gpar, fail)) { ok = false; break; }
          // the first P V of an item overwrites O: the previous item's O must be read out
          if (t == 0 && k > 0 && !pwait(&bar_ofree, static_cast<uint32_t>(k - 1) & 1u, fail)) { ok = false; break; }
          tc_fence_after();
          const int vs = Jt & 1;
          const int nv = it.L - t * kBK;  // rows of this value tile inside the history
          if (nv < kBK) {
            // rows past the history may hold anything; P is 0 there, so make them 0
            for (int row = max(nv, 0); row < kBK; ++row)
              for (int box = 0; box < 3; ++box)
                for (int ch = 0; ch < 8; ++ch)
                  *reinterpret_cast<uint4*>(smem + kOffV + vs * kKStage + box * 16384 + row * 128 + ch * 16) =
                      make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();
          }
          const uint32_t pa = tmem + kColS + (Jt & 1) * 128;  // bf16 P, 2 per column
          for (int kk = 0; kk < kBK / 16; ++kk) {
            const uint32_t vo = sV + vs * kKStage + kk * 2048;
            tc_mma_ts(tmem + kColOs, pa + kk * 8, smem_desc(vo, 16384, 1024, 2), id_v, (t > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&bar_ve[vs]);
          tc_commit(&bar_pv);
        }
        if (!ok) break;
        tc_commit(&bar_all);
        const int Jl = J + it.nkt - 1;
        // lift: O_s += bf16(O_z) (B^V)^T : M=128, N=128 (dh), K=64 (r); B^V and
        // bf16(O_z) sit in the key stage of the item's last tile
        ok = pwait(&bar_bv, static_cast<uint32_t>(k) & 1u, fail) && pwait(&bar_ozs, static_cast<uint32_t>(k) & 1u, fail);
        tc_fence_after();
        if (!ok) break;
        const uint32_t sBv = sK + (Jl & 1) * kKStage, sOz = sBv + 16384;
        for (int kk = 0; kk < kR / 16; ++kk)
          tc_mma_ss(tmem + kColOs, smem_desc(sOz + kk * 32, 16, 1024, 2), smem_desc(sBv + kk * 32, 16, 1024, 2),
                    id_l, 1);
        tc_commit(&bar_lift);
        J += it.nkt;
        it = item_of(p, cta, G, k + 1);
      }
      if (!ok) *fail = 1;
    }
  } else if (warp < 8) {
    // ========================================================= softmax ====
    // Warps w and w + 4 read the same 32 TMEM lanes (lane quadrant w % 4): one
    // query row per lane; the first warp takes key columns 0-63 of every tile,
    // the second columns 64-127.  The two halves of a row swap their maxima
    // and, at the end of an item, their sums through shared memory, each swap
    // between two 64-thread named barriers of the quadrant.  These warps never
    // leave their loops early (a failed wait is skipped, not retried), so the
    // named barriers always pair up.
    const int quad = warp & 3, half = warp >> 2;
    const int row = quad * 32 + lane;                // query row in the tile
    const uint32_t lane_off = static_cast<uint32_t>(quad * 32) << 16;
    const float sc = p.scale_log2;
    bool ok = true;
    // Pq -> high and low bf16 parts, written back over the fp32 Pq columns
    // (high [448,480), low [480,512)) as the A operands of S += Pq Z_k^T;
    // each half converts its 32 values once both halves have read theirs
    auto split_pq = [&](int k) {
      ok = ok && pwait(&bar_pq, static_cast<uint32_t>(k) & 1u, fail);
      tc_fence_after();
      uint32_t v[32], hi[16], lo[16];
      tmem_ld32_wait(tmem + lane_off + kColPq + half * 32, v);
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        const float f0 = __uint_as_float(v[e]), f1 = __uint_as_float(v[e + 1]);
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(f0, f1);
        const __nv_bfloat162 l2 = __floats2bfloat162_rn(f0 - __low2float(h2), f1 - __high2float(h2));
        hi[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
        lo[e / 2] = *reinterpret_cast<const uint32_t*>(&l2);
      }
      named_bar(1 + quad, 64);
      tmem_st16(tmem + lane_off + kColPq + half * 16, hi);
      tmem_st16(tmem + lane_off + kColPq + 32 + half * 16, lo);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive_cta(&bar_pqs);
    };
    int J = 0;
    Item it = item_of(p, cta, G, 0);
    if (it.valid) split_pq(0);
    for (int k = 0; it.valid; ++k) {
      const Item nx = item_of(p, cta, G, k + 1);
      const int qpos = it.off + it.q0 + row;         // absolute position of this query
      float m_ref = -INFINITY, l_sum = 0.f;
      for (int t = 0; t < it.nkt; ++t) {
        const int Jt = J + t;
        const uint32_t sb = tmem + lane_off + kColS + (Jt & 1) * 128;
        // post-projection RMSNorm: this half's 64 key scales (lane l loads keys
        // 2l, 2l+1; every row of the tile shares them), fetched before the wait
        float ks0 = 1.f, ks1 = 1.f;
        if (KS) {
          const int kb = t * kBK + half * 64 + 2 * lane;
          const float* kp = p.key_scale + (static_cast<size_t>(it.b) * p.H + it.h) * p.max_len;
          if (kb < p.max_len) ks0 = __ldg(kp + kb);
          if (kb + 1 < p.max_len) ks1 = __ldg(kp + kb + 1);
        }
        ok = ok && pwait(&bar_sf[Jt & 1], static_cast<uint32_t>(Jt >> 1) & 1u, fail);
        tc_fence_after();
        uint32_t v[64];
        tmem_ld64_wait(sb + half * 64, v);
        if (KS) {
#pragma unroll
          for (int e = 0; e < 64; e += 2) {
            v[e] = __float_as_uint(__uint_as_float(v[e]) * __shfl_sync(0xffffffffu, ks0, e >> 1));
            v[e + 1] = __float_as_uint(__uint_as_float(v[e + 1]) * __shfl_sync(0xffffffffu, ks1, e >> 1));
          }
        }
        // keys t*128 + half*64 + c are visible iff c <= lim (causal and length)
        const int lim = min(qpos, it.L - 1) - t * kBK - half * 64;
        if (lim < 63) {
#pragma unroll
          for (int e = 0; e < 64; ++e)
            if (e > lim) v[e] = __float_as_uint(-INFINITY);
        }
        float mx = -INFINITY;
#pragma unroll
        for (int e = 0; e < 64; e += 2) mx = fmax3(mx, __uint_as_float(v[e]), __uint_as_float(v[e + 1]));
        xchg[half][row] = mx;
        named_bar(1 + quad, 64);
        mx = fmaxf(mx, xchg[half ^ 1][row]);
        named_bar(1 + quad, 64);                       // both read before either writes again
        const float mloc = mx * sc;                    // scale > 0
        const bool need = t > 0 && mloc > m_ref + 8.f;
        if (t == 0) m_ref = mloc;
        if (__any_sync(0xffffffffu, need)) {
          // rare: rescale this half's share of the row's accumulators (O_s and
          // O_z, 96 of the 192 columns) once the previous P V is done
          const float alpha = need ? ex2_approx(m_ref - mloc) : 1.f;
          ok = ok && pwait(&bar_pv, static_cast<uint32_t>(Jt - 1) & 1u, fail);
          tc_fence_after();
          for (int c = half * 3; c < half * 3 + 3; ++c) {
            const uint32_t col = c < 4 ? kColOs + c * 32 : kColOz + (c - 4) * 32;
            uint32_t o[32];
            tmem_ld32_wait(tmem + lane_off + col, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
            tmem_st32(tmem + lane_off + col, o);
          }
          tmem_wait_st();
          l_sum *= alpha;
          if (need) m_ref = mloc;
        }
        // probabilities against m_ref, bf16 pairs written over this half's
        // share of the S buffer's first 64 columns
        const float nm = -m_ref;
        uint32_t pk[32];
        float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
        for (int e = 0; e < 64; e += 2) {
          const float p0 = ex2_approx(fmaf(__uint_as_float(v[e]), sc, nm));
          const float p1 = ex2_approx(fmaf(__uint_as_float(v[e + 1]), sc, nm));
          ls0 += p0;
          ls1 += p1;
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(p0, p1);
          pk[e / 2] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        l_sum += ls0 + ls1;
        tmem_st32(sb + half * 32, pk);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_cta(&bar_pf[Jt & 1]);
      }
      xchg[half][row] = l_sum;
      named_bar(1 + quad, 64);
      l_sum += xchg[half ^ 1][row];
      named_bar(1 + quad, 64);
      const int Jl = J + it.nkt - 1;
      // ---- O_z -> bf16 in shared memory for the lift (each half 32 columns) ----
      ok = ok && pwait(&bar_all, static_cast<uint32_t>(k) & 1u, fail);
      tc_fence_after();
      {
        uint32_t v[32];
        tmem_ld32_wait(tmem + lane_off + kColOz + half * 32, v);
        unsigned char* obase = smem + kOffK + (Jl & 1) * kKStage + 16384;
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          const __nv_bfloat162 v2 = __floats2bfloat162_rn(__uint_as_float(v[e]), __uint_as_float(v[e + 1]));
          *reinterpret_cast<__nv_bfloat162*>(obase + sw128(row, half * 32 + e)) = v2;
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive_cta(&bar_ozs);  // bf16(O_z) ready
      }
      // the next item's Pq parts while this item's lift runs
      if (nx.valid) split_pq(k + 1);
      ok = ok && pwait(&bar_lift, static_cast<uint32_t>(k) & 1u, fail);
      tc_fence_after();
      // o = O_s / l: read this half's 64 columns, free O for the next item's
      // first P V, then store from registers (rows past q_len are skipped)
      uint32_t v[64];
      tmem_ld64_wait(tmem + lane_off + kColOs + half * 64, v);
      tc_fence_before();
      mbar_arrive_cta(&bar_ofree);
      const int tq = it.q0 + row;
      if (ok && !*fail && tq < p.Tq) {
        const float inv_l = 1.f / l_sum;
        float* dst = p.out + ((static_cast<size_t>(it.b) * p.Tq + tq) * p.H + it.h) * kDH + half * 64;
        if (p.out_v8) {
#pragma unroll
          for (int e = 0; e < 64; e += 8) {
            float o[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) o[u] = __uint_as_float(v[e + u]) * inv_l;
            st_global_v8(dst + e, o);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 64; e += 4)
            *reinterpret_cast<float4*>(dst + e) =
                make_float4(__uint_as_float(v[e]) * inv_l, __uint_as_float(v[e + 1]) * inv_l,
                            __uint_as_float(v[e + 2]) * inv_l, __uint_as_float(v[e + 3]) * inv_l);
        }
        if (half == 0 && p.lse)
          p.lse[(static_cast<size_t>(it.b) * p.H + it.h) * p.Tq + tq] = (m_ref + log2f(l_sum)) * kPfLn2;
      }
      J += it.nkt;
      it = nx;
    }
    if (!ok) *fail = 1;
  }
  tc_fence_before();
  __syncthreads();
  if (threadIdx.x == 0 && *fail) atomicOr(p.status, 1u);
  if (warp == 0) tmem_dealloc(tmem, 512);
}

}  // namespace lrkv

namespace {

bool a16p(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

// bf16 tensor map of rank n (dims innermost first; strides in bytes of dims
// 1..n-1), 128-byte swizzle.
bool make_map(CUtensorMap* m, const void* base, int n, const uint64_t* dims, const uint64_t* strides,
              const uint32_t* box, CUtensorMapDataType ty = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16) {
  auto fn = encoder();
  if (!fn) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < n; ++i) { d[i] = dims[i]; bx[i] = box[i]; es[i] = 1; }
  for (int i = 0; i < n - 1; ++i) s[i] = strides[i];
  return fn(m, ty, n, const_cast<void*>(base), d, s, bx, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// Host checks of the prefill shape (no pointers): LRKV_OK when the kernel
// implements it.
static lrkv_status check_prefill_dims(const lrkv_dims* dims, int q_len) {
  if (!dims) return LRKV_ERR_INVALID_ARG;
  const lrkv_dims& d = *dims;
  if (d.batch < 1 || d.heads < 1 || d.head_dim < 1 || d.rank < 0 || d.max_len < 1 || q_len < 1)
    return LRKV_ERR_INVALID_ARG;
  if (d.dtype != LRKV_BF16 && d.dtype != LRKV_F32) return LRKV_ERR_INVALID_ARG;
  if (!(d.scale == d.scale)) return LRKV_ERR_INVALID_ARG;
  if (d.dtype != LRKV_BF16 || d.head_dim != 128 || d.rank != 64) return LRKV_ERR_UNSUPPORTED;
  if (q_len > d.max_len || d.heads > 65535 || d.batch > 65535) return LRKV_ERR_UNSUPPORTED;
  return LRKV_OK;
}

// The prefill's workspace: the device status word (the kernel needs no other
// scratch memory).
constexpr size_t kPrefillWorkspaceBytes = 16;

extern "C" lrkv_status lrkv_prefill_workspace_size(const lrkv_dims* dims, int q_len, size_t* bytes) {
  if (!bytes) return LRKV_ERR_INVALID_ARG;
  const lrkv_status st = check_prefill_dims(dims, q_len);
  if (st != LRKV_OK) return st;
  *bytes = kPrefillWorkspaceBytes;
  return LRKV_OK;
}

static lrkv_status prefill_impl(const lrkv_dims* dims, int q_len, const void* q, const void* k_s,
                                const void* v_s, const void* z_k, const void* z_v, const void* b_k,
                                const void* b_v, const float* key_scale, const int32_t* seq_lens, float* out,
                                float* lse, void* ws, size_t ws_bytes, lrkv_stream_t stream,
                                const int32_t* block_table = nullptr, int page_size = 0, int num_pages = 0) {
  const lrkv_status cst = check_prefill_dims(dims, q_len);
  if (cst != LRKV_OK) return cst;
  const lrkv_dims& d = *dims;
  if (!q || !k_s || !v_s || !z_k || !z_v || !b_k || !b_v || !seq_lens || !out) return LRKV_ERR_INVALID_ARG;
  if (!a16p(q) || !a16p(k_s) || !a16p(v_s) || !a16p(z_k) || !a16p(z_v) || !a16p(b_k) || !a16p(b_v) || !a16p(out))
    return LRKV_ERR_INVALID_ARG;
  if (!ws || ws_bytes < kPrefillWorkspaceBytes) return LRKV_ERR_WORKSPACE;
  if (!a16p(ws)) return LRKV_ERR_INVALID_ARG;

  const int B = d.batch, H = d.heads, Lm = d.max_len;
  const uint64_t dh = 128, r = 64;
  // tensor-map extents of the cache: (rows, sequences), or (page_size, pages) for a paged cache
  const uint64_t rows = static_cast<uint64_t>(block_table ? page_size : Lm);
  const uint64_t seqs = static_cast<uint64_t>(block_table ? num_pages : B);
  lrkv::PrefillMaps maps;
  std::memset(&maps, 0, sizeof(maps));
  {
    // q [B][Tq][H][128] seen as {64 columns, Tq, 2 halves, H, B}: one box of
    // 128 rows x both halves lands as [half][row][64]
    const uint64_t dm[5] = {64, static_cast<uint64_t>(q_len), 2, static_cast<uint64_t>(H), static_cast<uint64_t>(B)};
    const uint64_t st[4] = {H * dh * 2, 128, dh * 2, static_cast<uint64_t>(q_len) * H * dh * 2};
    const uint32_t bx[5] = {64, 128, 2, 1, 1};
    if (!make_map(&maps.q, q, 5, dm, st, bx)) return LRKV_ERR_CUDA;
  }
  {
    // k_s, v_s [B][max_len][128] seen as {64 columns, max_len, 2 halves, B}
    // (paged: [pages][page_size][128] as {64, page_size, 2, pages})
    const uint64_t dm[4] = {64, rows, 2, seqs};
    const uint64_t st[3] = {dh * 2, 128, rows * dh * 2};
    const uint32_t bx[4] = {64, 128, 2, 1};
    if (!make_map(&maps.ks, k_s, 4, dm, st, bx) || !make_map(&maps.vs, v_s, 4, dm, st, bx)) return LRKV_ERR_CUDA;
  }
  {
    const uint64_t dm[4] = {r, static_cast<uint64_t>(H), rows, seqs};
    const uint64_t st[3] = {r * 2, H * r * 2, rows * H * r * 2};
    const uint32_t bx[4] = {64, 1, 128, 1};
    if (!make_map(&maps.zk, z_k, 4, dm, st, bx) || !make_map(&maps.zv, z_v, 4, dm, st, bx)) return LRKV_ERR_CUDA;
  }
  {
    const uint64_t dm[3] = {r, dh, static_cast<uint64_t>(H)};
    const uint64_t st[2] = {r * 2, dh * r * 2};
    const uint32_t bx[3] = {64, 128, 1};
    if (!make_map(&maps.bk, b_k, 3, dm, st, bx) || !make_map(&maps.bv, b_v, 3, dm, st, bx)) return LRKV_ERR_CUDA;
  }
  lrkv::PrefillParams p;
  p.B = B; p.H = H; p.Tq = q_len; p.max_len = Lm;

  const float scale = d.scale > 0.f ? d.scale : 1.f / std::sqrt(static_cast<float>(d.head_dim));
  p.scale_log2 = scale * lrkv::kPfLog2e;
  p.seq_lens = seq_lens; p.out = out; p.lse = lse;
  p.key_scale = key_scale;
  p.block_table = block_table;
  p.max_blocks = block_table ? Lm / page_size : 0;
  p.page_shift = 0;
  while (block_table && (1 << p.page_shift) < page_size) ++p.page_shift;
  p.num_pages = num_pages;
  auto kern = key_scale ? lrkv::lrkv_prefill_kernel<true> : lrkv::lrkv_prefill_kernel<false>;
  p.out_v8 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
  p.status = static_cast<uint32_t*>(ws);

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(ws, 0, 4, s) != cudaSuccess) return LRKV_ERR_CUDA;
  if (lrkv::ensure_kernel_smem(reinterpret_cast<const void*>(kern), lrkv::kSmem) != cudaSuccess)
    return LRKV_ERR_CUDA;
  // persistent: one CTA per SM (the kernel deals the (sequence, head, query
  // tile) items out itself)
  const int nsm = lrkv::device_sm_count();
  if (nsm < 1) return LRKV_ERR_CUDA;
  const long long items = static_cast<long long>((q_len + lrkv::kBQ - 1) / lrkv::kBQ) * H * B;
  if (items > (1ll << 30)) return LRKV_ERR_UNSUPPORTED;
  const int grid = static_cast<int>(std::min<long long>(nsm, items));
  kern<<<grid, lrkv::kThreads, lrkv::kSmem, s>>>(p, maps);
  return cudaGetLastError() == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

extern "C" lrkv_status lrkv_prefill(const lrkv_dims* dims, int q_len, const void* q, const void* k_s,
                                    const void* v_s, const void* z_k, const void* z_v, const void* b_k,
                                    const void* b_v, const int32_t* seq_lens, float* out, float* lse, void* ws,
                                    size_t ws_bytes, lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_prefill");
  return prefill_impl(dims, q_len, q, k_s, v_s, z_k, z_v, b_k, b_v, nullptr, seq_lens, out, lse, ws, ws_bytes,
                      stream);
}

extern "C" lrkv_status lrkv_prefill_normed(const lrkv_dims* dims, int q_len, const void* q, const void* k_s,
                                           const void* v_s, const void* z_k, const void* z_v, const void* b_k,
                                           const void* b_v, const float* key_scale, const int32_t* seq_lens,
                                           float* out, float* lse, void* ws, size_t ws_bytes,
                                           lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_prefill_normed");
  if (!key_scale) return LRKV_ERR_INVALID_ARG;
  return prefill_impl(dims, q_len, q, k_s, v_s, z_k, z_v, b_k, b_v, key_scale, seq_lens, out, lse, ws, ws_bytes,
                      stream);
}

extern "C" lrkv_status lrkv_prefill_paged(const lrkv_dims* dims, int q_len, const void* q, int page_size,
                                          int num_pages, const int32_t* block_table, const void* k_s,
                                          const void* v_s, const void* z_k, const void* z_v, const void* b_k,
                                          const void* b_v, const int32_t* seq_lens, float* out, float* lse,
                                          void* ws, size_t ws_bytes, lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_prefill_paged");
  if (!dims || !block_table) return LRKV_ERR_INVALID_ARG;
  if (page_size < 128 || (page_size & (page_size - 1)) != 0 || num_pages < 1) return LRKV_ERR_INVALID_ARG;
  if (dims->max_len % page_size != 0) return LRKV_ERR_INVALID_ARG;
  if (static_cast<long long>(num_pages) * page_size > (1LL << 31) - 1) return LRKV_ERR_UNSUPPORTED;
  return prefill_impl(dims, q_len, q, k_s, v_s, z_k, z_v, b_k, b_v, nullptr, seq_lens, out, lse, ws, ws_bytes,
                      stream, block_table, page_size, num_pages);
}
