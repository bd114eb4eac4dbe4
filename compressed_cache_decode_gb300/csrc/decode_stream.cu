// decode_stream.cu — the bf16 split-KV scan on the tensor cores.
//
// Grid (range CTAs, row tiles): CTA (c, m) owns a range of the concatenated
// histories (see decode.cu) and the 16 heads of row tile m.  16-token tiles
// stream through a ring of shared-memory stages, four tensor copies per tile:
// the shared rows k_s and v_s as 128-byte-swizzled boxes, and this row tile's
// latents z_k, z_v as one box of [segment][token][segment row] where a
// segment holds the latents of `hs` heads and each segment row is padded to
// an odd number of 16-byte chunks (the box is 8 elements wider than the
// segment; TMA fills the excess with zeros), so that ldmatrix over 8 token
// rows is free of bank conflicts.
//
// The 8 warps form 4 pairs: pair p takes every 4th tile of the CTA's range
// (tile i in stage i % stages), each warp of the pair 8 of the 16 heads, and
// the second warp of the pair to finish a stage refills it with the tile
// `stages` ahead.  Per tile and warp, FlashAttention-2 style, the products on
// the tensor cores (bf16 mma.sync, fp32 accumulation):
//   * scores, transposed (tokens are the M dimension):
//       S^T = K_s q^T + Z_k P_bd, where P_bd is block diagonal: column h
//       holds p_h = q_h B_h^K on the rows of head h's latents.  p_h is split
//       into bf16 hi + lo parts, so the private score keeps ~16 bits of p.
//   * ONE online softmax per head over the summed scores ("Low-Rank Key
//     Value Attention | What a shared cache can preserve", §3, fused
//     online-softmax paragraph), with a lazily raised reference maximum.
//   * the probabilities are transposed in registers (movmatrix) into the B
//     operand of the transposed value products
//       O_s^T += V_s^T P^T      (shared values: rows of the head dim)
//       O_z^T += Z_v^T P^T      (private values: the half's latent rows; only
//                                the entries on a head's own rows are kept).
// At the end of each (sequence, range) piece every pair writes its state
// (m, l, O_s, O_z of its heads) as one partial; the merge kernel (decode.cu)
// merges the pairs' and the pieces' partials.  The first launch phase (lengths,
// first copies, absorb of p, set-up) runs code the SM has not fetched yet;
// the last warp runs the tile code once on no tokens meanwhile, so that the
// tiles find it in the instruction cache.
#include <cmath>
#include <algorithm>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <type_traits>
#include <utility>

#include <cuda.h>

#include "decode_common.cuh"
#include "decode_plan.h"
#include "ptx.cuh"
#include "tmap.h"

namespace lrkv {

using namespace dec;

namespace {

constexpr int kT = 16;                       // tokens per tile
constexpr int kWarps = kStreamConsumers;     // token streams per CTA
constexpr int kThreadsS = 32 * kWarps;
constexpr int kPairs = kWarps / 2;           // a tile is shared by a pair (8 heads each)
constexpr float kRescaleLog2 = 8.f;          // raise the reference max only past 2^8
constexpr int kCursorOff = 640;              // shared bytes of the pairs' tile cursors (2 per pair)
constexpr int kQLastOff = 896;               // [2] last piece whose q went into each p/q buffer
constexpr int kHeaderBytes = 1024;           // barriers, stage records, step offsets, cursors
constexpr int kKsBoxT = 20;                  // tokens per staged key-scale row (16 from a row 4-aligned below)

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&v);
}

__device__ __forceinline__ void named_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Arrive at named barrier `id` (of `nthreads` threads) without waiting.
__device__ __forceinline__ void named_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Pieces of this CTA's token range: (sequence b, rows [t_lo, t_end)), in
// tiles of kT rows from row t_beg.  For a paged cache the first piece's tiles
// start on the 16-row grid of the sequence (t_beg = t_lo rounded down; the
// rows before t_lo, the previous CTA's, are masked), so that no tile spans
// two pages; otherwise t_beg = t_lo.  Later pieces start at row 0.
struct Piece {
  int b, t_beg, t_end, ntiles, t_lo;
};

__device__ __forceinline__ bool piece_first(Piece& p, const int* pre, int B, int g0, int g1, bool align) {
  TileWalk w;
  if (!walk_first(w, pre, B, g0, g1)) return false;
  p.b = w.b; p.t_lo = w.t0; p.t_end = w.t_end;
  p.t_beg = align ? (w.t0 & ~(kT - 1)) : w.t0;
  p.ntiles = (p.t_end - p.t_beg + kT - 1) / kT;
  return true;
}

__device__ __forceinline__ bool piece_next(Piece& p, const int* pre, int B, int g1) {
  int b = p.b + 1;
  while (b < B && pre[b] < g1 && pre[b + 1] == pre[b]) ++b;
  if (b >= B || pre[b] >= g1) return false;
  p.b = b; p.t_beg = 0; p.t_lo = 0; p.t_end = min(pre[b + 1], g1) - pre[b];
  p.ntiles = (p.t_end + kT - 1) / kT;
  return true;
}

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

// The copies of tile (sequence b, rows t0..t0+15) into stage s (one thread).
// Tensor-map coordinates (sequence or page, row) of logical row t of
// sequence b; false when the block table names no page of the pool (the copy
// then reads the fill value, zeros, and the caller records the bound).
__device__ __forceinline__ bool cache_coords(const DecodePlan& P, int b, int t, int& seq, int& row) {
  if (!P.block_table) {
    seq = b;
    row = t;
    return true;
  }
  seq = __ldg(P.block_table + static_cast<size_t>(b) * P.max_blocks + (t >> P.page_shift));
  row = t & ((1 << P.page_shift) - 1);
  return seq >= 0 && seq < P.num_pages;
}

__device__ __forceinline__ bool stream_issue(const DecodePlan& P, const CUtensorMap* tk, const CUtensorMap* tv,
                                             const CUtensorMap* tzk, const CUtensorMap* tzv, const CUtensorMap* tks,
                                             unsigned char* smem, uint64_t* full, int s, int b_log, int t_log,
                                             int zseg0, int m0, const int* pre) {
  // In a decode step the launch before writes each sequence's newest row
  // (row L_b - 1): only a copy of the tile that holds it waits for that
  // launch; every other tile streams at once.
  if (P.after_append && t_log + kT >= pre[b_log + 1] - pre[b_log]) pdl_wait();
  int b, t0;  // a 16-token tile never spans two pages (page_size is a multiple of 16)
  const bool in_pool = cache_coords(P, b_log, t_log, b, t0);
  unsigned char* ks = smem + P.off_kv + static_cast<size_t>(s) * P.stage_bytes;
  unsigned char* vs = ks + P.kv_bytes;
  unsigned char* zk = vs + P.kv_bytes;
  unsigned char* zv = zk + P.zt_bytes;
  mbar_arrive_expect_tx(&full[s], 2u * P.nbox * kT * 128u + 2u * static_cast<uint32_t>(P.zt_bytes) +
                                       (P.ks_tma ? static_cast<uint32_t>(P.ks_bytes) : 0u));
  // the key scales of the tile's 16 logical rows (from the row rounded down
  // to a multiple of 4, the copy's alignment) and the row tile's 16 heads
  if (P.ks_tma) tma_load_3d(ks + P.off_ks, tks, t_log & ~3, m0, b_log, &full[s]);
  for (int cb = 0; cb < P.nbox; ++cb) {
    tma_load_3d(ks + cb * kT * 128, tk, cb * 64, t0, b, &full[s]);
    tma_load_3d(vs + cb * kT * 128, tv, cb * 64, t0, b, &full[s]);
  }
  if (P.r > 0) {
    tma_load_4d(zk, tzk, 0, t0, zseg0, b, &full[s]);
    tma_load_4d(zv, tzv, 0, t0, zseg0, b, &full[s]);
  }
  return in_pool;
}

// q (bf16) of the row tile's heads of sequence b into p/q buffer `buf`
// (one thread).
__device__ __forceinline__ void q_issue(const DecodePlan& P, unsigned char* smem, uint64_t* pbar, int buf, int b,
                                        int m0, int piece) {
  // the last piece whose q went into buffer `buf` (drained before exit)
  reinterpret_cast<volatile int*>(smem + kQLastOff)[buf] = piece;
  const uint32_t qbytes = static_cast<uint32_t>(min(16, P.H - m0) * P.dh * 2);
  unsigned char* dst = smem + P.off_pq + buf * P.pq_bytes;
  mbar_arrive_expect_tx(&pbar[buf], qbytes);
  tma_load_1d(dst, static_cast<const unsigned char*>(P.q) + (static_cast<size_t>(b) * P.H + m0) * P.dh * 2, qbytes,
              &pbar[buf]);
}

// Absorbed query p_h = q_h B_h^K ("Low-Rank Key Value Attention | What a
// shared cache can preserve", §3, Algorithm 2 step 02) of the row tile's 16
// heads, for one or two sequences at once (their q rows in shared memory),
// in fp32.  Thread role: head hl, columns 4 cg .. 4 cg + 3, head-dim part dp
// of bk_dsplit; B^K is read with 8-byte loads, kBkChunk of them in flight,
// the first chunk issued early by bk_load (before the tile copies, so that
// it does not queue behind them).
constexpr int kBkChunk = 32;

struct BkRole {
  int hl, cg, dp, nd;
  bool on;
};

__device__ __forceinline__ BkRole bk_role(const DecodePlan& P, int m0, int tid) {
  BkRole R;
  const int per_head = (P.r / 4) * P.bk_dsplit;
  R.hl = tid / max(per_head, 1);
  const int rem = tid - R.hl * per_head;
  R.cg = rem / P.bk_dsplit;
  R.dp = rem % P.bk_dsplit;
  R.nd = P.dh / P.bk_dsplit;
  R.on = P.r > 0 && R.hl < 16 && m0 + R.hl < P.H;
  return R;
}

// Head-dim rows d = i bk_dsplit + dp (i = d0 .. d0 + kBkChunk - 1) of this
// thread's B^K columns.
__device__ __forceinline__ void bk_load(const DecodePlan& P, int m0, const BkRole& R, int d0, uint2 (&v)[kBkChunk]) {
  const __nv_bfloat16* base = static_cast<const __nv_bfloat16*>(P.b_k) +
                              (static_cast<size_t>(m0 + R.hl) * P.dh + R.dp) * P.r + 4 * R.cg;
  const size_t step = static_cast<size_t>(P.bk_dsplit) * P.r;
#pragma unroll
  for (int u = 0; u < kBkChunk; ++u)
    v[u] = (R.on && d0 + u < R.nd) ? *reinterpret_cast<const uint2*>(base + (d0 + u) * step) : make_uint2(0u, 0u);
}

// p[hl][4 cg .. 4 cg + 3] into the private-score table: entry hl r/2 + c/2
// holds {hi(p[c]), hi(p[c+1])}, {lo(p[c]), lo(p[c+1])} (bf16 high parts and
// the bf16 of what they leave), the same 8 bytes per column pair as the fp32
// row would take: one 16-byte store of two entries.
__device__ __forceinline__ void store_p_entries(float* prow, const float (&a)[4]) {
  float h[4];
#pragma unroll
  for (int u = 0; u < 4; ++u) h[u] = __bfloat162float(__float2bfloat16_rn(a[u]));
  *reinterpret_cast<uint4*>(prow) = make_uint4(pack_bf16(h[0], h[1]), pack_bf16(a[0] - h[0], a[1] - h[1]),
                                               pack_bf16(h[2], h[3]), pack_bf16(a[2] - h[2], a[3] - h[3]));
}

// The same from a shared-memory copy of the row tile's B^K: head hl's
// [dh][r] bf16 block at hl * bk_head_bytes, head-dim rows d = i bk_dsplit + dp.
__device__ __forceinline__ void absorb_rows_smem(const DecodePlan& P, const BkRole& R,
                                                 const unsigned char* bks, const __nv_bfloat16* qa,
                                                 const __nv_bfloat16* qb, float* pa, float* pb) {
  float aa[4] = {0.f, 0.f, 0.f, 0.f}, ab[4] = {0.f, 0.f, 0.f, 0.f};
  if (R.on) {
    const __nv_bfloat16* bk =
        reinterpret_cast<const __nv_bfloat16*>(bks + R.hl * P.bk_head_bytes) + R.dp * P.r + 4 * R.cg;
    const __nv_bfloat16* xa = qa + R.hl * P.dh + R.dp;
    const __nv_bfloat16* xb = qb ? qb + R.hl * P.dh + R.dp : nullptr;
    const int step = P.bk_dsplit * P.r, qstep = P.bk_dsplit;
#pragma unroll 4
    for (int i = 0; i < R.nd; ++i) {  // runs once per launch: a short unroll keeps loads in flight
      const uint2 v = *reinterpret_cast<const uint2*>(bk + i * step);
      const float b0 = bf_lo(v.x), b1 = bf_hi(v.x), b2 = bf_lo(v.y), b3 = bf_hi(v.y);
      const float x = __bfloat162float(xa[i * qstep]);
      aa[0] = fmaf(x, b0, aa[0]); aa[1] = fmaf(x, b1, aa[1]); aa[2] = fmaf(x, b2, aa[2]); aa[3] = fmaf(x, b3, aa[3]);
      if (xb) {
        const float y = __bfloat162float(xb[i * qstep]);
        ab[0] = fmaf(y, b0, ab[0]); ab[1] = fmaf(y, b1, ab[1]); ab[2] = fmaf(y, b2, ab[2]); ab[3] = fmaf(y, b3, ab[3]);
      }
    }
  }
  for (int o = 1; o < P.bk_dsplit; o <<= 1)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      aa[u] += __shfl_xor_sync(0xffffffffu, aa[u], o);
      ab[u] += __shfl_xor_sync(0xffffffffu, ab[u], o);
    }
  // heads past H get zero entries
  if (R.hl < 16 && R.dp == 0) {
    store_p_entries(pa + R.hl * P.r + 4 * R.cg, aa);
    if (pb) store_p_entries(pb + R.hl * P.r + 4 * R.cg, ab);
  }
}

// p rows of up to two sequences (q rows qa, qb: [16][dh] bf16; p rows pa, pb:
// [16][r] private-score table entries); v holds the first chunk of B^K already.
__device__ __forceinline__ void absorb_rows(const DecodePlan& P, int m0, const BkRole& R, uint2 (&v)[kBkChunk],
                                            const __nv_bfloat16* qa, const __nv_bfloat16* qb, float* pa, float* pb) {
  float aa[4] = {0.f, 0.f, 0.f, 0.f}, ab[4] = {0.f, 0.f, 0.f, 0.f};
  for (int d0 = 0; d0 < R.nd; d0 += kBkChunk) {
    if (d0 > 0) bk_load(P, m0, R, d0, v);
#pragma unroll
    for (int u = 0; u < kBkChunk; ++u) {
      if (d0 + u < R.nd) {
        const int d = (d0 + u) * P.bk_dsplit + R.dp;
        const float b0 = bf_lo(v[u].x), b1 = bf_hi(v[u].x), b2 = bf_lo(v[u].y), b3 = bf_hi(v[u].y);
        if (R.on) {
          const float x = __bfloat162float(qa[R.hl * P.dh + d]);
          aa[0] = fmaf(x, b0, aa[0]); aa[1] = fmaf(x, b1, aa[1]); aa[2] = fmaf(x, b2, aa[2]); aa[3] = fmaf(x, b3, aa[3]);
          if (qb) {
            const float y = __bfloat162float(qb[R.hl * P.dh + d]);
            ab[0] = fmaf(y, b0, ab[0]); ab[1] = fmaf(y, b1, ab[1]); ab[2] = fmaf(y, b2, ab[2]); ab[3] = fmaf(y, b3, ab[3]);
          }
        }
      }
    }
  }
  // sum the head-dim parts (lanes dp of one (head, column group) are adjacent)
  for (int o = 1; o < P.bk_dsplit; o <<= 1)
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      aa[u] += __shfl_xor_sync(0xffffffffu, aa[u], o);
      ab[u] += __shfl_xor_sync(0xffffffffu, ab[u], o);
    }
  // heads past H get zero entries
  if (R.hl < 16 && R.dp == 0) {
    store_p_entries(pa + R.hl * P.r + 4 * R.cg, aa);
    if (pb) store_p_entries(pb + R.hl * P.r + 4 * R.cg, ab);
  }
}

__device__ __forceinline__ void prefetch_tmap(const void* p) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(p) : "memory");
}

// Stage s holds tile issued[s]; a consumer waits for its tile to be issued
// before it waits on the stage's barrier, so the parity it waits for always
// names the barrier's current phase (a waiter two phases ahead would take
// the completed phase two back for its own).  Bounded like the barrier wait.
__device__ __forceinline__ bool wait_issued(const int* issued, int want, long long limit) {
  const volatile int* p = issued;
  if (*p >= want) return true;
  const long long t0 = clock64();
  while (*p < want) {
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

// L2 prefetch of the cache rows [r0, r1) of sequence b: the shared rows and
// the latent rows of all heads (each contiguous in memory), by bulk copies
// with no destination, so that HBM streams ahead of the shared-memory ring.
__device__ __forceinline__ void l2_prefetch_rows(const DecodePlan& P, int b, int r0, int r1) {
  const uint32_t kv = static_cast<uint32_t>(P.dh) * 2u, zr = static_cast<uint32_t>(P.H * P.r) * 2u;
  while (r0 < r1) {
    // rows of one page at a time (all rows at once for a contiguous cache)
    const int r_end = P.block_table ? min(r1, ((r0 >> P.page_shift) + 1) << P.page_shift) : r1;
    int sq, rw;
    if (cache_coords(P, b, r0, sq, rw)) {
      const size_t row0 = static_cast<size_t>(sq) * P.map_len + rw;
      const uint32_t n = static_cast<uint32_t>(r_end - r0);
      l2_prefetch_bulk(static_cast<const unsigned char*>(P.k_s) + row0 * kv, n * kv);
      l2_prefetch_bulk(static_cast<const unsigned char*>(P.v_s) + row0 * kv, n * kv);
      if (zr) {
        l2_prefetch_bulk(static_cast<const unsigned char*>(P.z_k) + row0 * zr, n * zr);
        l2_prefetch_bulk(static_cast<const unsigned char*>(P.z_v) + row0 * zr, n * zr);
      }
    }
    r0 = r_end;
  }
}

// L2 prefetch of the tiles [t0, t1) of a CTA's range in tile order, in
// chunks of up to kPrefetchChunk tiles of one piece (one thread).
constexpr int kPrefetchChunk = 4;
__device__ __forceinline__ void l2_prefetch_tiles(const DecodePlan& P, const int* pre, int B, int g0, int g1,
                                                  int t0, int t1) {
  TileCursor cur;
  cur.more = piece_first(cur.pc, pre, B, g0, g1, P.block_table != nullptr);
  cur.ibase = 0;
  int j = t0;
  while (j < t1 && cur.seek(j, pre, B, g1)) {
    const int e = min(min(t1, j + kPrefetchChunk), cur.ibase + cur.pc.ntiles);
    const int r0 = cur.pc.t_beg + (j - cur.ibase) * kT;
    l2_prefetch_rows(P, cur.pc.b, r0, min(cur.pc.t_end, cur.pc.t_beg + (e - cur.ibase) * kT));
    j = e;
  }
}

}  // namespace

// EXACT: the launch's latent step count equals MZMAX (its loops need no
// per-step guard); otherwise at most MZMAX steps, guarded at run time.
template <int DHT, int MZMAX, bool EXACT>
__global__ void __launch_bounds__(kThreadsS, 1)
    lrkv_decode_stream_kernel(const __grid_constant__ DecodePlan P, const __grid_constant__ CUtensorMap tm_k,
                              const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_zk,
                              const __grid_constant__ CUtensorMap tm_zv, const __grid_constant__ CUtensorMap tm_ks) {
  constexpr int MZA = MZMAX > 0 ? MZMAX : 1;
  constexpr int BS = MZA > 16 ? 2 : 4;       // private-score steps per load batch
  constexpr int BZ = MZA > 16 ? 4 : 8;       // private-value steps per load batch
  constexpr int KB = DHT > 4 ? 4 : DHT;      // head-dim steps per load batch of the shared rows
  const int kst = EXACT ? MZA : P.kst;       // latent steps per warp (a constant when EXACT)
  // Private values by head group (EXACT: r = 2 MZMAX): a group is GH heads
  // whose latents start on a 16-byte boundary (one head when r is a multiple
  // of 8, else two); accumulator tile s holds the group's latent columns
  // 16 s .. 16 s + 15 (column h = head hb + h), each group's product taking
  // the probabilities of its own heads' columns only.  Entry (s, row, h) is
  // latent 16 s + row - (h % GH) r of head h, or no latent (never written).
  // Otherwise one tile per 16-column step of the half's 8 r latents, of
  // which the diagonal blocks are kept.
  constexpr bool PH = EXACT && MZMAX > 0;
  constexpr int GH = (2 * MZMAX) % 8 == 0 ? 1 : 2;          // heads per value group
  constexpr int NZH = PH ? (GH * 2 * MZMAX + 15) / 16 : 1;  // tiles per group
  constexpr int NZV = PH ? NZH : MZA;                       // private value accumulator tiles
  extern __shared__ __align__(16) unsigned char smem_raw[];
  __shared__ int s_timeout;
  __shared__ int s_nopage;  // a block table entry named no page of the pool
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);

  // the merge kernel may launch now: it waits for this grid before it reads
  // (its few CTAs take the SMs this grid leaves free)
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int pair = warp >> 1, hf = warp & 1;     // tile stream, half of the row tile's heads
  const int g = lane >> 2, q4 = lane & 3;
  const int arow = lane & 15, ahalf = lane >> 4;            // ldmatrix rows for the score A operand
  const int trow = (lane & 7) + 8 * (lane >> 4), tcol = (lane >> 3) & 1;  // ... for transposed A
  const int B = P.B, H = P.H, dh = P.dh, r = P.r;
  const int m0 = blockIdx.y * 16;                 // first head of the row tile
  const int zseg0 = blockIdx.y * P.nsb;           // its first latent segment

  uint64_t* full = reinterpret_cast<uint64_t*>(smem);
  int* issued = reinterpret_cast<int*>(smem + 128);   // [16] tile in each stage
  int* cons = reinterpret_cast<int*>(smem + 192);     // [16] warps done with each stage
  uint64_t* pbar = reinterpret_cast<uint64_t*>(smem + 256);  // [2] p/q buffers
  int* zo = reinterpret_cast<int*>(smem + 320);       // [2][32] latent step offsets
  int* zhead = reinterpret_cast<int*>(smem + 576);    // [16] shared byte offset of each head's latents
  int* pre = reinterpret_cast<int*>(smem + P.off_prefix);
  uint2* qf = reinterpret_cast<uint2*>(smem + P.off_pf);    // shared-score B fragments (q)

  // ---- 1. barriers, sequence starts (clamped lengths) ----------------------
  // the first lengths are read before anything else (their latency is the
  // start of the chain to the first tile)
  const int len0 = tid < B ? P.seq_lens[tid] : 0;
  // without the shared-memory B^K: the first chunk of this thread's B^K
  // columns is loaded now, its latency hidden behind the set-up below
  const BkRole bkr = bk_role(P, m0, tid);
  uint2 bkv[kBkChunk];
  if (P.bk_stages == 0) bk_load(P, m0, bkr, 0, bkv);
  {
    // one read per 64-byte line of the launch plan, all at once, so that the
    // later dependent reads of its fields hit the constant cache
    constexpr int kPlanLines = (static_cast<int>(sizeof(DecodePlan)) + 63) / 64;
    if (tid >= 32 && tid < 32 + kPlanLines) {
      const int v = reinterpret_cast<const int*>(&P)[(tid - 32) * 16];
      if (v == 0x7f7f7f7f && tid == 0) s_timeout = v;  // never true: keeps the read
    }
  }
  // barriers and records set up by several threads at once (one thread
  // doing all of it delayed the whole block by ~1.3K cycles)
  if (tid == 0) {
    // with bk_stages > 0 the row tile's B^K lands in the last bk_stages ring
    // stages (one bulk copy, issued first: it depends on nothing) and those
    // stages get their tiles once the first two pieces are absorbed
    uint64_t* bkb = reinterpret_cast<uint64_t*>(smem + 272);
    mbar_init(bkb, 1);
    fence_barrier_init();
    if (P.bk_stages > 0) {
      const uint32_t bytes = static_cast<uint32_t>(min(16, H - m0) * dh * r * 2);
      mbar_arrive_expect_tx(bkb, bytes);
      tma_load_1d(smem + P.off_kv + static_cast<size_t>(P.stages - P.bk_stages) * P.stage_bytes,
                  static_cast<const __nv_bfloat16*>(P.b_k) + static_cast<size_t>(m0) * dh * r, bytes, bkb);
    }
  } else if (tid == 1) {
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_v);
  } else if (tid == 2) {
    if (r > 0) {
      prefetch_tmap(&tm_zk);
      prefetch_tmap(&tm_zv);
    }
    if (P.ks_tma) prefetch_tmap(&tm_ks);
  } else if (tid == 3) {
    s_timeout = 0;
    s_nopage = 0;
    reinterpret_cast<int*>(smem + kQLastOff)[0] = -1;
    reinterpret_cast<int*>(smem + kQLastOff)[1] = -1;
    mbar_init(&pbar[0], 1);
    mbar_init(&pbar[1], 1);
    fence_barrier_init();
  } else if (tid >= 96 && tid < 96 + P.stages) {
    const int s = tid - 96;
    mbar_init(&full[s], 1);
    issued[s] = -1;
    cons[s] = 0;
    fence_barrier_init();
  }
  if (tid < 64) zo[tid] = P.zo[tid >> 5][tid & 31];
  if (PH && tid < 16) zhead[tid] = (tid / P.hs) * kT * P.segp * 2 + (tid % P.hs) * r * 2;
  int bad = 0;
  for (int b = tid; b < B; b += blockDim.x) {
    int L = b == tid ? len0 : P.seq_lens[b];
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
    // the launch before may still read the workspace: wait before writing it
    pdl_wait();
    if (blockIdx.x == 0 && blockIdx.y == 0) {
      for (int b = tid; b <= B; b += blockDim.x) P.prefix[b] = pre[b];
      if (tid == 0) { P.meta[0] = N; P.meta[1] = G; }
    }
    if (tid == 0) {
      // the B^K copy must land before the block's shared memory is released
      const bool drained = P.bk_stages == 0 || mbar_wait_bounded(reinterpret_cast<uint64_t*>(smem + 272), 0u);
      *cta_status = (bad ? kDevBounds : 0u) | (drained ? 0u : kDevTimeout);
    }
    return;
  }
  const int c = blockIdx.x;
  int g0, g1;
  if (static_cast<unsigned long long>(N) * G < (1ull << 32)) {  // 32-bit division when it fits
    g0 = static_cast<int>(static_cast<unsigned>(c) * static_cast<unsigned>(N) / static_cast<unsigned>(G));
    g1 = static_cast<int>(static_cast<unsigned>(c + 1) * static_cast<unsigned>(N) / static_cast<unsigned>(G));
  } else {
    g0 = static_cast<int>(static_cast<long long>(c) * N / G);
    g1 = static_cast<int>(static_cast<long long>(c + 1) * N / G);
  }
  // ---- 2. q of the first two pieces, then the first `stages` tiles (warp w
  // issues tiles w, w + 8, ...), so that the small copies land first ---------
  Piece pc;
  bool more = piece_first(pc, pre, B, g0, g1, P.block_table != nullptr);
  Piece pc1 = pc;
  const bool two = piece_next(pc1, pre, B, g1);
  uint64_t* bkbar = reinterpret_cast<uint64_t*>(smem + 272);  // the B^K copy (issued at entry)
  const int first_burst = P.stages - P.bk_stages;
  // The last warp, when it has no absorb role (warm: see below), issues the
  // q copies and the first burst of tiles, one tile per lane, so that the
  // absorbing warps wait only for q (a tile's four copies take a lane ~1.5K
  // cycles to issue), and after its warm-up pass the tiles of the stages
  // that held B^K; otherwise lane 0 of warp w issues tiles w, w + 8, ... and
  // thread 0 the q copies, and the absorbing warps the later stages' tiles.
  const bool warm = warp == kWarps - 1 && warp >= P.bk_warps;
  const bool lone = P.bk_warps < kWarps;  // there is such a warp
  const bool issuer = !lone || warm;
  if (issuer && (lone ? lane >= 30 : tid < 2)) {
    const int qi = lone ? 31 - lane : tid;
    if (qi == 0) q_issue(P, smem, pbar, 0, pc.b, m0, 0);
    else if (two) q_issue(P, smem, pbar, 1, pc1.b, m0, 1);
  }
  if (issuer && (lone ? lane < first_burst : lane == 0)) {
    TileCursor cur;
    cur.pc = pc;
    cur.more = more;
    cur.ibase = 0;
    for (int j = lone ? lane : warp; j < first_burst && cur.seek(j, pre, B, g1); j += lone ? 32 : kWarps) {
      if (!stream_issue(P, &tm_k, &tm_v, &tm_zk, &tm_zv, &tm_ks, smem, full, j, cur.pc.b,
                        cur.pc.t_beg + (j - cur.ibase) * kT, zseg0, m0, pre))
        *reinterpret_cast<volatile int*>(&s_nopage) = 1;
      *reinterpret_cast<volatile int*>(&issued[j]) = j;
    }
  }
  float acc_v[DHT][4] = {};      // O_s^T: rows d = 16 m + g (+8), columns heads 2 q4 + e
  float acc_z[NZV][4] = {};      // O_z^T: rows latent column 16 m + g (+8) of this half (PH: of each head)
  float mc[2] = {-INFINITY, -INFINITY}, lc[2] = {0.f, 0.f};  // reference max, denominator
  const int zrow = P.segp * 2;  // bytes per segment row
  const int hb = 8 * hf;        // first head (row-tile local) of this half
  const uint2* qfl = qf + hf * DHT * 32 + lane;   // this lane's q fragments
  const unsigned char* pqcur = smem + P.off_pq;  // the current piece's q / p buffer
  // steps kk whose latent column 16 kk + 2 q4 (bit of vmask0), or that
  // column + 8 (vmask1), belongs to this lane's head g within the half
  // (head g's columns are g r .. g r + r - 1; unrolled and without a
  // division: this runs once per launch, on the way to the first tile)
  uint32_t vmask0 = 0u, vmask1 = 0u;
  {
    const int rr = (EXACT && MZMAX > 0) ? 2 * MZMAX : r;
    const int lo = g * rr, hi = lo + rr;
#pragma unroll
    for (int kk = 0; kk < MZA; ++kk) {
      if (kk < kst) {
        const int j = 16 * kk + 2 * q4;
        vmask0 |= (j >= lo && j < hi ? 1u : 0u) << kk;
        vmask1 |= (j + 8 >= lo && j + 8 < hi ? 1u : 0u) << kk;
      }
    }
  }

  // The last warp, when it has no absorb role, first runs one tile of the
  // scan's code on no tokens (nvalid 0: every score is masked, no value row
  // kept, no stage consumed) while the other warps absorb, so that the tile
  // code is in the SM's instruction cache when the first tiles arrive.
  bool ok = true;
  if (MZMAX > 0 && !warm) {
    // p of the first two pieces, from their q rows and B^K
    ok = mbar_wait_bounded(&pbar[0], 0u, P.wait_limit) && (!two || mbar_wait_bounded(&pbar[1], 0u, P.wait_limit));
    unsigned char* pq0 = smem + P.off_pq;
    unsigned char* pq1 = pq0 + P.pq_bytes;
    const __nv_bfloat16* qa = reinterpret_cast<const __nv_bfloat16*>(pq0);
    const __nv_bfloat16* qb2 = two ? reinterpret_cast<const __nv_bfloat16*>(pq1) : nullptr;
    float* pa = reinterpret_cast<float*>(pq0 + 16 * dh * 2);
    float* pb = two ? reinterpret_cast<float*>(pq1 + 16 * dh * 2) : nullptr;
    if (P.bk_stages > 0) {
      const bool bk_in = ok && mbar_wait_bounded(bkbar, 0u, P.wait_limit);  // drained before exit in any case
      ok = ok && bk_in;
      absorb_rows_smem(P, bkr, smem + P.off_kv + static_cast<size_t>(first_burst) * P.stage_bytes, qa, qb2, pa,
                       pb);
    } else {
      absorb_rows(P, m0, bkr, bkv, qa, qb2, pa, pb);
    }
    if (!ok) *reinterpret_cast<volatile int*>(&s_timeout) = 1;
  }
  if (P.bk_stages > 0 && warp < P.bk_warps && lone) {
    // B^K is consumed (by the warps that absorb): the warm-up warp gives the
    // last stages their tiles
    fence_proxy_async_smem();
    named_arrive(2, 32 * (P.bk_warps + 1));
  } else if (P.bk_stages > 0 && warp < P.bk_warps) {
    // B^K is consumed (by the warps that absorb): the last stages get their tiles
    fence_proxy_async_smem();
    named_sync(2, 32 * P.bk_warps);
    if (lane == 0 && ok) {
      TileCursor cur;
      cur.pc = pc;
      cur.more = more;
      cur.ibase = 0;
      for (int j = first_burst + warp; j < P.stages && cur.seek(j, pre, B, g1); j += P.bk_warps) {
        if (!stream_issue(P, &tm_k, &tm_v, &tm_zk, &tm_zv, &tm_ks, smem, full, j, cur.pc.b,
                          cur.pc.t_beg + (j - cur.ibase) * kT, zseg0, m0, pre))
          *reinterpret_cast<volatile int*>(&s_nopage) = 1;
        *reinterpret_cast<volatile int*>(&issued[j]) = j;
      }
    }
  }
  // with an L2 prefetch window (a tuning option, off by default): the tiles
  // after the ring's start streaming into L2, issued by thread 0 once it has
  // absorbed and released B^K (the ring's copies are queued by then, and the
  // warm-up warp, which issues them, is not held up)
  if (tid == 0 && P.pfw > 0) l2_prefetch_tiles(P, pre, B, g0, g1, P.stages, P.stages + P.pfw);
  // this pair's next tile (tiles pair, pair + 4, ... across the pieces), its
  // ring stage and that stage's phase parity, advanced without a division
  int inext = pair, snext = pair % P.stages;
  uint32_t pnext = static_cast<uint32_t>(pair / P.stages) & 1u;
  // ldmatrix row addresses within the shared rows' 128-byte-swizzled boxes
  // for head-dim steps n with n & 3 = m (step n is in box n >> 2): chunk
  // 2 m + (lane half) of row arow (scores) or trow (transposed values),
  // XORed with the row's low bits
  int koff[4], voff[4];
#pragma unroll
  for (int m = 0; m < 4; ++m) {
    koff[m] = arow * 128 + (((2 * m + ahalf) ^ (arow & 7)) << 4);
    voff[m] = trow * 128 + (((2 * m + tcol) ^ (trow & 7)) << 4);
  }
  int ibase = 0;      // tile index of the piece's first tile
  int kp = warm ? -1 : 0;  // piece counter (p/q buffer kp & 1); -1: the warm-up pass
  // this pair's cursors over its tiles to issue (tile + stages) and to
  // prefetch into L2, kept in shared memory (used once per tile, by lane 0
  // of whichever warp of the pair refills; the stage counters' atomics order
  // the two warps' turns)
  TileCursor* pcur = reinterpret_cast<TileCursor*>(smem + kCursorOff) + 2 * pair;
  if (hf == 0 && lane == 0) {
    TileCursor c0;
    c0.more = piece_first(c0.pc, pre, B, g0, g1, P.block_table != nullptr);
    c0.ibase = 0;
    pcur[0] = c0;
    pcur[1] = c0;
  }
  while (more) {
    const bool dry = kp < 0;
    if (!dry) {
    // ---- piece set-up: p and q of the row tile --------------------------------
    // The first piece's set-up is built by the warps other than the warm-up
    // warp (which may still be in its pass); they signal it on barrier 3.
    const bool split = kp == 0 && P.bk_warps < kWarps;
    const int nset = split ? kThreadsS - 32 : kThreadsS;  // threads that build the set-up
    if (!(split && warm))
      named_sync(1, nset);  // the p rows are written; the previous piece is done with the buffers
    const int buf = kp & 1;
    // (only while this warp has seen every earlier copy into that buffer land:
    // a second copy must never join a phase that is still pending)
    if (tid == 0 && kp >= 1 && ok && !*reinterpret_cast<volatile int*>(&s_timeout)) {
      Piece nx = pc;
      if (piece_next(nx, pre, B, g1)) {  // prefetch the next piece's q (pieces 0, 1 came first)
        fence_proxy_async_smem();
        q_issue(P, smem, pbar, buf ^ 1, nx.b, m0, kp + 1);
      }
    }
    if (ok && *reinterpret_cast<volatile int*>(&s_timeout)) ok = false;  // another warp gave up: stop waiting
    if (ok) {
      ok = mbar_wait_bounded(&pbar[buf], static_cast<uint32_t>(kp >> 1) & 1u, P.wait_limit);
      if (!ok) *reinterpret_cast<volatile int*>(&s_timeout) = 1;
    }
    unsigned char* pqb = smem + P.off_pq + buf * P.pq_bytes;
    pqcur = pqb;
    const int nh = min(16, H - m0);
    if (MZMAX > 0 && kp >= 2) {  // p of a third or later piece (the first two came before)
      uint2 v[kBkChunk];
      bk_load(P, m0, bkr, 0, v);
      absorb_rows(P, m0, bkr, v, reinterpret_cast<const __nv_bfloat16*>(pqb), nullptr,
                  reinterpret_cast<float*>(pqb + 16 * dh * 2), nullptr);
      named_sync(1, kThreadsS);  // p rows ready
    }
    mc[0] = mc[1] = -INFINITY;
    lc[0] = lc[1] = 0.f;
#pragma unroll
    for (int n = 0; n < DHT; ++n)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc_v[n][k] = 0.f;
#pragma unroll
    for (int n = 0; n < NZV; ++n)
#pragma unroll
      for (int k = 0; k < 4; ++k) acc_z[n][k] = 0.f;
    {
      // q as the B operand of the shared scores: entry (h2, kk, L) holds
      // q[hl][k, k+1] and q[hl][k+8, k+9] of head hl = 8 h2 + (L >> 2),
      // k = 16 kk + 2 (L & 3), zero past H: one conflict-free 8-byte load
      // per step and lane in the tile loop
      const __nv_bfloat16* qsm = reinterpret_cast<const __nv_bfloat16*>(pqb);
      const int nq = 2 * DHT * 32;
      for (int e = tid; e < (tid < nset ? nq : 0); e += nset) {
        const int L = e & 31, kk = (e >> 5) % DHT, h2 = (e >> 5) / DHT;
        const int hl = 8 * h2 + (L >> 2), k = 16 * kk + 2 * (L & 3);
        uint2 v = make_uint2(0u, 0u);
        if (hl < nh) {
          v.x = *reinterpret_cast<const uint32_t*>(qsm + hl * dh + k);
          v.y = *reinterpret_cast<const uint32_t*>(qsm + hl * dh + k + 8);
        }
        qf[e] = v;
      }
    }
    if (!split) {
      named_sync(1, kThreadsS);  // fragments ready
    } else if (!warm) {
      named_sync(1, nset);       // fragments ready (the builders)
      named_arrive(3, kThreadsS);
    } else {
      named_sync(3, kThreadsS);  // fragments ready (the warm-up warp)
    }
    }

    // ---- this pair's tiles of the piece ----------------------------------------
    // rows of the piece's sequence: a tile reaching past them may hold
    // unwritten rows (any bits, NaN included)
    const int seq_rows = pre[pc.b + 1] - pre[pc.b];
    while (inext < ibase + pc.ntiles) {
      const int i = inext, s = snext;
      const uint32_t par = pnext;
      const int t0 = pc.t_beg + (i - ibase) * kT;
      const int nvalid = dry ? 0 : min(kT, pc.t_end - t0);
      const int lo = max(0, pc.t_lo - t0);  // rows [lo, nvalid) of the tile are this CTA's
      if (ok && !dry && *reinterpret_cast<volatile int*>(&s_timeout)) ok = false;  // stop waiting
      if (ok && !dry) {
        ok = wait_issued(&issued[s], i, P.wait_limit) &&
             mbar_wait_bounded(&full[s], par, P.wait_limit);
        if (!ok) *reinterpret_cast<volatile int*>(&s_timeout) = 1;
      }
      if (ok && !*reinterpret_cast<volatile int*>(&s_timeout)) {
        unsigned char* ks = smem + P.off_kv + static_cast<size_t>(s) * P.stage_bytes;
        unsigned char* vs = ks + P.kv_bytes;
        unsigned char* zk = vs + P.kv_bytes;
        unsigned char* zv = zk + P.zt_bytes;
        // token masks of the value operands: rows past the history (unwritten
        // cache rows) must not meet their zero probabilities as 0 x NaN
        auto mine = [&](int row) { return row >= lo && row < nvalid; };
        const uint32_t keep0 = (mine(2 * q4) ? 0x0000ffffu : 0u) | (mine(2 * q4 + 1) ? 0xffff0000u : 0u);
        const uint32_t keep1 = (mine(2 * q4 + 8) ? 0x0000ffffu : 0u) | (mine(2 * q4 + 9) ? 0xffff0000u : 0u);

        // post-projection RMSNorm: the joint reciprocal scale of each key
        // (token g / g+8, head hb + 2 q4 + e) multiplies its summed score;
        // loaded now, used after the score MMAs
        float ksc[4] = {1.f, 1.f, 1.f, 1.f};
        if (P.ks_tma) {
          // from the stage: [16 heads][kKsBoxT rows from t0 & ~3] (rows and
          // heads past the extents read as zeros, their scores are masked)
          const float* kss = reinterpret_cast<const float*>(ks + P.off_ks) + (hb + 2 * q4) * kKsBoxT + (t0 & 3) + g;
          ksc[0] = kss[0];
          ksc[1] = kss[kKsBoxT];
          ksc[2] = kss[8];
          ksc[3] = kss[kKsBoxT + 8];
        } else if (P.key_scale) {
          const int hl = m0 + hb + 2 * q4;
          const float* kp = P.key_scale + (static_cast<size_t>(pc.b) * H + hl) * P.max_len + t0;
          if (g < nvalid) {
            if (hl < H) ksc[0] = __ldg(kp + g);
            if (hl + 1 < H) ksc[1] = __ldg(kp + P.max_len + g);
          }
          if (g + 8 < nvalid) {
            if (hl < H) ksc[2] = __ldg(kp + g + 8);
            if (hl + 1 < H) ksc[3] = __ldg(kp + P.max_len + g + 8);
          }
        }
        // scores S^T (rows = tokens g / g+8, columns = heads hb + 2 q4 + e),
        // four independent accumulation chains
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        float la[4] = {0.f, 0.f, 0.f, 0.f}, lb[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k0 = 0; k0 < DHT; k0 += KB) {  // batches of KB head-dim steps (fewer live registers)
          uint32_t a[KB][4];
          uint2 qv[KB];
#pragma unroll
          for (int u = 0; u < KB; ++u) {
            ldsm_x4(a[u][0], a[u][1], a[u][2], a[u][3], ks + ((k0 + u) >> 2) * (kT * 128) + koff[(k0 + u) & 3]);
            qv[u] = qfl[(k0 + u) * 32];
          }
#pragma unroll
          for (int u = 0; u < KB; ++u)
            mma_bf16_16816(((k0 + u) & 1) ? sb : sa, a[u][0], a[u][1], a[u][2], a[u][3], qv[u].x, qv[u].y);
        }
        if (MZMAX > 0) {
          // B fragment of step kk (latent columns j = 16 kk + 2 q4 (+1, +8,
          // +9) of this half; column g = head hb + g): the pairs 8 kk + q4 and
          // 8 kk + q4 + 4 of the half's p table, kept where their head is g
          // (bit kk of vmask0 / vmask1) and zero elsewhere (block diagonal)
          const unsigned char* z0 = zk + arow * zrow + ahalf * 16;
          const int* zoh = zo + 32 * hf;
          const uint2* pt = reinterpret_cast<const uint2*>(pqcur + 16 * dh * 2) + 4 * hf * r + q4;
          // (6 batches unrolled with the per-group values: measured faster than none
          // or all of them, which runs out of registers)
#pragma unroll (PH ? 6 : 1)
          for (int kk = 0; kk < kst; kk += BS) {  // batches of BS steps (kst is even)
            uint32_t a[BS][4];
            uint2 f0[BS], f1[BS];
#pragma unroll
            for (int u = 0; u < BS; ++u)
              if (kk + u < kst) {
                ldsm_x4(a[u][0], a[u][1], a[u][2], a[u][3], z0 + zoh[kk + u]);
                f0[u] = pt[8 * (kk + u)];
                f1[u] = pt[8 * (kk + u) + 4];
              }
#pragma unroll
            for (int u = 0; u < BS; ++u)
              if (kk + u < kst) {
                const bool k0v = (vmask0 >> (kk + u)) & 1u, k1v = (vmask1 >> (kk + u)) & 1u;
                const uint32_t h0 = k0v ? f0[u].x : 0u, l0 = k0v ? f0[u].y : 0u;
                const uint32_t h1 = k1v ? f1[u].x : 0u, l1 = k1v ? f1[u].y : 0u;
                mma_bf16_16816((u & 1) ? sb : sa, a[u][0], a[u][1], a[u][2], a[u][3], h0, h1);
                mma_bf16_16816((u & 1) ? lb : la, a[u][0], a[u][1], a[u][2], a[u][3], l0, l1);
              }
          }
        }

        // scale, mask rows past the piece's end, tile max per head
        const bool v0 = mine(g), v1 = mine(g + 8);
        float sc[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float t = ((sa[u] + sb[u]) + (la[u] + lb[u])) * P.scale_log2 * ksc[u];
          sc[u] = (u < 2 ? v0 : v1) ? t : -INFINITY;
        }
        float mx[2] = {fmaxf(sc[0], sc[2]), fmaxf(sc[1], sc[3])};
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
          mx[0] = fmaxf(mx[0], __shfl_xor_sync(0xffffffffu, mx[0], o));
          mx[1] = fmaxf(mx[1], __shfl_xor_sync(0xffffffffu, mx[1], o));
        }
        const bool up = mx[0] > mc[0] + kRescaleLog2 || mx[1] > mc[1] + kRescaleLog2;
        if (__any_sync(0xffffffffu, up)) {
          // raise the reference max of the heads that outgrew it; rescale the
          // accumulator columns of those heads (held by this lane)
          float al[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float mn = mx[e] > mc[e] + kRescaleLog2 ? mx[e] : mc[e];
            al[e] = mc[e] == -INFINITY ? 0.f : exp2f(mc[e] - mn);
            mc[e] = mn;
            lc[e] *= al[e];
          }
#pragma unroll
          for (int n = 0; n < DHT; ++n) {
            acc_v[n][0] *= al[0]; acc_v[n][1] *= al[1]; acc_v[n][2] *= al[0]; acc_v[n][3] *= al[1];
          }
#pragma unroll
          for (int n = 0; n < NZV; ++n) {
            acc_z[n][0] *= al[0]; acc_z[n][1] *= al[1]; acc_z[n][2] *= al[0]; acc_z[n][3] *= al[1];
          }
        }
        const float p0 = exp2f(sc[0] - mc[0]), p1 = exp2f(sc[1] - mc[1]);
        const float p2 = exp2f(sc[2] - mc[0]), p3 = exp2f(sc[3] - mc[1]);
        lc[0] += p0 + p2;
        lc[1] += p1 + p3;
        // P^T (tokens x heads) as the B operand: transpose the 8x8 blocks so
        // that lane (g, q4) holds head g at tokens 2 q4, 2 q4 + 1 (and + 8)
        const uint32_t pb0 = movmatrix_trans(pack_bf16(p0, p1));  // tokens 0-7
        const uint32_t pb1 = movmatrix_trans(pack_bf16(p2, p3));  // tokens 8-15

        // Values.  The A operands of tokens outside [lo, nvalid) meet zero
        // probabilities; only a tile reaching past the sequence's rows may
        // hold non-finite bits there (unwritten rows), where 0 x NaN must not
        // reach the sums: that tile (and the warm-up pass) zeroes those
        // tokens' operand halves, every other tile runs unmasked.
        auto values = [&](auto masked) {
          constexpr bool M = decltype(masked)::value;
          const uint32_t k0 = M ? keep0 : 0xffffffffu, k1 = M ? keep1 : 0xffffffffu;
          // shared values: O_s^T += V_s^T P^T (rows = head dim)
#pragma unroll
          for (int n0 = 0; n0 < DHT; n0 += KB) {
            uint32_t a[KB][4];
#pragma unroll
            for (int u = 0; u < KB; ++u)
              ldsm_x4_trans(a[u][0], a[u][1], a[u][2], a[u][3], vs + ((n0 + u) >> 2) * (kT * 128) + voff[(n0 + u) & 3]);
#pragma unroll
            for (int u = 0; u < KB; ++u) {
              if (M)
                mma_bf16_16816(acc_v[n0 + u], a[u][0] & k0, a[u][1] & k0, a[u][2] & k1, a[u][3] & k1, pb0, pb1);
              else
                mma_bf16_16816(acc_v[n0 + u], a[u][0], a[u][1], a[u][2], a[u][3], pb0, pb1);
            }
          }
          // private values, per head group: O_z,grp^T += Z_v,grp^T P^T with
          // P^T kept in the group's columns only (this lane's column g)
          if (PH) {
            const unsigned char* zvb = zv + trow * zrow + tcol * 16;
#pragma unroll
            for (int h = 0; h < 8; h += GH) {
              const bool own = g / GH == h / GH;
              const uint32_t b0 = own ? pb0 : 0u, b1 = own ? pb1 : 0u;
              const unsigned char* zb = zvb + zhead[hb + h];
              uint32_t a[NZH][4];
#pragma unroll
              for (int u = 0; u < NZH; ++u) ldsm_x4_trans(a[u][0], a[u][1], a[u][2], a[u][3], zb + 32 * u);
#pragma unroll
              for (int u = 0; u < NZH; ++u) {
                if (M)
                  mma_bf16_16816(acc_z[u], a[u][0] & k0, a[u][1] & k0, a[u][2] & k1, a[u][3] & k1, b0, b1);
                else
                  mma_bf16_16816(acc_z[u], a[u][0], a[u][1], a[u][2], a[u][3], b0, b1);
              }
            }
          } else if (MZMAX > 0) {
            // private values: O_z^T += Z_v^T P^T over this half's latent columns
            const unsigned char* z0 = zv + trow * zrow + tcol * 16;
            const int* zoh = zo + 32 * hf;
#pragma unroll
            for (int n0 = 0; n0 < MZA; n0 += BZ) {  // batches of BZ steps
              uint32_t a[BZ][4];
#pragma unroll
              for (int u = 0; u < BZ; ++u)
                if (n0 + u < kst) ldsm_x4_trans(a[u][0], a[u][1], a[u][2], a[u][3], z0 + zoh[n0 + u]);
#pragma unroll
              for (int u = 0; u < BZ; ++u)
                if (n0 + u < kst) {
                  if (M)
                    mma_bf16_16816(acc_z[(n0 + u) % NZV], a[u][0] & k0, a[u][1] & k0, a[u][2] & k1, a[u][3] & k1,
                                   pb0, pb1);
                  else
                    mma_bf16_16816(acc_z[(n0 + u) % NZV], a[u][0], a[u][1], a[u][2], a[u][3], pb0, pb1);
                }
            }
          }
        };
        if (dry || t0 + kT > seq_rows)
          values(std::true_type{});
        else
          values(std::false_type{});
      }
      if (dry) break;
      // done with the stage: the second warp of the pair refills it with
      // tile i + stages
      const int j = i + P.stages;
      fence_proxy_async_smem();  // this warp's generic accesses before the async writes
      __syncwarp();
      if (lane == 0) {
        __threadfence_block();  // this warp's cursor writes before its count (release)
        const bool second = (atomicAdd(&cons[s], 1) & 1) != 0;
        __threadfence_block();  // the other warp's cursor writes after its count (acquire)
        if (second) {
          TileCursor rc = pcur[0];
          if (rc.seek(j, pre, B, g1)) {
            fence_proxy_async_smem();
            if (ok && !*reinterpret_cast<volatile int*>(&s_timeout)) {
              if (!stream_issue(P, &tm_k, &tm_v, &tm_zk, &tm_zv, &tm_ks, smem, full, s, rc.pc.b,
                                rc.pc.t_beg + (j - rc.ibase) * kT, zseg0, m0, pre))
                *reinterpret_cast<volatile int*>(&s_nopage) = 1;
              *reinterpret_cast<volatile int*>(&issued[s]) = j;
            }
            // keep the L2 prefetch window pfw tiles ahead of the ring
            const int jp = j + P.pfw;
            if (ok && P.pfw > 0) {
              TileCursor pfc = pcur[1];
              if (pfc.seek(jp, pre, B, g1)) {
                const int rr = pfc.pc.t_beg + (jp - pfc.ibase) * kT;
                l2_prefetch_rows(P, pfc.pc.b, rr, min(pfc.pc.t_end, rr + kT));
              }
              pcur[1] = pfc;
            }
          }
          pcur[0] = rc;
        }
      }
      __syncwarp();
      inext += kPairs;
      snext += kPairs;
      while (snext >= P.stages) {
        snext -= P.stages;
        pnext ^= 1u;
      }
    }

    if (dry) {  // warm-up pass done: the real first piece
      if (P.bk_stages > 0) {
        // the stages that held B^K get their tiles once the absorbing warps
        // are done with it (one tile per lane)
        named_sync(2, 32 * (P.bk_warps + 1));
        if (lane < P.bk_stages && ok && !*reinterpret_cast<volatile int*>(&s_timeout)) {
          TileCursor cur;
          cur.pc = pc;
          cur.more = true;
          cur.ibase = 0;
          const int j = first_burst + lane;
          if (cur.seek(j, pre, B, g1)) {
            if (!stream_issue(P, &tm_k, &tm_v, &tm_zk, &tm_zv, &tm_ks, smem, full, j, cur.pc.b,
                              cur.pc.t_beg + (j - cur.ibase) * kT, zseg0, m0, pre))
              *reinterpret_cast<volatile int*>(&s_nopage) = 1;
            *reinterpret_cast<volatile int*>(&issued[j]) = j;
          }
        }
      }
      kp = 0;
      continue;
    }
    // ---- end of the piece: full denominators ------------------------------------
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      lc[0] += __shfl_xor_sync(0xffffffffu, lc[0], o);
      lc[1] += __shfl_xor_sync(0xffffffffu, lc[1], o);
    }

    // ---- this pair's state is one partial of the piece: (m, l) per head and
    // the unnormalised O_s and O_z rows, written straight from the
    // accumulators; the combine kernel merges the pairs' partials
    if (kp == 0) {
      // first write to the workspace: the launch before may still read it
      pdl_wait();
      if (blockIdx.x == 0 && blockIdx.y == 0) {
        for (int b = tid; b <= B; b += blockDim.x) P.prefix[b] = pre[b];
        if (tid == 0) { P.meta[0] = N; P.meta[1] = G; }
      }
    }
    {
      const size_t slot = static_cast<size_t>(pc.b + c) * kPairs + pair;
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int hl = hb + 2 * q4 + e, h = m0 + hl;
        if (h < H) {
          if (g == 0) {
            float* pml = P.part_ml + (slot * H + h) * 2;
            pml[0] = mc[e];
            pml[1] = lc[e];
          }
          float* o = P.part_acc + (slot * H + h) * (dh + r);
#pragma unroll
          for (int n = 0; n < DHT; ++n) {
            o[16 * n + g] = acc_v[n][e];
            o[16 * n + g + 8] = acc_v[n][2 + e];
          }
          if (PH) {
            // tile n, row g (+8) holds latent 16 n + g (+8) - (hl % GH) r of head hl
            const int c0 = ((hl - hb) % GH) * r;
#pragma unroll
            for (int n = 0; n < NZH; ++n) {
              const int ca = 16 * n + g - c0, cb = ca + 8;
              if (ca >= 0 && ca < r) o[dh + ca] = acc_z[n][e];
              if (cb >= 0 && cb < r) o[dh + cb] = acc_z[n][2 + e];
            }
          } else if (MZMAX > 0) {
            // row j (this half) holds latent column j - (hl - hb) r of head hl
#pragma unroll
            for (int n = 0; n < MZA; ++n) {
              if (n < kst) {
                const int ca = 16 * n + g - (hl - hb) * r, cb = ca + 8;
                if (ca >= 0 && ca < r) o[dh + ca] = acc_z[n % NZV][e];
                if (cb >= 0 && cb < r) o[dh + cb] = acc_z[n % NZV][2 + e];
              }
            }
          }
        }
      }
    }
    ibase += pc.ntiles;
    ++kp;
    more = piece_next(pc, pre, B, g1);
  }
  if (!ok) *reinterpret_cast<volatile int*>(&s_timeout) = 1;
  named_sync(1, kThreadsS);
  if (tid == 0) {
    // Before the CTA exits, every copy it issued must have landed: a wait
    // that gave up skipped its stage, so wait (at the full bound) for the
    // last tile issued into each stage, the last q copy of each buffer and
    // the B^K copy.
    bool drained = true;
    for (int st = 0; st < P.stages; ++st) {
      const int j = *reinterpret_cast<volatile int*>(&issued[st]);
      if (j >= 0) drained = mbar_wait_bounded(&full[st], static_cast<uint32_t>(j / P.stages) & 1u) && drained;
    }
    for (int bq = 0; bq < 2; ++bq) {
      const int k = reinterpret_cast<volatile int*>(smem + kQLastOff)[bq];
      if (k >= 0) drained = mbar_wait_bounded(&pbar[bq], static_cast<uint32_t>(k >> 1) & 1u) && drained;
    }
    if (P.bk_stages > 0) drained = mbar_wait_bounded(bkbar, 0u) && drained;
    if (!drained) *reinterpret_cast<volatile int*>(&s_timeout) = 1;
    *cta_status = (bad || *reinterpret_cast<volatile int*>(&s_nopage) ? kDevBounds : 0u) |
                  (*reinterpret_cast<volatile int*>(&s_timeout) ? kDevTimeout : 0u);
  }
}

// ======================================================================= host
namespace {

using StreamFn = void (*)(const DecodePlan, const CUtensorMap, const CUtensorMap, const CUtensorMap,
                          const CUtensorMap, const CUtensorMap);

// The latent steps a warp keeps accumulators for: exactly kst for the ranks
// 28, 32, 48, 56 and 64 (loops without guards, accumulators sized exactly:
// no register spills), else the smallest of 16 and 32 that holds kst.
template <int DHT>
StreamFn pick_mz(const DecodePlan& P) {
  if (P.r == 0) return lrkv_decode_stream_kernel<DHT, 0, false>;
  switch (P.kst) {
    case 14: return lrkv_decode_stream_kernel<DHT, 14, true>;
    case 16: return lrkv_decode_stream_kernel<DHT, 16, true>;
    case 24: return lrkv_decode_stream_kernel<DHT, 24, true>;
    case 28: return lrkv_decode_stream_kernel<DHT, 28, true>;
    case 32: return lrkv_decode_stream_kernel<DHT, 32, true>;
    default:
      return P.kst < 16 ? lrkv_decode_stream_kernel<DHT, 16, false> : lrkv_decode_stream_kernel<DHT, 32, false>;
  }
}

StreamFn stream_fn(const DecodePlan& P) {
  switch (P.dh / 16) {
    case 4: return pick_mz<4>(P);
    case 8: return pick_mz<8>(P);
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
  if (r % 4 != 0 || r > 64) return LRKV_ERR_UNSUPPORTED;
  P.stream = 1;
  P.T = kT;
  P.Hp = round_up(H, 16);
  P.mt = P.Hp / 16;
  P.grid = std::max(1, P.grid / P.mt);
  P.ngw = kPairs;  // one partial per warp pair and piece
  P.nthreads = kThreadsS;
  P.span = 128;
  P.box_cols = 64;
  P.nbox = dh / 64;
  P.kv_bytes = round_up(kT * dh * 2, 1024);
  if (r > 0) {
    // latent segment: hs heads (a power of two dividing H) whose hs r
    // latents are a multiple of 16 elements and fit a box with 8 spare
    P.hs = 0;
    for (int hs = 16; hs >= 1; hs >>= 1)
      if (H % hs == 0 && (hs * r) % 16 == 0 && hs * r + 8 <= 256) { P.hs = hs; break; }
    if (P.hs == 0) return LRKV_ERR_UNSUPPORTED;
    P.segw = P.hs * r;
    P.segp = P.segw + 8;  // (segw / 8) is even, so segp / 8 is odd
    P.nsb = 16 / P.hs;
    P.zt_bytes = P.nsb * kT * P.segp * 2;
    P.kst = r / 2;  // 16-wide steps over the 8 r latents of 8 heads
    if (P.kst > 32) return LRKV_ERR_UNSUPPORTED;
    // shared offset of step n of half h2: latent column j = 8 h2 r + 16 n
    for (int h2 = 0; h2 < 2; ++h2)
      for (int n = 0; n < 32; ++n) {
        const int j = 8 * h2 * r + 16 * std::min(n, P.kst - 1);
        P.zo[h2][n] = (j / P.segw) * kT * P.segp * 2 + (j % P.segw) * 2;
      }
  } else {
    P.hs = 1; P.segw = 0; P.segp = 0; P.nsb = 0; P.zt_bytes = 0; P.kst = 0;
    for (int h2 = 0; h2 < 2; ++h2)
      for (int n = 0; n < 32; ++n) P.zo[h2][n] = 0;
  }
  P.pq_bytes = round_up(16 * dh * 2 + 16 * r * 4, 128);
  // absorb roles: 16 heads x r/4 column groups x bk_dsplit head-dim parts
  P.bk_dsplit = 1;
  while (r > 0 && 16 * (r / 4) * P.bk_dsplit * 2 <= kThreadsS && P.bk_dsplit * 2 <= dh / 4) P.bk_dsplit *= 2;
  P.bk_warps = r > 0 ? (16 * (r / 4) * P.bk_dsplit + 31) / 32 : 1;
  P.stage_bytes = round_up(2 * P.kv_bytes + 2 * P.zt_bytes, 1024);
  // the key-scale slot (post-projection RMSNorm decode) when the stages
  // still fit as many of it (set below)
  P.off_ks = 2 * P.kv_bytes + 2 * P.zt_bytes;  // 256-byte aligned
  P.ks_bytes = 0;
  P.ks_tma = 0;
  const int pf_bytes = 2 * (dh / 16) * 32 * 8;  // q fragments of both halves

  // shared memory: barriers | prefix | p/q buffers | q fragments | ring
  auto layout = [&](int stages) {
    int off = kHeaderBytes;  // barriers, stage records, step offsets, tile cursors
    P.off_prefix = off; off = round_up(off + (P.B + 1) * 4, 128);
    P.off_pq = off; off = round_up(off + 2 * P.pq_bytes, 128);
    P.off_pf = off; off = round_up(off + std::max(pf_bytes, 16), 1024);
    P.off_kv = off; off += stages * P.stage_bytes;
    return off + 1024;  // alignment slack
  };
  const int budget = 226 * 1024;  // opt-in limit (227 KB) less static shared memory
  const char* cap_env = std::getenv("LRKV_DECODE_STREAM_STAGES");  // tuning: at most this many stages
  const int cap = (cap_env && *cap_env) ? std::max(2, std::atoi(cap_env)) : 16;
  int stages = 0;
  while (stages < std::min(16, cap) && layout(stages + 1) <= budget) ++stages;
  if (stages < 2) return LRKV_ERR_UNSUPPORTED;
  P.stages = stages;
  {
    const int plain = P.stage_bytes;
    P.stage_bytes = round_up(P.off_ks + 16 * kKsBoxT * 4, 1024);
    if (layout(P.stages) <= budget)
      P.ks_bytes = 16 * kKsBoxT * 4;
    else
      P.stage_bytes = plain;
  }
  P.smem_bytes = layout(P.stages);
  // B^K of a row tile staged through the last ring stages when it fits
  // (leaving at least one stage for the first tiles), those stages getting
  // their tiles after the absorb; otherwise each absorb thread loads its
  // columns at entry.  Tuning: LRKV_DECODE_BK_REGS=1 takes the register
  // path whenever a thread's columns are one chunk (d_h / bk_dsplit <=
  // kBkChunk rows); measured slower on 8 x 4K rows of 16 heads, rank 28:
  // the absorb from registers took ~5.5K cycles against ~2.4K from shared
  // memory.
  {
    P.bk_head_bytes = dh * r * 2;
    const long long bk_bytes = 16ll * P.bk_head_bytes;
    const int nbk = r > 0 ? static_cast<int>((bk_bytes + P.stage_bytes - 1) / P.stage_bytes) : 0;
    const char* regs_env = std::getenv("LRKV_DECODE_BK_REGS");
    const bool one_chunk = dh / P.bk_dsplit <= kBkChunk && regs_env && regs_env[0] == '1';
    P.bk_stages = (r > 0 && nbk < stages && !one_chunk) ? nbk : 0;
  }
  P.pfw = 0;  // L2 prefetch window beyond the ring (tiles); set with the grid
  return stream_fn(P) ? LRKV_OK : LRKV_ERR_UNSUPPORTED;
}

// Host preparation of a streaming launch: the latent tensor maps and the
// kernel's shared-memory attribute (set once per kernel and size).
lrkv_status stream_prepare(const DecodePlan& P, CUtensorMap* tm_zk, CUtensorMap* tm_zv, CUtensorMap* tm_ks) {
  const StreamFn kern = stream_fn(P);
  if (!kern) return LRKV_ERR_UNSUPPORTED;
  std::memset(tm_zk, 0, sizeof(*tm_zk));
  std::memset(tm_zv, 0, sizeof(*tm_zv));
  std::memset(tm_ks, 0, sizeof(*tm_ks));
  // key scales [B][H][max_len] fp32 in boxes of [16 heads][kKsBoxT rows]
  if (P.ks_tma &&
      !make_tmap_3d_f32(tm_ks, P.key_scale, static_cast<uint64_t>(P.max_len), static_cast<uint64_t>(P.H),
                        static_cast<uint64_t>(P.B), kKsBoxT, 16u))
    return LRKV_ERR_CUDA;
  if (P.r > 0) {
    // z[b][t][h][c] viewed as [b][segment][t][hs r]: dims (inner first)
    // {hs r, rows, H / hs, sequences}, strides t: H r, segment: hs r, b: rows H r
    // (rows, sequences) = (max_len, B), or (page_size, pages) for a paged cache
    const uint64_t row = static_cast<uint64_t>(P.H) * P.r * 2;
    const uint64_t dims[4] = {static_cast<uint64_t>(P.segw), static_cast<uint64_t>(P.map_len),
                              static_cast<uint64_t>(P.H / P.hs), static_cast<uint64_t>(P.map_seqs)};
    const uint64_t strides[3] = {row, static_cast<uint64_t>(P.segw) * 2, row * P.map_len};
    const uint32_t box[4] = {static_cast<uint32_t>(P.segp), static_cast<uint32_t>(kT),
                             static_cast<uint32_t>(P.nsb), 1u};
    if (!make_tmap_4d_bf16_strided(tm_zk, P.z_k, dims, strides, box) ||
        !make_tmap_4d_bf16_strided(tm_zv, P.z_v, dims, strides, box))
      return LRKV_ERR_CUDA;
  }
  // the largest size set so far per kernel (per device: the attribute is a
  // property of the function in the current context)
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> set_bytes;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LRKV_ERR_CUDA;
  std::lock_guard<std::mutex> lock(mu);
  int& have = set_bytes[{dev, reinterpret_cast<const void*>(kern)}];
  if (have < P.smem_bytes) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, P.smem_bytes) != cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared) !=
            cudaSuccess)
      return LRKV_ERR_CUDA;
    have = P.smem_bytes;
  }
  return LRKV_OK;
}

lrkv_status stream_launch(const DecodePlan& P, cudaStream_t stream, bool pdl, const CUtensorMap& tm_k,
                          const CUtensorMap& tm_v, const CUtensorMap& tm_zk, const CUtensorMap& tm_zv,
                          const CUtensorMap& tm_ks) {
  const StreamFn kern = stream_fn(P);
  if (!kern) return LRKV_ERR_UNSUPPORTED;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(P.grid, P.mt);
  cfg.blockDim = dim3(P.nthreads);
  cfg.dynamicSmemBytes = P.smem_bytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, P, tm_k, tm_v, tm_zk, tm_zv, tm_ks) == cudaSuccess ? LRKV_OK : LRKV_ERR_CUDA;
}

}  // namespace lrkv
