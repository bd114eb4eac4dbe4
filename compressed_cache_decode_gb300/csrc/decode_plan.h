// decode_plan.h — host-computed launch plan of the split-KV decode, passed by
// value to the three decode kernels (absorb, split, combine).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "lrkv.h"

namespace lrkv {

constexpr int kMaxBatch = 4096;  // sequence-start prefix lives in shared memory
constexpr int kMaxRank = 64;     // q_h B_h^K of a head lives in registers
constexpr int kMaxTile = 32;     // a tile's scores of one head live in registers
constexpr int kMaxPPT = 4;       // tokens per thread in the private-score phase
constexpr int kMaxCW = 16;       // value columns per thread
constexpr int kMaxValueTiles = 4;  // value-MMA accumulator tiles per warp (bf16)
constexpr int kThreads = 256;
constexpr int kStreamConsumers = 8;  // consumer warps of the streaming kernel

// Bits of the device status word (first 4 bytes of a workspace).
constexpr uint32_t kDevTimeout = 1u;  // a bounded wait ran out
constexpr uint32_t kDevBounds = 2u;   // a length or position was clamped

struct DecodePlan {
  // problem
  int B, H, dh, r, max_len;
  float scale_log2;  // scale * log2(e): scores live in the base-2 domain
  int bf16;          // storage dtype
  int esz;           // bytes per stored element
  // tiling and thread roles
  int T;             // tokens per tile
  int ntg;           // token groups in the private-score phase (thread = head x group)
  int nrg;           // column groups in the value phase (thread = head x group)
  int cw;            // value columns per thread
  int vec;           // elements per latent vector load
  int stages;        // TMA ring depth
  int grid;          // split CTAs launched (upper bound of the CTAs used)
  int min_tokens;    // a split CTA gets at least this many tokens
  int Hp;            // heads padded to 16 (bf16 MMA rows)
  int span;          // bf16: swizzle span (bytes) of one k_s/v_s box row
  int box_cols;      // bf16: elements per box row
  int nbox;          // bf16: boxes per token row
  int kv_bytes;      // shared bytes of one k_s (or v_s) tile
  int z_row;         // bytes of one token's latents (H r esz)
  int z_bytes;       // shared bytes of one latent tile
  int q_stride;      // elements per q row in shared memory
  int s_stride;      // floats per token row of the score tiles
  int w_stride;      // bf16 elements per head row of the weight tile
  // shared-memory carve-up (bytes from the dynamic base)
  int off_prefix, off_q, off_ssh, off_sp, off_w, off_alpha, off_red, off_stage;
  int stage_bytes, smem_bytes;
  int combine_smem;
  int combine_ctas;  // grid of the combine kernel (one warp per (sequence, head), grid-stride)
  int wide_merge;    // 1: the merge runs as one CTA per (sequence, head) (large caches)
  int wide_warps;    // warps of each wide-merge CTA (8 or 16; other values: 8)
  // bf16 streaming kernel: grid (range CTAs, row tiles of 16 heads); the 8
  // warps of a CTA form 4 pairs, pair p takes every 4th 16-token tile of the
  // CTA's range (tile i in stage i % stages) and each warp of the pair 8 of
  // the 16 heads; at the end of each (sequence, range) piece every pair
  // writes its own partial.  `ngw` partials per piece (4 here, 1 for the
  // tile-synchronous kernel).
  int stream;        // 1: bf16 streaming kernel, 0: tile-synchronous kernel
  int nthreads;      // block size of the scan kernel
  int mt;            // 16-head row tiles (grid.y of the streaming kernel)
  int ngw;
  int hs;            // heads per latent segment (a power of two dividing H)
  int segw;          // latent elements per segment (hs r, a multiple of 16)
  int segp;          // padded elements per segment row in shared memory (segw + 8)
  int nsb;           // segments per row tile (16 / hs)
  int zt_bytes;      // shared bytes of one latent tile (z_k or z_v) of a row tile
  int kst;           // 16-wide steps over the latents of 8 heads (r / 2)
  int pfw;           // tiles a CTA keeps prefetched into L2 beyond its ring
  int after_append;  // 1: the launch before writes cache rows: the scan waits for it before its first copy
  long long wait_limit;  // SM cycles a wait for a copy may take before it gives up (drains keep the full bound)
  int bk_dsplit;     // head-dim parts of the in-kernel q B^K (threads per output group)
  int bk_stages;     // ring stages that first hold the row tile's B^K (0: B^K read from global)
  int bk_warps;      // warps with absorb work (the first ones)
  int bk_head_bytes; // shared bytes per head of the staged B^K (padded)
  int zo[2][32];     // shared byte offset of 16-column latent step n of head half h2
  int pq_bytes;      // one p/q buffer: q rows [16][dh] bf16 then p rows [16][r] fp32
  // key scales of a post-projection RMSNorm decode staged with each tile: a
  // [16 heads][kKsBoxT tokens] fp32 box at stage offset off_ks (ks_bytes per
  // stage, 0: no slot) from the row rounded down to a multiple of 4;
  // ks_tma: 1 when the call stages them (else each lane loads its own)
  int ks_bytes, off_ks, ks_tma;
  int off_pq, off_pf, off_kv;
  // workspace carve-up
  uint32_t* status;
  int* meta;         // [0] = total tokens N, [1] = CTAs used
  int* prefix;       // [B+1] sequence starts in the concatenated token order
  float* p_abs;      // [B][H][r]  q_h B_h^K
  float* part_ml;    // [slots][H][2]  running max (log2 domain), denominator
  float* part_acc;   // [slots][H][dh + r]  unnormalised shared and private sums
  uint32_t* cta_status;  // [mt][grid] status bits of each streaming CTA, written every launch
  // operands
  const void* q;
  const void* k_s;
  const void* v_s;
  const void* z_k;
  const void* z_v;
  const void* b_k;
  const void* b_v;
  const int32_t* seq_lens;
  const float* key_scale;  // [B][H][max_len] reciprocal key RMS (post-projection RMSNorm) or NULL
  // cache layout: contiguous ([B][max_len] rows), or paged: logical row t of
  // sequence b is row t & (2^page_shift - 1) of page block_table[b][t >> page_shift]
  // of a pool [num_pages][2^page_shift]; the tensor maps span (map_len rows,
  // map_seqs sequences or pages)
  const int32_t* block_table;  // [B][max_blocks] or NULL (contiguous)
  int max_blocks, page_shift, num_pages;
  int map_len, map_seqs;
  float* out;
  float* lse;
  // full-RoPE decode: the cos/sin table [max_pos][dh] (pairs (cos, sin) per
  // frequency) and its staged tile ([16][cs_row] fp32 per ring stage)
  const float* rope_cs;
  int cs_row, cs_bytes, rope_max_pos;
};

// Fills everything but the operand pointers; returns the workspace size.
lrkv_status decode_make_plan(const lrkv_dims& d, int num_sms, DecodePlan& P, size_t* ws_bytes);
lrkv_status key_scale_launch(const lrkv_dims& dm, float eps, int n_new, const void* k_s, const void* z_k,
                             const void* b_k, const int32_t* start_pos, float* key_scale, void* stream);
lrkv_status step_append_launch(const lrkv_dims& dm, int d_model, const void* x, const void* w_sk,
                               const void* w_sv, const void* u_k, const void* u_v, const int32_t* seq_lens,
                               void* k_s, void* v_s, void* z_k, void* z_v, int num_sms, void* stream,
                               const int32_t* block_table = nullptr, int page_size = 0, int num_pages = 0);
void decode_bind_workspace(DecodePlan& P, void* ws);
size_t decode_workspace_bytes(const DecodePlan& P);
// The merge of a streaming decode's partials (wide or narrow, per the plan),
// launched with programmatic dependent launch when `pdl`.
lrkv_status decode_merge_launch(const DecodePlan& P, void* stream, bool pdl);
lrkv_status decode_launch(const DecodePlan& P, void* stream, void* ev_begin = nullptr, void* ev_end = nullptr);

}  // namespace lrkv
