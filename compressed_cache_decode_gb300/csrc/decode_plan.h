// decode_plan.h — host-computed launch plan of the split-KV decode, passed by
// value to the three decode kernels (absorb, split, combine).
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/lrkv.h"

namespace lrkv {

constexpr int kMaxBatch = 4096;   // sequence-start prefix lives in shared memory
constexpr int kMaxRank = 64;      // private accumulators live in registers
constexpr int kMaxPPT = 4;        // tokens per lane per tile
constexpr int kMaxValueTiles = 4; // value-MMA accumulator tiles per warp (bf16)
constexpr int kMaxThreads = 256;

// Bits of the device status word (first 4 bytes of a workspace).
constexpr uint32_t kDevTimeout = 1u;  // a bounded wait ran out
constexpr uint32_t kDevBounds = 2u;   // a length or position was clamped

struct DecodePlan {
  // problem
  int B, H, dh, r, max_len;
  float scale_log2;  // scale * log2(e): scores live in the base-2 domain
  int bf16;          // storage dtype
  int esz;           // bytes per stored element
  // tiling
  int T;             // tokens per tile
  int lph;           // lanes per head (power of two <= 32)
  int ppt;           // tokens per lane per tile (T / lph)
  int nthreads;      // split-kernel block size
  int stages;        // TMA ring depth
  int grid;          // split CTAs launched (upper bound of the CTAs used)
  int min_tokens;    // a split CTA gets at least this many tokens
  int Hp;            // heads padded to 16 (bf16 MMA rows)
  int ksplit;        // K-split of the logits MMA over warps
  int vec;           // elements per private-latent load
  // bytes copied per token row, and padded shared-memory row strides
  int ks_row, z_row, ks_stride, z_stride;
  int q_stride;      // elements
  int p_stride;      // floats
  int w_stride;      // elements of the W (attention weight) tile
  // shared-memory carve-up (bytes from the dynamic base)
  int off_prefix, off_q, off_p, off_s, off_w, off_alpha, off_stage;
  int stage_bytes, smem_bytes;
  int combine_smem;
  // workspace carve-up
  uint32_t* status;
  int* meta;         // [0] = total tokens N, [1] = CTAs used
  int* prefix;       // [B+1] sequence starts in the concatenated token order
  float* p_abs;      // [B][H][r]  q_h B_h^K
  float* part_ml;    // [slots][H][2]  running max (log2 domain), denominator
  float* part_acc;   // [slots][H][dh + r]  unnormalised shared and private sums
  // operands
  const void* q;
  const void* k_s;
  const void* v_s;
  const void* z_k;
  const void* z_v;
  const void* b_k;
  const void* b_v;
  const int32_t* seq_lens;
  float* out;
  float* lse;
};

// Fills everything but the operand pointers; returns the workspace size.
lrkv_status decode_make_plan(const lrkv_dims& d, int num_sms, DecodePlan& P, size_t* ws_bytes);
void decode_bind_workspace(DecodePlan& P, void* ws);
lrkv_status decode_launch(const DecodePlan& P, void* stream);

}  // namespace lrkv
