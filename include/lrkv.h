/*
 * lrkv.h — C ABI of the GB300 (sm_103a) LRKV factored-cache attention library.
 *
 * Low-Rank Key-Value attention writes each head's key/value projection as a
 * shared dense matrix plus a per-head rank-r residual, W_h = W_s + U_h B_h^T
 * ("Low-Rank Key Value Attention：中文研读笔记", §2.1, Eqs. (2)-(5)).  A token
 * therefore caches one shared row k_s, v_s (d_h each) plus per-head latents
 * z_k,h = x U_h^K and z_v,h = x U_h^V (r each) (same page, §2.3), and attention
 * runs directly on that factored cache by associativity (same page, §2.4,
 * Eqs. (6)-(7); "Low-Rank Key Value Attention | What a shared cache can
 * preserve", §3, Algorithm 2):
 *
 *   score_{h,j} = (q_h . k_s,j + (q_h B_h^K) . z_k,h,j) / sqrt(d_h)
 *   a_h        = softmax over the visible j of the summed scores (ONE softmax)
 *   o_h        = sum_j a_{h,j} v_s,j + (sum_j a_{h,j} z_v,h,j) (B_h^V)^T
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  * Memory.  Every pointer argument except `dims`, `bytes` and `out_status`
 *    is a DEVICE pointer on the current CUDA device.  The caller owns and
 *    allocates every buffer, including the workspace; the library allocates
 *    nothing and keeps no state between calls.  All work is enqueued on
 *    `stream` (a cudaStream_t passed as void*; NULL is the legacy default
 *    stream) and the calls return without synchronising.
 *  * Element types.  `dims->dtype` fixes the storage type of q, the cache
 *    (k_s, v_s, z_k, z_v), the bases (b_k, b_v) and the append inputs:
 *    LRKV_F32 (IEEE binary32) or LRKV_BF16 (bfloat16).  Accumulation is fp32.
 *    Outputs `out` and `lse` are always fp32.
 *  * Layouts (row-major, C order):
 *      k_s, v_s   [batch][max_len][head_dim]
 *      z_k, z_v   [batch][max_len][heads][rank]
 *      b_k, b_v   [heads][head_dim][rank]       (B_h is d_h x r; K_h = S + R_h B_h^T)
 *      seq_lens   [batch] int32, visible history length of each sequence
 *  * Alignment.  Cache pointers, q, x and the append weights must be 16-byte
 *    aligned, and head_dim*sizeof(elem) and heads*rank*sizeof(elem) must be
 *    multiples of 16 bytes (every row is moved by the Tensor Memory
 *    Accelerator, which copies 16-byte-aligned spans).
 *  * Errors.  Arguments are checked on the host before anything is enqueued;
 *    a failed check returns a status and enqueues nothing.  A CUDA launch
 *    failure returns LRKV_ERR_CUDA.  Problems only the device can see (a
 *    seq_lens entry outside [0, max_len], a bounded wait that ran out) never
 *    trap: the kernels clamp, finish, and record the status in the workspace,
 *    readable with lrkv_read_device_status().  A wait of the bf16 decode scan
 *    for its copies gives up after LRKV_WAIT_LIMIT_CYCLES SM cycles (an
 *    environment variable read at each call; default 2e9, about 1 s); the
 *    scan then skips the work that depended on it, still waits at the full
 *    bound for every copy it issued, and records LRKV_ERR_TIMEOUT.  Set the
 *    variable only to exercise that path.
 *  * Planning.  Launch grids and workspace sizes follow the current device's
 *    SM count, or LRKV_SM_COUNT when that environment variable holds a
 *    positive number (read at each call: workspace sizes without a device;
 *    results are the same for any value).
 *  * Scale.  dims->scale <= 0 selects 1/sqrt(head_dim), the scale of the
 *    summed score (technical review, §3 "Associative decode").
 *  * Positions.  Without RoPE the decode and prefill carry no position
 *    encoding; lrkv_decode_rope applies full RoPE to the keys exactly.
 */
#ifndef LRKV_H_
#define LRKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define LRKV_ABI_VERSION 1

typedef enum {
  LRKV_OK = 0,
  LRKV_ERR_INVALID_ARG = 1,   /* null pointer, non-positive size, bad dtype          */
  LRKV_ERR_UNSUPPORTED = 2,   /* valid but outside the shapes the kernels implement */
  LRKV_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required          */
  LRKV_ERR_CUDA = 4,          /* a CUDA runtime call or kernel launch failed         */
  LRKV_ERR_TIMEOUT = 5,       /* device: a bounded wait ran out (reported, not trapped) */
  LRKV_ERR_DEVICE_BOUNDS = 6  /* device: a length, position or page out of range; clamped or skipped */
} lrkv_status;

typedef enum { LRKV_F32 = 0, LRKV_BF16 = 1 } lrkv_dtype;

typedef struct {
  int batch;       /* B >= 1                                                  */
  int heads;       /* H >= 1                                                  */
  int head_dim;    /* d_h >= 1                                                */
  int rank;        /* r >= 0; r = 0 is MQA-style sharing (notes §2.1)         */
  int max_len;     /* token capacity of each sequence's cache rows            */
  lrkv_dtype dtype;
  float scale;     /* <= 0 selects 1/sqrt(head_dim)                           */
} lrkv_dims;

typedef void* lrkv_stream_t; /* a cudaStream_t */

/* ABI version of the loaded library (LRKV_ABI_VERSION). */
int lrkv_abi_version(void);

/* Human-readable name of a status code; never NULL. */
const char* lrkv_status_string(lrkv_status status);

/* Cache elements one token adds per layer: 2 (d_h + H r)
 * ("Low-Rank Key Value Attention：中文研读笔记", §2.5, Eq. (8)).
 * Returns 0 if any argument is negative. */
size_t lrkv_cache_elems_per_token(int heads, int head_dim, int rank);

/* Bytes of device workspace lrkv_decode needs for `dims` on the current
 * device (the split-KV partials depend on its SM count).  The workspace may
 * hold anything on entry; only its first 16 bytes (the device status word)
 * keep meaning after a call. */
lrkv_status lrkv_decode_workspace_size(const lrkv_dims* dims, size_t* bytes);

/*
 * One decode step of every head of every sequence against its factored
 * history ("Low-Rank Key Value Attention | What a shared cache can preserve",
 * §3, Algorithm 2, and the fused online-softmax paragraph after it;
 * "Low-Rank Key Value Attention：中文研读笔记", §2.4, Eqs. (6)-(7)).
 *
 *   q        [batch][heads][head_dim]  query of the new token (dtype)
 *   k_s, v_s, z_k, z_v                 the factored cache (layouts above); the
 *                                       new token's rows must already be in it
 *   b_k, b_v [heads][head_dim][rank]   reconstruction bases (dtype)
 *   seq_lens [batch] int32             sequence b attends rows [0, seq_lens[b]);
 *                                       0 gives out = 0 and lse = -inf
 *   out      [batch][heads][head_dim]  fp32 result o_h (heads not concatenated,
 *                                       no output projection)
 *   lse      [batch][heads] fp32 or NULL: natural-log log-sum-exp of the scaled
 *                                       scores
 *   ws, ws_bytes                        workspace of at least
 *                                       lrkv_decode_workspace_size() bytes
 * z_k, z_v, b_k, b_v may be NULL when rank == 0.
 * Supported: dtype BF16 with head_dim a multiple of 16 (<= 256) and rank <= 64,
 * ceil(heads/16) * head_dim / 8 <= 32; dtype F32 with rank <= 64,
 * head_dim <= 8 * (lanes per head); batch <= 4096.  Others return
 * LRKV_ERR_UNSUPPORTED.
 * The call's kernels use programmatic dependent launch: its inputs must be
 * complete when the launch before it on the stream lets its dependents start
 * (a kernel that does not do so explicitly lets them start when it ends).
 */
lrkv_status lrkv_decode(const lrkv_dims* dims, const void* q, const void* k_s, const void* v_s,
                        const void* z_k, const void* z_v, const void* b_k, const void* b_v,
                        const int32_t* seq_lens, float* out, float* lse, void* ws, size_t ws_bytes,
                        lrkv_stream_t stream);

/*
 * lrkv_decode, plus two CUDA events (cudaEvent_t passed as void*, created by
 * the caller) recorded on `stream` immediately before and after the split-KV
 * kernel, the HBM-bound scan that dominates a decode step.  Used to time that
 * kernel alone; with the events in place the kernels of the step run
 * strictly one after another instead of overlapping their launch.  While
 * `stream` is being captured into a CUDA graph the events are recorded as
 * external event-record nodes, so that graph replays can be timed with them.
 * Both events are required (LRKV_ERR_INVALID_ARG otherwise).
 */
lrkv_status lrkv_decode_profiled(const lrkv_dims* dims, const void* q, const void* k_s,
                                 const void* v_s, const void* z_k, const void* z_v, const void* b_k,
                                 const void* b_v, const int32_t* seq_lens, float* out, float* lse,
                                 void* ws, size_t ws_bytes, lrkv_stream_t stream,
                                 void* ev_split_begin, void* ev_split_end);

/*
 * Size of the workspace array built into the library for
 * lrkv_decode_static_scratch: 16 MiB of device memory on every GPU that loads
 * the library, held until the process exits.
 */
#define LRKV_STATIC_SCRATCH_BYTES (16u * 1024u * 1024u)

/*
 * lrkv_decode for callers that cannot allocate device memory.  The LRKV pages
 * have no counterpart of this entry point: it only changes where the decode
 * workspace comes from.
 *
 * Some callers cannot hand lrkv_decode a workspace: a plugin inside a host
 * runtime that owns all device memory through its own pool, or a serving path
 * that must not allocate (and so possibly synchronise or fail) in the middle
 * of a request.  This call takes the workspace from a fixed array of
 * LRKV_STATIC_SCRATCH_BYTES compiled into the library and allocates nothing
 * (no cudaMalloc, cudaFree or allocating library routine).  Arguments and
 * results are those of lrkv_decode, without ws/ws_bytes.
 *
 *  * Shapes whose workspace (lrkv_decode_workspace_size) exceeds
 *    LRKV_STATIC_SCRATCH_BYTES return LRKV_ERR_WORKSPACE and enqueue nothing.
 *  * The first call on a device looks up the array's device address with the
 *    device current; make that first call before any stream capture.
 *  * All calls on a device share the array and it keeps the last call's
 *    contents; nothing in it has to start at zero.  Calls whose kernels
 *    overlap on the GPU (unordered streams) race on it.
 *  * The device status word lives at offset 0 of that array;
 *    lrkv_read_static_scratch_status reads it back (the last call's).
 */
lrkv_status lrkv_decode_static_scratch(const lrkv_dims* dims, const void* q, const void* k_s,
                                       const void* v_s, const void* z_k, const void* z_v,
                                       const void* b_k, const void* b_v, const int32_t* seq_lens,
                                       float* out, float* lse, lrkv_stream_t stream);

/*
 * The device status of the last lrkv_decode_static_scratch call on the
 * current device, as lrkv_read_device_status reports a workspace's: waits
 * for `stream` to drain, then sets *out_status to LRKV_OK,
 * LRKV_ERR_DEVICE_BOUNDS or LRKV_ERR_TIMEOUT.  Returns LRKV_ERR_INVALID_ARG
 * for a null out_status, LRKV_ERR_CUDA when the copy fails.  Allocates nothing.
 */
lrkv_status lrkv_read_static_scratch_status(lrkv_stream_t stream, lrkv_status* out_status);

/*
 * Append new tokens to the factored cache ("Low-Rank Key Value Attention |
 * What a shared cache can preserve", §3, Algorithm 1; "Low-Rank Key Value
 * Attention：中文研读笔记", §2.3): for every new token row x of sequence b,
 *   k_s = x W_sK^T, v_s = x W_sV^T (d_h each), and for every head h
 *   z_k,h = x U_h^K, z_v,h = x U_h^V (r each),
 * stored at cache row start_pos[b] + t.  One GEMM on the tensor cores with
 * fp32 accumulation; results rounded to bf16.
 *
 *   x          [batch][n_new][d_model]            layer input (bf16)
 *   w_sk, w_sv [head_dim][d_model]                shared projections, stored
 *                                                  output-major (row = output
 *                                                  column, like a Linear weight)
 *   u_k, u_v   [heads * rank][d_model]            per-head residual factors,
 *                                                  output-major; row h*r + c is
 *                                                  column c of U_h
 *   start_pos  [batch] int32 (device)             first cache row written
 *   k_s, v_s, z_k, z_v                            the cache (layouts above)
 *   ws, ws_bytes >= 16                            device status word
 * Supported: dtype BF16; d_model, head_dim and heads*rank multiples of 64.
 * Rows with start_pos[b] + t outside [0, max_len) are not written and set
 * LRKV_ERR_DEVICE_BOUNDS in the status word.
 */
lrkv_status lrkv_append(const lrkv_dims* dims, int d_model, int n_new, const void* x, const void* w_sk,
                        const void* w_sv, const void* u_k, const void* u_v, const int32_t* start_pos,
                        void* k_s, void* v_s, void* z_k, void* z_v, void* ws, size_t ws_bytes,
                        lrkv_stream_t stream);

/*
 * Causal attention of q_len new queries per sequence against the factored
 * cache, on the tensor cores ("Low-Rank Key Value Attention：中文研读笔记",
 * §2.4, Eqs. (6)-(7); "Low-Rank Key Value Attention | What a shared cache can
 * preserve", §3): logits [q_h | q_h B_h^K] . [k_s | z_k,h] / sqrt(d_h), one
 * causal softmax, values sum_j a_j v_s,j + (sum_j a_j z_v,h,j) (B_h^V)^T.
 *
 *   q        [batch][q_len][heads][head_dim]   queries (dtype)
 *   cache    rows [0, seq_lens[b]) hold the history including the q_len new
 *            tokens (append them first); query i sits at position
 *            seq_lens[b] - q_len + i and sees keys j <= that position
 *   out      [batch][q_len][heads][head_dim] fp32
 *   lse      [batch][heads][q_len] fp32 or NULL (natural log)
 *   ws, ws_bytes >= lrkv_prefill_workspace_size()  device status word (16-byte
 *                                              aligned)
 * q_h B_h^K enters its tensor-core contraction with the latents as the sum
 * of two bf16 parts (about 16 significant bits).  Supported: dtype BF16,
 * head_dim 128, rank 64.  seq_lens[b]
 * outside [q_len, max_len] is clamped and sets LRKV_ERR_DEVICE_BOUNDS.
 */
lrkv_status lrkv_prefill(const lrkv_dims* dims, int q_len, const void* q, const void* k_s, const void* v_s,
                         const void* z_k, const void* z_v, const void* b_k, const void* b_v,
                         const int32_t* seq_lens, float* out, float* lse, void* ws, size_t ws_bytes,
                         lrkv_stream_t stream);

/*
 * Bytes of device workspace lrkv_prefill, lrkv_prefill_normed and
 * lrkv_prefill_paged need for `dims` and `q_len` queries per sequence
 * ("Low-Rank Key Value Attention | What a shared cache can preserve", §3: the
 * prefill is Algorithm 2 for a block of causal queries).  The workspace holds
 * the device status word; the prefill kernel keeps its partial results on
 * chip and needs no other scratch memory.  Returns LRKV_ERR_INVALID_ARG or
 * LRKV_ERR_UNSUPPORTED for the shapes lrkv_prefill rejects (the same checks,
 * without the pointers); a prefill given fewer bytes returns
 * LRKV_ERR_WORKSPACE and enqueues nothing.
 */
lrkv_status lrkv_prefill_workspace_size(const lrkv_dims* dims, int q_len, size_t* bytes);

/*
 * One decode step of a layer: the new token's cache rows from its layer
 * input x, then attention over the cache that now holds them ("Low-Rank Key
 * Value Attention | What a shared cache can preserve", §3, Algorithm 1 for
 * one token, then Algorithm 2; "Low-Rank Key Value Attention：中文研读笔记",
 * §2.3-§2.4).  For every sequence b the token's
 *   k_s = x W_sK^T, v_s = x W_sV^T, z_k,h = x U_h^K, z_v,h = x U_h^V
 * (fp32 accumulation, rounded to bf16) are written at cache row
 * seq_lens[b] - 1, then the call decodes exactly like lrkv_decode over rows
 * [0, seq_lens[b]).  Two launches chained by programmatic dependent launch
 * (the decode's set-up overlaps the projection), plus the decode's merge.
 *
 *   x          [batch][d_model]               the new token's layer input
 *   w_sk, w_sv [head_dim][d_model]            as in lrkv_append (output-major)
 *   u_k, u_v   [heads * rank][d_model]        as in lrkv_append
 *   q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, out, lse, ws, ws_bytes: as in
 *              lrkv_decode; seq_lens[b] counts the new token (seq_lens[b] = 0:
 *              no row is written and that sequence decodes as empty)
 * Supported: dtype BF16, rank >= 1, d_model a multiple of 8 (16-byte rows);
 * the decode's own limits.  Lengths outside [0, max_len] write no row and
 * set LRKV_ERR_DEVICE_BOUNDS through the decode.
 */
lrkv_status lrkv_decode_step(const lrkv_dims* dims, int d_model, const void* x, const void* w_sk,
                             const void* w_sv, const void* u_k, const void* u_v, const void* q, void* k_s,
                             void* v_s, void* z_k, void* z_v, const void* b_k, const void* b_v,
                             const int32_t* seq_lens, float* out, float* lse, void* ws, size_t ws_bytes,
                             lrkv_stream_t stream);

/*
 * Post-projection RMSNorm of the keys ("Low-Rank Key Value Attention | What a
 * shared cache can preserve", §8, "Post-projection normalization has a cache
 * cost"): the key of head h at token j, k = s_j + z_j B_h^T, is divided by its
 * joint RMS n = sqrt(mean_d k[d]^2 + eps) (never the two parts apart).  In a
 * kernel without RoPE the exact treatment caches one reciprocal scale per
 * head and token and multiplies the summed score by it; a per-head gain of
 * the norm is folded into q by the caller.
 *
 * lrkv_key_scales writes key_scale[b][h][t] = 1 / n (fp32) for the rows
 * t = start_pos[b] .. start_pos[b] + n_new - 1 of every sequence, from the
 * cached k_s, z_k (bf16, as stored) and B^K; rows outside [0, max_len) are
 * skipped.  Call it after appending the rows.
 *   key_scale  [batch][heads][max_len] fp32 (device), caller-allocated
 * Supported: dtype BF16, 1 <= rank <= 64, head_dim a multiple of 32 (at most
 * 256); k_s 16-byte aligned (else LRKV_ERR_INVALID_ARG).
 *
 * lrkv_decode_normed is lrkv_decode with every summed score multiplied by
 * key_scale[b][h][j] before the softmax (values are not normalised).
 * Supported: the shapes on which lrkv_decode streams bf16 (others return
 * LRKV_ERR_UNSUPPORTED).
 *
 * lrkv_prefill_normed is lrkv_prefill with the same per-key multiplication
 * of the summed scores (before the causal mask and the softmax); key_scale
 * must hold rows [0, seq_lens[b]) of every sequence.  key_scale NULL returns
 * LRKV_ERR_INVALID_ARG.  Supported: the shapes of lrkv_prefill.
 */
lrkv_status lrkv_key_scales(const lrkv_dims* dims, float eps, int n_new, const void* k_s, const void* z_k,
                            const void* b_k, const int32_t* start_pos, float* key_scale, lrkv_stream_t stream);
lrkv_status lrkv_decode_normed(const lrkv_dims* dims, const void* q, const void* k_s, const void* v_s,
                               const void* z_k, const void* z_v, const void* b_k, const void* b_v,
                               const float* key_scale, const int32_t* seq_lens, float* out, float* lse, void* ws,
                               size_t ws_bytes, lrkv_stream_t stream);
lrkv_status lrkv_prefill_normed(const lrkv_dims* dims, int q_len, const void* q, const void* k_s,
                                const void* v_s, const void* z_k, const void* z_v, const void* b_k,
                                const void* b_v, const float* key_scale, const int32_t* seq_lens, float* out,
                                float* lse, void* ws, size_t ws_bytes, lrkv_stream_t stream);

/*
 * Decode over a paged factored cache (page boundaries as a serving concern:
 * "Low-Rank Key Value Attention | What a shared cache can preserve", §4 and
 * §9; the pages give no layout).  The rows of every sequence live in pages
 * of page_size rows drawn from one pool per cache tensor:
 *   k_s, v_s     [num_pages][page_size][head_dim]
 *   z_k, z_v     [num_pages][page_size][heads][rank]
 *   block_table  [batch][max_len / page_size] int32 (device): logical row t
 *                of sequence b is row t % page_size of page
 *                block_table[b][t / page_size]; entries of blocks at or past
 *                seq_lens[b] are not read
 * dims->max_len is the logical capacity of a sequence (a multiple of
 * page_size).  Everything else (q, b_k, b_v, seq_lens, out, lse, ws, the
 * workspace size from lrkv_decode_workspace_size(dims)) is as in lrkv_decode,
 * and so is the result over the logical rows [0, seq_lens[b]).
 * page_size: a power of two >= 16 (a 16-token tile never spans two pages);
 * num_pages * page_size < 2^31.  A block table entry outside [0, num_pages)
 * reads as zero rows and sets LRKV_ERR_DEVICE_BOUNDS in the status word.
 * Supported: the shapes on which lrkv_decode streams bf16 (others return
 * LRKV_ERR_UNSUPPORTED).
 */
lrkv_status lrkv_decode_paged(const lrkv_dims* dims, int page_size, int num_pages, const int32_t* block_table,
                              const void* q, const void* k_s, const void* v_s, const void* z_k, const void* z_v,
                              const void* b_k, const void* b_v, const int32_t* seq_lens, float* out, float* lse,
                              void* ws, size_t ws_bytes, lrkv_stream_t stream);

/*
 * Appends into a paged cache (pools, block table and page_size as in
 * lrkv_decode_paged): after a prefill, at any position, across page
 * boundaries.
 *
 * lrkv_append_paged is lrkv_append writing logical row start_pos[b] + t of
 * sequence b through the block table; a row whose block names no page of the
 * pool is not written and sets LRKV_ERR_DEVICE_BOUNDS in the status word
 * (as a row past max_len does).
 *
 * lrkv_decode_step_paged is lrkv_decode_step over a paged cache: the token's
 * rows go to logical row seq_lens[b] - 1 through the block table (a page
 * outside the pool: no row; the decode flags it), then lrkv_decode_paged.
 */
/*
 * Causal prefill over a paged cache (pools, block table as in
 * lrkv_decode_paged): lrkv_prefill over the logical rows [0, seq_lens[b]);
 * the chunk's own rows are appended first (lrkv_append_paged), the rows
 * before them are the cached prefix.  page_size: a power of two >= 128 (a
 * 128-key tile never spans two pages).  A block table entry outside the pool
 * reads as zero rows and sets LRKV_ERR_DEVICE_BOUNDS.  Supported: the shapes
 * of lrkv_prefill.
 */
lrkv_status lrkv_prefill_paged(const lrkv_dims* dims, int q_len, const void* q, int page_size, int num_pages,
                               const int32_t* block_table, const void* k_s, const void* v_s, const void* z_k,
                               const void* z_v, const void* b_k, const void* b_v, const int32_t* seq_lens,
                               float* out, float* lse, void* ws, size_t ws_bytes, lrkv_stream_t stream);
lrkv_status lrkv_append_paged(const lrkv_dims* dims, int d_model, int n_new, const void* x, const void* w_sk,
                              const void* w_sv, const void* u_k, const void* u_v, const int32_t* start_pos,
                              int page_size, int num_pages, const int32_t* block_table, void* k_s, void* v_s,
                              void* z_k, void* z_v, void* ws, size_t ws_bytes, lrkv_stream_t stream);
lrkv_status lrkv_decode_step_paged(const lrkv_dims* dims, int d_model, const void* x, const void* w_sk,
                                   const void* w_sv, const void* u_k, const void* u_v, const void* q,
                                   int page_size, int num_pages, const int32_t* block_table, void* k_s, void* v_s,
                                   void* z_k, void* z_v, const void* b_k, const void* b_v, const int32_t* seq_lens,
                                   float* out, float* lse, void* ws, size_t ws_bytes, lrkv_stream_t stream);

/*
 * Decode with full rotary position embedding (RoPE) of the keys, exactly
 * ("Low-Rank Key Value Attention | What a shared cache can preserve", §8,
 * "Full RoPE needs a stronger identity"; "Low-Rank Key Value
 * Attention：中文研读笔记", §2.7).  A key rotation cannot be moved into the
 * rank-r latent for a generic basis, so the cache keeps unrotated rows and the
 * decode rebuilds each key, k_j = s_j + z_j B_h^T, turns it by the rotation of
 * its position j and takes the dot product with the query, which the caller
 * passes already rotated to its own position (the review's q~).  Values are
 * not rotated.  For head h and row j of sequence b:
 *   score = scale * q~_h . (k_j D_j),  D_j: each pair (2k, 2k+1) turned by the
 *   angle j theta_k (as the complex number x_2k + i x_2k+1 times
 *   exp(i j theta_k)), theta_k = base^(-2k / head_dim);
 * one softmax over the rows [0, seq_lens[b]); o_h as in lrkv_decode.  Row j
 * of the cache sits at position j.
 *
 * lrkv_rope_table writes the rotation table cos_sin [max_pos][head_dim] fp32
 * (device, caller-allocated): cos_sin[j][2k] = cos(j theta_k),
 * cos_sin[j][2k+1] = sin(j theta_k), with the angle and both functions in
 * fp64, rounded once to fp32.  Compute it once per model; base > 1, head_dim
 * even.
 *
 * lrkv_decode_rope takes the arguments of lrkv_decode (q is q~, [B][H][d_h]
 * in the cache dtype) plus the table and its row count max_pos (at least
 * dims->max_len, else LRKV_ERR_INVALID_ARG), and a workspace of
 * lrkv_decode_rope_workspace_size() bytes.  Supported: dtype BF16,
 * head_dim 64 or 128, rank 16, 32, 48 or 64, heads a multiple of 8, a
 * contiguous cache; others return LRKV_ERR_UNSUPPORTED.  The rebuild costs
 * head_dim x rank multiply-adds per (row, head) on the tensor cores beyond
 * lrkv_decode.
 */
lrkv_status lrkv_rope_table(int max_pos, int head_dim, float base, float* cos_sin, lrkv_stream_t stream);
lrkv_status lrkv_decode_rope_workspace_size(const lrkv_dims* dims, size_t* bytes);
lrkv_status lrkv_decode_rope(const lrkv_dims* dims, const void* q_rot, const void* k_s, const void* v_s,
                             const void* z_k, const void* z_v, const void* b_k, const void* b_v,
                             const float* cos_sin, int max_pos, const int32_t* seq_lens, float* out, float* lse,
                             void* ws, size_t ws_bytes, lrkv_stream_t stream);

/*
 * Comparison decodes on the same box ("Low-Rank Key Value Attention | What a
 * shared cache can preserve", §4 "Weight count and the two decode regimes"
 * and §5: a fair serving comparison runs optimized GQA, dense MHA and
 * absorbed MLA beside the factored kernel at the same batch, length and
 * dtype).  They are not part of the LRKV method; they measure the layouts it
 * replaces.
 *
 * lrkv_dense_decode: one decode step over materialised K/V (bf16),
 *   q [batch][heads][head_dim], k, v [batch][max_len][kv_heads][head_dim];
 *   query head h attends KV head h / (heads / kv_heads) over rows
 *   [0, seq_lens[b]) with one softmax (MHA: kv_heads = heads; GQA; MQA:
 *   kv_heads = 1); out [batch][heads][head_dim] fp32, lse [batch][heads] or
 *   NULL.  No position encoding.  Supported: head_dim 64 or 128,
 *   heads / kv_heads in {1, 2, 4, 8}.  Workspace:
 *   lrkv_dense_decode_workspace_size() bytes; status word and errors as in
 *   lrkv_decode.
 */
typedef struct {
  int batch;       /* B >= 1                                 */
  int heads;       /* query heads H >= 1                     */
  int kv_heads;    /* KV heads, dividing H                   */
  int head_dim;    /* d                                      */
  int max_len;     /* rows per sequence in k and v           */
  float scale;     /* <= 0 selects 1/sqrt(head_dim)          */
} lrkv_dense_dims;

lrkv_status lrkv_dense_decode_workspace_size(const lrkv_dense_dims* dims, size_t* bytes);
lrkv_status lrkv_dense_decode(const lrkv_dense_dims* dims, const void* q, const void* k, const void* v,
                              const int32_t* seq_lens, float* out, float* lse, void* ws, size_t ws_bytes,
                              lrkv_stream_t stream);

/*
 * lrkv_mla_decode: absorbed multi-head latent attention over one latent row
 * per token for all heads (review §5: the head computes (q_h A_h) Z^T instead
 * of materialising its keys; the values likewise), bf16 storage:
 *   q [batch][heads][head_dim], c [batch][max_len][latent_dim],
 *   w_uk, w_uv [heads][head_dim][latent_dim] (K_h = C W_uk[h]^T,
 *   V_h = C W_uv[h]^T), score q_h . k_h,j * scale (scale <= 0:
 *   1/sqrt(head_dim)), one softmax, out [batch][heads][head_dim] fp32, lse as
 *   in lrkv_decode.  Three launches: q_h W_uk[h] (fp32, in the workspace),
 *   the scan over c (q_c split into two bf16 parts for the tensor cores), and
 *   the merge, which lifts the latent sum through W_uv[h]^T.  Supported:
 *   latent_dim 256 or 512, heads 8, 16 or 32, head_dim <= 128; c 16-byte
 *   aligned.  Workspace: lrkv_mla_decode_workspace_size() bytes.
 */
typedef struct {
  int batch;
  int heads;
  int head_dim;    /* d_h of q and of the output                          */
  int latent_dim;  /* d_c of the cached latent rows                       */
  int max_len;
  float scale;     /* <= 0 selects 1/sqrt(head_dim)                       */
} lrkv_mla_dims;

lrkv_status lrkv_mla_decode_workspace_size(const lrkv_mla_dims* dims, size_t* bytes);
lrkv_status lrkv_mla_decode(const lrkv_mla_dims* dims, const void* q, const void* c, const void* w_uk,
                            const void* w_uv, const int32_t* seq_lens, float* out, float* lse, void* ws,
                            size_t ws_bytes, lrkv_stream_t stream);

/*
 * Read the device status word that the kernels of the last call(s) using
 * `ws` recorded (LRKV_OK, LRKV_ERR_TIMEOUT or LRKV_ERR_DEVICE_BOUNDS).
 * Synchronises `stream`.  Each lrkv_decode/lrkv_prefill call sets the word
 * afresh: a decode writes the bits its kernels recorded (no clearing needed
 * before a call), a prefill clears it when it starts.
 */
lrkv_status lrkv_read_device_status(const void* ws, lrkv_stream_t stream, lrkv_status* out_status);

#ifdef __cplusplus
}
#endif

#endif /* LRKV_H_ */
