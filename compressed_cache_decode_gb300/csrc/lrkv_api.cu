// lrkv_api.cu — the extern "C" entry points declared in include/lrkv.h:
// argument checks (host only, before anything touches the GPU), workspace
// sizing, and dispatch to the kernels.
#include <cuda_runtime.h>

#include <cstdint>

#include "host_cache.h"
#include "lrkv.h"
#include "trace.h"
#include "decode_plan.h"

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Checks that need no GPU.  Returns LRKV_OK when `d` describes a shape the
// decode kernels implement.
lrkv_status check_decode_dims(const lrkv_dims* d) {
  if (!d) return LRKV_ERR_INVALID_ARG;
  if (d->batch < 1 || d->heads < 1 || d->head_dim < 1 || d->rank < 0 || d->max_len < 1)
    return LRKV_ERR_INVALID_ARG;
  if (d->dtype != LRKV_F32 && d->dtype != LRKV_BF16) return LRKV_ERR_INVALID_ARG;
  if (!(d->scale == d->scale)) return LRKV_ERR_INVALID_ARG;  // NaN scale
  const int esz = d->dtype == LRKV_BF16 ? 2 : 4;
  if ((static_cast<long long>(d->head_dim) * esz) % 16 != 0) return LRKV_ERR_UNSUPPORTED;
  if ((static_cast<long long>(d->heads) * d->rank * esz) % 16 != 0) return LRKV_ERR_UNSUPPORTED;
  if (d->batch > lrkv::kMaxBatch || d->rank > lrkv::kMaxRank || d->head_dim > 256 || d->heads > 256)
    return LRKV_ERR_UNSUPPORTED;
  if (d->dtype == LRKV_BF16 && d->head_dim % 16 != 0) return LRKV_ERR_UNSUPPORTED;
  if (static_cast<long long>(d->batch) * d->max_len > (1LL << 31) - 1) return LRKV_ERR_UNSUPPORTED;
  return LRKV_OK;
}

lrkv_status current_sm_count(int* n) {
  *n = lrkv::device_sm_count();
  return *n > 0 ? LRKV_OK : LRKV_ERR_CUDA;
}

}  // namespace

extern "C" {

int lrkv_abi_version(void) { return LRKV_ABI_VERSION; }

const char* lrkv_status_string(lrkv_status s) {
  switch (s) {
    case LRKV_OK: return "LRKV_OK";
    case LRKV_ERR_INVALID_ARG: return "LRKV_ERR_INVALID_ARG";
    case LRKV_ERR_UNSUPPORTED: return "LRKV_ERR_UNSUPPORTED";
    case LRKV_ERR_WORKSPACE: return "LRKV_ERR_WORKSPACE";
    case LRKV_ERR_CUDA: return "LRKV_ERR_CUDA";
    case LRKV_ERR_TIMEOUT: return "LRKV_ERR_TIMEOUT";
    case LRKV_ERR_DEVICE_BOUNDS: return "LRKV_ERR_DEVICE_BOUNDS";
  }
  return "LRKV_ERR_UNKNOWN";
}

size_t lrkv_cache_elems_per_token(int heads, int head_dim, int rank) {
  if (heads < 0 || head_dim < 0 || rank < 0) return 0;
  return 2 * (static_cast<size_t>(head_dim) + static_cast<size_t>(heads) * static_cast<size_t>(rank));
}

lrkv_status lrkv_decode_workspace_size(const lrkv_dims* dims, size_t* bytes) {
  if (!bytes) return LRKV_ERR_INVALID_ARG;
  lrkv_status st = check_decode_dims(dims);
  if (st != LRKV_OK) return st;
  int sms = 0;
  if ((st = current_sm_count(&sms)) != LRKV_OK) return st;
  lrkv::DecodePlan P;
  return lrkv::decode_make_plan(*dims, sms, P, bytes);
}

}  // extern "C"

namespace {

// A paged cache: pools of num_pages pages of page_size rows, block_table [B][max_len / page_size].
struct PagedCache {
  const int32_t* block_table;
  int page_size, num_pages;
};

// Sets the paging fields of a plan (checks done by the caller).
void set_paging(lrkv::DecodePlan& P, const lrkv_dims& d, const PagedCache& pc) {
  int shift = 0;
  while ((1 << shift) < pc.page_size) ++shift;
  P.block_table = pc.block_table;
  P.max_blocks = d.max_len / pc.page_size;
  P.page_shift = shift;
  P.num_pages = pc.num_pages;
  P.map_len = pc.page_size;
  P.map_seqs = pc.num_pages;
}

lrkv_status check_paging(const lrkv_dims* dims, const PagedCache& pc) {
  if (!dims || !pc.block_table) return LRKV_ERR_INVALID_ARG;
  if (pc.page_size < 16 || (pc.page_size & (pc.page_size - 1)) != 0 || pc.num_pages < 1) return LRKV_ERR_INVALID_ARG;
  if (dims->max_len % pc.page_size != 0) return LRKV_ERR_INVALID_ARG;
  if (static_cast<long long>(pc.num_pages) * pc.page_size > (1LL << 31) - 1) return LRKV_ERR_UNSUPPORTED;
  return LRKV_OK;
}


lrkv_status decode_common(const lrkv_dims* dims, const void* q, const void* k_s, const void* v_s,
                          const void* z_k, const void* z_v, const void* b_k, const void* b_v,
                          const int32_t* seq_lens, float* out, float* lse, void* ws, size_t ws_bytes,
                          lrkv_stream_t stream, void* ev_begin, void* ev_end,
                          const float* key_scale = nullptr, const PagedCache* paged = nullptr) {
  lrkv_status st = check_decode_dims(dims);
  if (st != LRKV_OK) return st;
  if (!q || !k_s || !v_s || !seq_lens || !out) return LRKV_ERR_INVALID_ARG;
  if (dims->rank > 0 && (!z_k || !z_v || !b_k || !b_v)) return LRKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_s) || !aligned16(v_s)) return LRKV_ERR_INVALID_ARG;
  if (dims->rank > 0 && (!aligned16(z_k) || !aligned16(z_v))) return LRKV_ERR_INVALID_ARG;
  if (!ws) return LRKV_ERR_WORKSPACE;
  if (!aligned16(ws)) return LRKV_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = current_sm_count(&sms)) != LRKV_OK) return st;
  lrkv::DecodePlan P;
  size_t need = 0;
  if ((st = lrkv::decode_make_plan(*dims, sms, P, &need)) != LRKV_OK) return st;
  if (ws_bytes < need) return LRKV_ERR_WORKSPACE;
  // post-projection RMSNorm and the paged cache: the streaming scan only
  if ((key_scale || paged) && !P.stream) return LRKV_ERR_UNSUPPORTED;
  if (paged) set_paging(P, *dims, *paged);
  lrkv::decode_bind_workspace(P, ws);
  P.q = q; P.k_s = k_s; P.v_s = v_s; P.z_k = z_k; P.z_v = z_v; P.b_k = b_k; P.b_v = b_v;
  P.seq_lens = seq_lens; P.out = out; P.lse = lse;
  P.key_scale = key_scale;
  // key scales staged with the tiles: a slot in the ring stages and rows of
  // a multiple of 16 bytes (the copy's stride rule); else each lane loads its own
  P.ks_tma = key_scale && P.ks_bytes > 0 && dims->max_len % 4 == 0 && aligned16(key_scale);
  return lrkv::decode_launch(P, stream, ev_begin, ev_end);
}

}  // namespace

extern "C" {

lrkv_status lrkv_decode(const lrkv_dims* dims, const void* q, const void* k_s, const void* v_s,
                        const void* z_k, const void* z_v, const void* b_k, const void* b_v,
                        const int32_t* seq_lens, float* out, float* lse, void* ws, size_t ws_bytes,
                        lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_decode");
  return decode_common(dims, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, out, lse, ws, ws_bytes, stream,
                       nullptr, nullptr);
}

lrkv_status lrkv_decode_profiled(const lrkv_dims* dims, const void* q, const void* k_s, const void* v_s,
                                 const void* z_k, const void* z_v, const void* b_k, const void* b_v,
                                 const int32_t* seq_lens, float* out, float* lse, void* ws,
                                 size_t ws_bytes, lrkv_stream_t stream, void* ev_split_begin,
                                 void* ev_split_end) {
  LRKV_TRACE_CALL("lrkv_decode_profiled");
  if (!ev_split_begin || !ev_split_end) return LRKV_ERR_INVALID_ARG;
  return decode_common(dims, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, out, lse, ws, ws_bytes, stream,
                       ev_split_begin, ev_split_end);
}

lrkv_status lrkv_decode_paged(const lrkv_dims* dims, int page_size, int num_pages, const int32_t* block_table,
                              const void* q, const void* k_s, const void* v_s, const void* z_k, const void* z_v,
                              const void* b_k, const void* b_v, const int32_t* seq_lens, float* out, float* lse,
                              void* ws, size_t ws_bytes, lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_decode_paged");
  const PagedCache pc{block_table, page_size, num_pages};
  const lrkv_status st = check_paging(dims, pc);
  if (st != LRKV_OK) return st;
  if (dims->dtype != LRKV_BF16) return LRKV_ERR_UNSUPPORTED;
  return decode_common(dims, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, out, lse, ws, ws_bytes, stream, nullptr,
                       nullptr, nullptr, &pc);
}

lrkv_status lrkv_key_scales(const lrkv_dims* dims, float eps, int n_new, const void* k_s, const void* z_k,
                            const void* b_k, const int32_t* start_pos, float* key_scale, lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_key_scales");
  lrkv_status st = check_decode_dims(dims);
  if (st != LRKV_OK) return st;
  if (dims->dtype != LRKV_BF16 || dims->rank < 1 || dims->head_dim > 256) return LRKV_ERR_UNSUPPORTED;
  if (!(eps >= 0.f) || n_new < 1) return LRKV_ERR_INVALID_ARG;
  if (!k_s || !z_k || !b_k || !start_pos || !key_scale) return LRKV_ERR_INVALID_ARG;
  if (dims->rank > 64 || dims->head_dim % 32 != 0) return LRKV_ERR_UNSUPPORTED;
  if (!aligned16(k_s)) return LRKV_ERR_INVALID_ARG;  // rows read in 16-byte pieces
  return lrkv::key_scale_launch(*dims, eps, n_new, k_s, z_k, b_k, start_pos, key_scale, stream);
}

lrkv_status lrkv_decode_normed(const lrkv_dims* dims, const void* q, const void* k_s, const void* v_s,
                               const void* z_k, const void* z_v, const void* b_k, const void* b_v,
                               const float* key_scale, const int32_t* seq_lens, float* out, float* lse, void* ws,
                               size_t ws_bytes, lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_decode_normed");
  if (!key_scale || !dims) return LRKV_ERR_INVALID_ARG;
  if (dims->dtype != LRKV_BF16 || dims->rank < 1) return LRKV_ERR_UNSUPPORTED;
  return decode_common(dims, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, out, lse, ws, ws_bytes, stream, nullptr,
                       nullptr, key_scale);
}

}  // extern "C"

namespace {

lrkv_status decode_step_common(const lrkv_dims* dims, int d_model, const void* x, const void* w_sk,
                               const void* w_sv, const void* u_k, const void* u_v, const void* q, void* k_s,
                               void* v_s, void* z_k, void* z_v, const void* b_k, const void* b_v,
                               const int32_t* seq_lens, float* out, float* lse, void* ws, size_t ws_bytes,
                               lrkv_stream_t stream, const PagedCache* paged) {
  lrkv_status st = check_decode_dims(dims);
  if (st != LRKV_OK) return st;
  if (dims->dtype != LRKV_BF16 || dims->rank < 1) return LRKV_ERR_UNSUPPORTED;
  if (d_model < 8 || d_model % 8 != 0) return LRKV_ERR_UNSUPPORTED;
  if (!x || !w_sk || !w_sv || !u_k || !u_v) return LRKV_ERR_INVALID_ARG;
  if (!aligned16(x) || !aligned16(w_sk) || !aligned16(w_sv) || !aligned16(u_k) || !aligned16(u_v))
    return LRKV_ERR_INVALID_ARG;
  if (!q || !k_s || !v_s || !z_k || !z_v || !b_k || !b_v || !seq_lens || !out) return LRKV_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_s) || !aligned16(v_s) || !aligned16(z_k) || !aligned16(z_v))
    return LRKV_ERR_INVALID_ARG;
  if (!ws) return LRKV_ERR_WORKSPACE;
  if (!aligned16(ws)) return LRKV_ERR_INVALID_ARG;
  int sms = 0;
  if ((st = current_sm_count(&sms)) != LRKV_OK) return st;
  lrkv::DecodePlan P;
  size_t need = 0;
  if ((st = lrkv::decode_make_plan(*dims, sms, P, &need)) != LRKV_OK) return st;
  if (ws_bytes < need) return LRKV_ERR_WORKSPACE;
  if (paged && !P.stream) return LRKV_ERR_UNSUPPORTED;
  if (paged) set_paging(P, *dims, *paged);
  lrkv::decode_bind_workspace(P, ws);
  P.q = q; P.k_s = k_s; P.v_s = v_s; P.z_k = z_k; P.z_v = z_v; P.b_k = b_k; P.b_v = b_v;
  P.seq_lens = seq_lens; P.out = out; P.lse = lse;
  P.after_append = 1;
  // the token's rows first (every host check is done: nothing is enqueued on failure)
  if ((st = lrkv::step_append_launch(*dims, d_model, x, w_sk, w_sv, u_k, u_v, seq_lens, k_s, v_s, z_k, z_v, sms,
                                     stream, paged ? paged->block_table : nullptr, paged ? paged->page_size : 0,
                                     paged ? paged->num_pages : 0)) != LRKV_OK)
    return st;
  return lrkv::decode_launch(P, stream, nullptr, nullptr);
}

}  // namespace

extern "C" {

lrkv_status lrkv_decode_step(const lrkv_dims* dims, int d_model, const void* x, const void* w_sk,
                             const void* w_sv, const void* u_k, const void* u_v, const void* q, void* k_s,
                             void* v_s, void* z_k, void* z_v, const void* b_k, const void* b_v,
                             const int32_t* seq_lens, float* out, float* lse, void* ws, size_t ws_bytes,
                             lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_decode_step");
  return decode_step_common(dims, d_model, x, w_sk, w_sv, u_k, u_v, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens,
                            out, lse, ws, ws_bytes, stream, nullptr);
}

lrkv_status lrkv_decode_step_paged(const lrkv_dims* dims, int d_model, const void* x, const void* w_sk,
                                   const void* w_sv, const void* u_k, const void* u_v, const void* q,
                                   int page_size, int num_pages, const int32_t* block_table, void* k_s, void* v_s,
                                   void* z_k, void* z_v, const void* b_k, const void* b_v, const int32_t* seq_lens,
                                   float* out, float* lse, void* ws, size_t ws_bytes, lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_decode_step_paged");
  const PagedCache pc{block_table, page_size, num_pages};
  const lrkv_status st = check_paging(dims, pc);
  if (st != LRKV_OK) return st;
  return decode_step_common(dims, d_model, x, w_sk, w_sv, u_k, u_v, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens,
                            out, lse, ws, ws_bytes, stream, &pc);
}

lrkv_status lrkv_read_device_status(const void* ws, lrkv_stream_t stream, lrkv_status* out_status) {
  if (!ws || !out_status) return LRKV_ERR_INVALID_ARG;
  uint32_t word = 0;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(&word, ws, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess) return LRKV_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return LRKV_ERR_CUDA;
  *out_status = (word & lrkv::kDevTimeout) ? LRKV_ERR_TIMEOUT
                : (word & lrkv::kDevBounds) ? LRKV_ERR_DEVICE_BOUNDS
                                               : LRKV_OK;
  return LRKV_OK;
}

}  // extern "C"
