// decode_noalloc.cu — lrkv_decode for callers that cannot allocate device
// memory.
//
// lrkv_decode needs a caller-owned workspace (split partials, the sequence
// prefix, q_h B_h^K and the status word).  Some callers cannot obtain one at
// the point of the call: a plugin running inside a host runtime that owns every
// device allocation through its own pool and gives the plugin only its
// operand buffers, or a serving path that is not allowed to allocate (and so
// possibly synchronise or fail) while a request is in flight.  This entry point
// takes the workspace from a fixed array compiled into the library instead.
//
// The array lives in device memory of every GPU that loads the library and is
// held until the process exits.  All calls on a device share it and it keeps
// the previous call's contents; the decode kernels rewrite every byte they
// read before reading it, so nothing has to be zeroed between calls.  That
// includes the status word at offset 0: on the fp32 path the absorb kernel
// clears it; on the bf16 streaming path every scan CTA writes its own status
// word on every launch and the merge kernel folds those words into the status
// word.  lrkv_read_static_scratch_status reads it back.  Calls whose kernels
// overlap on the GPU (different streams without ordering) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "lrkv.h"
#include "trace.h"

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[LRKV_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device; looked up once per
// device (the first call on a device performs the lookup).
lrkv_status scratch_address(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return LRKV_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return LRKV_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || !p) return LRKV_ERR_CUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return LRKV_OK;
}

}  // namespace

extern "C" lrkv_status lrkv_decode_static_scratch(const lrkv_dims* dims, const void* q, const void* k_s,
                                                  const void* v_s, const void* z_k, const void* z_v,
                                                  const void* b_k, const void* b_v, const int32_t* seq_lens,
                                                  float* out, float* lse, lrkv_stream_t stream) {
  LRKV_TRACE_CALL("lrkv_decode_static_scratch");
  size_t need = 0;
  lrkv_status st = lrkv_decode_workspace_size(dims, &need);
  if (st != LRKV_OK) return st;
  if (need > static_cast<size_t>(LRKV_STATIC_SCRATCH_BYTES)) return LRKV_ERR_WORKSPACE;
  void* ws = nullptr;
  if ((st = scratch_address(&ws)) != LRKV_OK) return st;
  return lrkv_decode(dims, q, k_s, v_s, z_k, z_v, b_k, b_v, seq_lens, out, lse, ws,
                     static_cast<size_t>(LRKV_STATIC_SCRATCH_BYTES), stream);
}

extern "C" lrkv_status lrkv_read_static_scratch_status(lrkv_stream_t stream, lrkv_status* out_status) {
  if (!out_status) return LRKV_ERR_INVALID_ARG;
  void* ws = nullptr;
  const lrkv_status st = scratch_address(&ws);
  if (st != LRKV_OK) return st;
  return lrkv_read_device_status(ws, stream, out_status);
}
