// trace.h — NVTX ranges around the C-ABI calls, so that a profiler's timeline
// (Nsight Systems, ncu --nvtx) shows each library call as one named range
// over the kernels it enqueues.  NVTX v3 is header-only: with no tool
// attached a range costs a call through a null function pointer.
#pragma once

#include <nvtx3/nvToolsExt.h>

namespace lrkv {

class NvtxRange {
 public:
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
  NvtxRange(const NvtxRange&) = delete;
  NvtxRange& operator=(const NvtxRange&) = delete;
};

}  // namespace lrkv

// One range for the rest of the enclosing scope, named after the call.
#define LRKV_TRACE_CALL(name) ::lrkv::NvtxRange lrkv_trace_range_(name)
