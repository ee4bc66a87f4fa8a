// Internal host-side helpers of the entry points (defined in abi.cu), shared by every file that
// implements an extern "C" call so that all of them validate arguments the same way.
#pragma once
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>
#include <stddef.h>

#include "wan.h"

namespace wan {
// SM count of the current device (cached per device; 148 if the query fails).
int sm_count();
bool aligned16(const void* p);
// True if the byte ranges [a, a + abytes) and [b, b + bbytes) intersect (false for a null range).
bool overlap(const void* a, size_t abytes, const void* b, size_t bbytes);
wan_status cuda_status(cudaError_t e);
// The argument checks of wan_gn_silu: pointers, sizes, groups, eps, supported shape, alignment.
wan_status check_gn(const void* x, const void* y, const float* gamma, const float* beta, int N, int T, int H, int W,
                    int C, int groups, float eps);

// An NVTX range named after the entry point, open for the whole call (validation, workspace
// layout and every launch it enqueues): timeline profilers show each call by name, and ncu can
// select the kernels of one call (`--nvtx --nvtx-include "wan_resblock/"`). With no tool
// attached a push or pop is one test of a function pointer.
struct CallRange {
  explicit CallRange(const char* name) { nvtxRangePushA(name); }
  ~CallRange() { nvtxRangePop(); }
  CallRange(const CallRange&) = delete;
  CallRange& operator=(const CallRange&) = delete;
};
}  // namespace wan

#define WAN_CALL_RANGE() const ::wan::CallRange wan_call_range_(__func__)
