// Host-side launch helpers of the tensor-core kernels: the driver's cuTensorMapEncodeTiled, looked
// up once, and the number of CTA pairs a kernel can keep resident, queried once per device.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>
#include <stddef.h>

namespace wan {
// The encoder of tiled tensor maps (null if the driver has none); thread-safe, looked up on first use.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// CTA pairs (clusters of 2 CTAs of `threads` threads and `smem` bytes of dynamic shared memory)
// of `kern` that the current device holds at once: the persistent grids launch this many pairs so
// that none waits for a second wave (a pair lives in one GPC, so this can be below sms / 2). The
// occupancy query runs once per (kernel, device) and its answer is kept, guarded for calls from
// several host threads; sms / 2 (at least 1) when the query fails. The kernel's shared-memory
// attribute must already be set.
int resident_pairs(const void* kern, int threads, size_t smem, int sms);
}  // namespace wan
