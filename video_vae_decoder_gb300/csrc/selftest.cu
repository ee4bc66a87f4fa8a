// wan_selftest_wait_timeout: runs the timeout path of the library's bounded device waits on
// purpose, with a short bound and a wait that cannot complete, so that a caller (or a test) can
// check that a kernel which gives up a wait winds down, records WAN_ERR_TIMEOUT for
// wan_device_status(), and leaves the context usable. No wait here is unbounded and nothing
// faults: every waiting thread gives up after `wait_cycles` SM cycles and returns.
#include <cuda_runtime.h>

#include <stdint.h>

#include "abi_util.h"
#include "common.cuh"
#include "gn_silu.h"
#include "wan.h"

namespace wan {
namespace {

// One thread waits on an mbarrier whose phase needs two arrivals and gets one: the bounded wait
// of the tensor-core kernels' pipelines gives up after `limit` cycles and records its bit.
__global__ void mbar_timeout_kernel(unsigned* err, long long limit) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 2);
    fence_mbarrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    mbar_arrive(&bar);
    mbar_wait(&bar, 0, err, kDevErrTimeoutProducer, limit);
  }
}

}  // namespace
}  // namespace wan

extern "C" wan_status wan_selftest_wait_timeout(int which, long long wait_cycles, const wan_bf16* x, wan_bf16* y,
                                                const float* gamma, const float* beta, int N, int T, int H, int W,
                                                int C, int groups, float eps, void* ws, size_t ws_bytes,
                                                void* stream) {
  WAN_CALL_RANGE();
  using namespace wan;
  if (wait_cycles < 1000 || wait_cycles > 100000000LL || (which != 0 && which != 1)) return WAN_ERR_INVALID_ARG;
  if (which == 0) {
    wan_status st = check_gn(x, y, gamma, beta, N, T, H, W, C, groups, eps);
    if (st != WAN_OK) return st;
    const size_t bytes = (size_t)N * T * H * W * C * sizeof(wan_bf16);
    if (overlap(x, bytes, y, bytes)) return WAN_ERR_INVALID_ARG;
    const size_t need = wan_workspace_size(WAN_OP_GN_SILU, N, T, H, W, C, 0, groups);
    if (!ws || ws_bytes < need) return WAN_ERR_WORKSPACE;
    if (!aligned16(ws)) return WAN_ERR_MISALIGNED;
  }
  unsigned* err = device_error_word();
  if (!err) return WAN_ERR_CUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (which == 1) {
    mbar_timeout_kernel<<<1, 32, 0, s>>>(err, wait_cycles);
    return cuda_status(cudaGetLastError());
  }
  // wan_gn_silu's kernel with its first grid barrier one arrival beyond the grid: every CTA
  // arrives, waits `wait_cycles`, records the timeout and returns before writing y.
  return cuda_status(gn_silu_launch(x, y, gamma, beta, N, T, H, W, C, groups, eps, ws, sm_count(), s, true, nullptr,
                                    false, wait_cycles, 1u));
}
