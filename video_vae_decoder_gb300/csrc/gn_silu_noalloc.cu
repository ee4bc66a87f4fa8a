// wan_gn_silu_noalloc: GroupNorm + SiLU for callers that cannot allocate device memory.
//
// Some hosts hand a library nothing but the tensors themselves: an application that has already
// reserved all device memory for its own pool and gives plug-ins no allocator, or a latency-bound
// loop that may not call cudaMalloc (which can synchronise the device and stall other streams)
// and has no way to hand over a workspace. This entry point serves them: its scratch lives in
// the fixed-size array below, a file-scope __device__ array that every GPU which loads this
// library holds from module load until the process exits.
//
// The computation is the one of wan_gn_silu (the same argument checks, the same kernels launched
// by the same code); only the place of the scratch differs.
#include <cuda_runtime.h>

#include <atomic>
#include <stdint.h>

#include "abi_util.h"
#include "gn_silu.h"
#include "wan.h"

namespace wan {
namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)4 << 20;  // 4 MiB per device

// The scratch. In host code `g_noalloc_scratch` names a host-side stand-in, not the device
// array: its device address comes from cudaGetSymbolAddress below, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of the scratch on the current device, looked up (with that device current) on
// the first call made on each device and kept for the life of the process; nullptr if the
// lookup failed.
void* scratch_address() {
  static std::atomic<void*> cached[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = cached[dev].load(std::memory_order_acquire);
  if (!p) {
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    cached[dev].store(p, std::memory_order_release);
  }
  return p;
}

}  // namespace
}  // namespace wan

extern "C" wan_status wan_gn_silu_noalloc(const wan_bf16* x, wan_bf16* y, const float* gamma, const float* beta,
                                          int N, int T, int H, int W, int C, int groups, float eps, void* stream) {
  WAN_CALL_RANGE();
  using namespace wan;
  wan_status st = check_gn(x, y, gamma, beta, N, T, H, W, C, groups, eps);
  if (st != WAN_OK) return st;
  const size_t bytes = (size_t)N * T * H * W * C * sizeof(wan_bf16);
  if (overlap(x, bytes, y, bytes)) return WAN_ERR_INVALID_ARG;
  const int sms = sm_count();
  // Sizes whose scratch does not fit the static array are refused, never truncated.
  if (gn_silu_workspace(N, T, H, W, C, groups, sms) > kNoAllocScratchBytes) return WAN_ERR_WORKSPACE;
  void* scratch = scratch_address();
  if (!scratch) return WAN_ERR_CUDA;
  // The launcher clears the one scratch word that must start at zero (a grid-barrier counter)
  // at the start of every call; every other word the kernel reads it has written earlier in the
  // same call (the per-span partial sums, then the per-channel coefficients).
  return cuda_status(gn_silu_launch(x, y, gamma, beta, N, T, H, W, C, groups, eps, scratch, sms,
                                    static_cast<cudaStream_t>(stream)));
}
