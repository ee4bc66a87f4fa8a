// The driver entry point every tensor map of this library is encoded with, and the cache of the
// persistent kernels' resident CTA pairs.
#include <cuda_runtime.h>

#include <mutex>

#include "tma_host.h"

namespace wan {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
  }();
  return fn;
}

namespace {

struct PairsEntry {
  const void* kern;
  int dev;
  int pairs;
};

constexpr int kPairsEntries = 256;  // (kernel instance, device) pairs; a full table just stops caching
std::mutex g_pairs_mu;
PairsEntry g_pairs[kPairsEntries];
int g_pairs_used = 0;

}  // namespace

int resident_pairs(const void* kern, int threads, size_t smem, int sms) {
  const int fallback = sms / 2 > 0 ? sms / 2 : 1;
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return fallback;
  }
  std::lock_guard<std::mutex> lock(g_pairs_mu);
  for (int i = 0; i < g_pairs_used; ++i)
    if (g_pairs[i].kern == kern && g_pairs[i].dev == dev) return g_pairs[i].pairs;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * fallback, 1, 1);
  cfg.blockDim = dim3(threads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = fallback;
  }
  if (g_pairs_used < kPairsEntries) g_pairs[g_pairs_used++] = PairsEntry{kern, dev, n};
  return n;
}

}  // namespace wan
