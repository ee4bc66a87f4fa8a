// Host side of the TMA tensor maps: the driver's cuTensorMapEncodeTiled, looked up once.
#pragma once
#include <cuda.h>
#include <cudaTypedefs.h>

namespace wan {
// The encoder of tiled tensor maps (null if the driver has none); thread-safe, looked up on first use.
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();
}  // namespace wan
