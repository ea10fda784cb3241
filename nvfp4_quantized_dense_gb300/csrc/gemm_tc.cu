// tcgen05 tensor-core GEMMs (block-scaled NVFP4 MMA, accumulators in TMEM).
#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

// Status word of this device: a kernel that gives up a bounded wait records
// NVFP4_ERR_DEVICE_TIMEOUT here (first writer wins).
__device__ int g_device_status = 0;

cudaError_t read_and_clear_device_status(int *out) {
  const int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
}

bool tc_supported(TcMode, bool, int64_t, int64_t, int64_t) { return false; }

cudaError_t launch_tc(TcMode, bool, const void *, const uint8_t *, const uint8_t *, const uint8_t *,
                      const float *, const float *, uint16_t *, uint8_t *, uint8_t *, int64_t,
                      int64_t, int64_t, uint32_t, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace nvfp4
