// Decode GEMM entry point for callers that cannot allocate device memory.
//
// nvfp4_gemm with the weight-streaming tensor-core kernel splits K across
// CTAs and needs a scratch buffer for the fp32 partial tiles and the per-tile
// arrival counters, which nvfp4_gemm takes from its caller.  Some callers
// have no way to provide one: a host program that was handed its operand
// buffers but owns no allocator, a plugin running inside another framework
// that controls all device memory, or a latency-critical path that is not
// allowed to allocate.  For them this file keeps the scratch in a fixed-size
// array that lives in the library itself, so the call allocates nothing.
#include <cuda_runtime.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

// Largest scratch this entry point can use (split-K partials + counters).
constexpr size_t kStaticScratchBytes = size_t(8) << 20;   // 8 MiB

// The scratch itself.  Every GPU that loads the library holds one copy until
// the process exits.  In host code the name is only a handle: the device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch, looked up once per device (with that
// device current) on the first call made on it.
uint8_t *scratch_address(int dev, cudaError_t *err) {
  static uint8_t *addr[64] = {nullptr};
  static std::once_flag once[64];
  static cudaError_t status[64];
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::call_once(once[dev], [dev] {
    void *p = nullptr;
    status[dev] = cudaGetSymbolAddress(&p, g_static_scratch);
    if (status[dev] == cudaSuccess) addr[dev] = static_cast<uint8_t *>(p);
  });
  *err = status[dev];
  return addr[dev];
}

}  // namespace
}  // namespace nvfp4

using namespace nvfp4;

extern "C" nvfp4_status nvfp4_gemm_decode_noalloc(const uint8_t *a_fp4, const uint8_t *a_sf,
                                                  const uint8_t *b_fp4, const uint8_t *b_sf,
                                                  const float *alpha, uint16_t *d, int64_t m,
                                                  int64_t n, int64_t k, nvfp4_stream_t stream) {
  if (!a_fp4 || !a_sf || !b_fp4 || !b_sf || !alpha || !d || m < 0 || n <= 0 || k <= 0)
    return NVFP4_ERR_INVALID_ARG;
  const uintptr_t any = reinterpret_cast<uintptr_t>(a_fp4) | reinterpret_cast<uintptr_t>(a_sf) |
                        reinterpret_cast<uintptr_t>(b_fp4) | reinterpret_cast<uintptr_t>(b_sf) |
                        reinterpret_cast<uintptr_t>(d);
  if ((any & 15u) != 0 || !swapab_supported(TC_W4A4, m == 0 ? 1 : m, n, k))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return NVFP4_ERR_CUDA;
  if (major != 10 || minor != 3) return NVFP4_ERR_ARCH;
  const size_t need = swapab_workspace_bytes(TC_W4A4, m == 0 ? 1 : m, n, k);
  if (need > kStaticScratchBytes) return NVFP4_ERR_UNSUPPORTED_SHAPE;   // beyond the fixed size
  if (m == 0) return NVFP4_OK;
  cudaError_t err;
  uint8_t *scratch = scratch_address(dev, &err);
  if (err != cudaSuccess || scratch == nullptr) return NVFP4_ERR_CUDA;
  const cudaStream_t st = (cudaStream_t)stream;
  // The array keeps whatever the previous call left; the arrival counters at
  // its start must begin at zero.
  if (need > 0) {
    // (the kernel's counters: one per 128-row weight tile at most, at the
    // front of the counter area)
    const size_t used = ((size_t)((n + 127) / 128) * 4 + 255) / 256 * 256;
    const size_t counter_bytes = used < kCounterArea ? used : kCounterArea;
    if (cudaMemsetAsync(scratch, 0, counter_bytes, st) != cudaSuccess) return NVFP4_ERR_CUDA;
  }
  return launch_swapab(TC_W4A4, a_fp4, a_sf, b_fp4, b_sf, alpha, nullptr, d, nullptr, nullptr, m, n,
                       k, scratch, kStaticScratchBytes, wait_limit(), st) == cudaSuccess
             ? NVFP4_OK
             : NVFP4_ERR_CUDA;
}
