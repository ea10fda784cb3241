// C ABI of the NVFP4 dense-MLP library: host-side validation, the sm_103
// check, M-based kernel selection and launch.  Nothing here allocates.
#include <cuda_runtime.h>

#include <atomic>

#include "common.cuh"
#include "internal.h"

using namespace nvfp4;

namespace {

constexpr int kVersion = (1 << 16) | 0;
std::atomic<uint32_t> g_wait_limit{0};  // 0 = kernel default

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// The current device must be a GB300-class part (compute capability 10.3).
// Cached per device ordinal.
nvfp4_status check_arch() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (dev < 0 || dev >= 64) return NVFP4_ERR_ARCH;
  int c = cache[dev].load(std::memory_order_relaxed);
  if (c == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return NVFP4_ERR_CUDA;
    c = (major == 10 && minor == 3) ? 1 : 2;
    cache[dev].store(c, std::memory_order_relaxed);
  }
  return c == 1 ? NVFP4_OK : NVFP4_ERR_ARCH;
}

nvfp4_status from_cuda(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

// AUTO kernel choice: the weight-streaming tensor-core kernel (weights as
// the MMA's M operand) for decode-sized M, the prefill tensor-core kernel
// above, the CUDA-core GEMV where neither applies.
nvfp4_algo pick_algo(TcMode mode, int64_t m, int64_t n, int64_t k) {
  if (m <= 64 && swapab_supported(mode, m, n, k)) return NVFP4_ALGO_TC_SWAPAB;
  if (m > 16 && tc_supported(mode, m, n, k)) return NVFP4_ALGO_TC;
  return NVFP4_ALGO_GEMV;
}

nvfp4_status check_gemm_shape(int64_t m, int64_t n, int64_t k) {
  if (m < 0 || n <= 0 || k <= 0) return NVFP4_ERR_INVALID_ARG;
  if (k % 64 != 0 || n % 32 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (m > (int64_t(1) << 31) || n > (int64_t(1) << 31) || k > (int64_t(1) << 31))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  return NVFP4_OK;
}

}  // namespace

uint32_t nvfp4::wait_limit() { return g_wait_limit.load(); }

extern "C" {

const char *nvfp4_status_string(nvfp4_status s) {
  switch (s) {
    case NVFP4_OK: return "ok";
    case NVFP4_ERR_INVALID_ARG: return "invalid argument";
    case NVFP4_ERR_UNSUPPORTED_SHAPE: return "unsupported shape or alignment";
    case NVFP4_ERR_ARCH: return "device is not sm_103 (GB300)";
    case NVFP4_ERR_CUDA: return "CUDA runtime error";
    case NVFP4_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
  }
  return "unknown status";
}

int nvfp4_version(void) { return kVersion; }

size_t nvfp4_sf_bytes(int64_t rows, int64_t k, nvfp4_sf_layout layout) {
  if (rows < 0 || k <= 0 || k % 16 != 0) return 0;
  if (layout == NVFP4_SF_LINEAR) return (size_t)(rows * (k / 16));
  if (layout != NVFP4_SF_SWIZZLED_128x4) return 0;
  return (size_t)((rows + 127) / 128 * 128) * (size_t)((k / 16 + 3) / 4 * 4);
}

size_t nvfp4_workspace_bytes(int64_t m, int64_t n, int64_t k, nvfp4_algo algo) {
  if (m <= 0 || n <= 0 || k <= 0) return 0;
  if (algo == NVFP4_ALGO_AUTO) algo = pick_algo(TC_W4A4, m, n, k);
  if (algo != NVFP4_ALGO_TC_SWAPAB) return 0;
  return swapab_workspace_bytes(TC_W4A4, m, n, k);
}

nvfp4_status nvfp4_quantize(const uint16_t *x, int64_t m, int64_t k, const float *global_scale,
                            uint8_t *out_fp4, uint8_t *out_sf, nvfp4_sf_layout sf_layout,
                            nvfp4_stream_t stream) {
  if (!x || !global_scale || !out_fp4 || !out_sf || m < 0 || k <= 0) return NVFP4_ERR_INVALID_ARG;
  if (sf_layout != NVFP4_SF_LINEAR && sf_layout != NVFP4_SF_SWIZZLED_128x4)
    return NVFP4_ERR_INVALID_ARG;
  if (k % 16 != 0 || !aligned16(x) || !aligned16(out_fp4)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (nvfp4_status s = check_arch()) return s;
  if (m == 0) return NVFP4_OK;
  return from_cuda(launch_quantize(x, m, k, global_scale, out_fp4, out_sf,
                                   sf_layout == NVFP4_SF_SWIZZLED_128x4, (cudaStream_t)stream));
}

nvfp4_status silu_mul_nvfp4_quantize(const uint16_t *gate_up, int64_t m, int64_t i,
                                     const float *global_scale, uint8_t *out_fp4, uint8_t *out_sf,
                                     nvfp4_stream_t stream) {
  if (!gate_up || !global_scale || !out_fp4 || !out_sf || m < 0 || i <= 0)
    return NVFP4_ERR_INVALID_ARG;
  if (i % 16 != 0 || !aligned16(gate_up) || !aligned16(out_fp4)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (nvfp4_status s = check_arch()) return s;
  if (m == 0) return NVFP4_OK;
  return from_cuda(launch_silu_mul_quantize(gate_up, m, i, global_scale, out_fp4, out_sf,
                                            (cudaStream_t)stream));
}

nvfp4_status silu_mul_nvfp4_quantize_masked(const uint16_t *gate_up, const int32_t *masked_m, int64_t g,
                                            int64_t m_max, int64_t i, const float *global_scale,
                                            uint8_t *out_fp4, uint8_t *out_sf, nvfp4_stream_t stream) {
  if (!gate_up || !masked_m || !global_scale || !out_fp4 || !out_sf || g < 0 || m_max < 0 || i <= 0)
    return NVFP4_ERR_INVALID_ARG;
  if (i % 16 != 0 || !aligned16(gate_up) || !aligned16(out_fp4) || g > 65535)
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (nvfp4_status s = check_arch()) return s;
  if (g == 0 || m_max == 0) return NVFP4_OK;
  return from_cuda(launch_silu_mul_quantize_masked(gate_up, masked_m, g, m_max, i, global_scale, out_fp4,
                                                   out_sf, (cudaStream_t)stream));
}

nvfp4_status silu_mul_bf16(const uint16_t *gate_up, int64_t m, int64_t i, uint16_t *out,
                           nvfp4_stream_t stream) {
  if (!gate_up || !out || m < 0 || i <= 0) return NVFP4_ERR_INVALID_ARG;
  if (i % 8 != 0 || !aligned16(gate_up) || !aligned16(out)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (nvfp4_status s = check_arch()) return s;
  if (m == 0) return NVFP4_OK;
  return from_cuda(launch_silu_mul_bf16(gate_up, m, i, out, (cudaStream_t)stream));
}

}  // extern "C"

namespace {

nvfp4_status gemm_impl(const uint8_t *a_fp4, const uint8_t *a_sf, const float *a_row_scale,
                       const uint8_t *b_fp4, const uint8_t *b_sf, const float *alpha, uint16_t *d,
                       int64_t m, int64_t n, int64_t k, void *workspace, size_t ws_bytes,
                       nvfp4_algo algo, nvfp4_stream_t stream) {
  if (!a_fp4 || !a_sf || !b_fp4 || !b_sf || !alpha || !d) return NVFP4_ERR_INVALID_ARG;
  if (nvfp4_status s = check_gemm_shape(m, n, k)) return s;
  if (!aligned16(a_fp4) || !aligned16(a_sf) || !aligned16(b_fp4) || !aligned16(b_sf) || !aligned16(d))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (algo < NVFP4_ALGO_AUTO || algo > NVFP4_ALGO_TC_1SM) return NVFP4_ERR_INVALID_ARG;
  if (nvfp4_status s = check_arch()) return s;
  if (m == 0) return NVFP4_OK;
  const cudaStream_t st = (cudaStream_t)stream;
  if (algo == NVFP4_ALGO_AUTO) algo = pick_algo(TC_W4A4, m, n, k);
  if (algo == NVFP4_ALGO_GEMV)
    return from_cuda(launch_gemv(GEMV_W4A4, a_fp4, a_sf, b_fp4, b_sf, alpha, nullptr, d, nullptr,
                                 nullptr, m, n, k, st, a_row_scale));
  if (algo == NVFP4_ALGO_TC_SWAPAB) {
    if (!swapab_supported(TC_W4A4, m, n, k)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    return from_cuda(launch_swapab(TC_W4A4, a_fp4, a_sf, b_fp4, b_sf, alpha, nullptr, d, nullptr,
                                   nullptr, m, n, k, workspace, ws_bytes, g_wait_limit.load(), st,
                                   a_row_scale));
  }
  if (!tc_supported(TC_W4A4, m, n, k)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  return from_cuda(launch_tc(TC_W4A4, algo == NVFP4_ALGO_TC, a_fp4, a_sf, b_fp4, b_sf, alpha, nullptr, d, nullptr,
                             nullptr, m, n, k, g_wait_limit.load(), st, a_row_scale));
}

nvfp4_status swiglu_impl(const uint8_t *a_fp4, const uint8_t *a_sf, const float *a_row_scale,
                         const uint8_t *w_int_fp4, const uint8_t *w_int_sf, const float *alpha,
                         const float *out_global_scale, uint8_t *out_fp4, uint8_t *out_sf, int64_t m,
                         int64_t n, int64_t k, void *workspace, size_t ws_bytes, nvfp4_algo algo,
                         nvfp4_stream_t stream) {
  if (!a_fp4 || !a_sf || !w_int_fp4 || !w_int_sf || !alpha || !out_global_scale || !out_fp4 || !out_sf)
    return NVFP4_ERR_INVALID_ARG;
  if (nvfp4_status s = check_gemm_shape(m, n, k)) return s;
  if (n % 128 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(a_fp4) || !aligned16(a_sf) || !aligned16(w_int_fp4) || !aligned16(w_int_sf) ||
      !aligned16(out_fp4) || !aligned16(out_sf))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (algo < NVFP4_ALGO_AUTO || algo > NVFP4_ALGO_TC_1SM) return NVFP4_ERR_INVALID_ARG;
  if (nvfp4_status s = check_arch()) return s;
  if (m == 0) return NVFP4_OK;
  const cudaStream_t st = (cudaStream_t)stream;
  if (algo == NVFP4_ALGO_AUTO) algo = pick_algo(TC_W4A4_SWIGLU, m, n, k);
  if (algo == NVFP4_ALGO_GEMV)
    return from_cuda(launch_gemv(GEMV_W4A4_SWIGLU, a_fp4, a_sf, w_int_fp4, w_int_sf, alpha,
                                 out_global_scale, nullptr, out_fp4, out_sf, m, n, k, st, a_row_scale));
  if (algo == NVFP4_ALGO_TC_SWAPAB) {
    if (!swapab_supported(TC_W4A4_SWIGLU, m, n, k)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
    return from_cuda(launch_swapab(TC_W4A4_SWIGLU, a_fp4, a_sf, w_int_fp4, w_int_sf, alpha,
                                   out_global_scale, nullptr, out_fp4, out_sf, m, n, k, workspace,
                                   ws_bytes, g_wait_limit.load(), st, a_row_scale));
  }
  if (!tc_supported(TC_W4A4_SWIGLU, m, n, k)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  return from_cuda(launch_tc(TC_W4A4_SWIGLU, algo == NVFP4_ALGO_TC, a_fp4, a_sf, w_int_fp4, w_int_sf, alpha,
                             out_global_scale, nullptr, out_fp4, out_sf, m, n, k, g_wait_limit.load(),
                             st, a_row_scale));
}

}  // namespace

extern "C" {

nvfp4_status nvfp4_gemm_ex(const uint8_t *a_fp4, const uint8_t *a_sf, const uint8_t *b_fp4,
                           const uint8_t *b_sf, const float *alpha, uint16_t *d, int64_t m,
                           int64_t n, int64_t k, void *workspace, size_t ws_bytes, nvfp4_algo algo,
                           nvfp4_stream_t stream) {
  return gemm_impl(a_fp4, a_sf, nullptr, b_fp4, b_sf, alpha, d, m, n, k, workspace, ws_bytes, algo, stream);
}

nvfp4_status nvfp4_gemm_per_token(const uint8_t *a_fp4, const uint8_t *a_sf, const float *a_row_scale,
                                  const uint8_t *b_fp4, const uint8_t *b_sf, const float *alpha,
                                  uint16_t *d, int64_t m, int64_t n, int64_t k, void *workspace,
                                  size_t ws_bytes, nvfp4_algo algo, nvfp4_stream_t stream) {
  if (!a_row_scale) return NVFP4_ERR_INVALID_ARG;
  return gemm_impl(a_fp4, a_sf, a_row_scale, b_fp4, b_sf, alpha, d, m, n, k, workspace, ws_bytes, algo,
                   stream);
}

nvfp4_status nvfp4_gemm_swiglu_quant_per_token(const uint8_t *a_fp4, const uint8_t *a_sf,
                                               const float *a_row_scale, const uint8_t *w_int_fp4,
                                               const uint8_t *w_int_sf, const float *alpha,
                                               const float *out_global_scale, uint8_t *out_fp4,
                                               uint8_t *out_sf, int64_t m, int64_t n, int64_t k,
                                               void *workspace, size_t ws_bytes, nvfp4_algo algo,
                                               nvfp4_stream_t stream) {
  if (!a_row_scale) return NVFP4_ERR_INVALID_ARG;
  return swiglu_impl(a_fp4, a_sf, a_row_scale, w_int_fp4, w_int_sf, alpha, out_global_scale, out_fp4,
                     out_sf, m, n, k, workspace, ws_bytes, algo, stream);
}

nvfp4_status nvfp4_quantize_per_token(const uint16_t *x, int64_t m, int64_t k, uint8_t *out_fp4,
                                      uint8_t *out_sf, nvfp4_sf_layout sf_layout, float *out_row_scale,
                                      nvfp4_stream_t stream) {
  if (!x || !out_fp4 || !out_sf || !out_row_scale || m < 0 || k <= 0) return NVFP4_ERR_INVALID_ARG;
  if (sf_layout != NVFP4_SF_LINEAR && sf_layout != NVFP4_SF_SWIZZLED_128x4) return NVFP4_ERR_INVALID_ARG;
  if (k % 16 != 0 || !aligned16(x) || !aligned16(out_fp4) || m >= (int64_t(1) << 31))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (nvfp4_status s = check_arch()) return s;
  if (m == 0) return NVFP4_OK;
  return from_cuda(launch_quantize_per_token(x, m, k, out_fp4, out_sf, sf_layout == NVFP4_SF_SWIZZLED_128x4,
                                             out_row_scale, (cudaStream_t)stream));
}

nvfp4_status nvfp4_gemm(const uint8_t *a_fp4, const uint8_t *a_sf, const uint8_t *b_fp4,
                        const uint8_t *b_sf, const float *alpha, uint16_t *d, int64_t m, int64_t n,
                        int64_t k, void *workspace, size_t ws_bytes, nvfp4_stream_t stream) {
  return nvfp4_gemm_ex(a_fp4, a_sf, b_fp4, b_sf, alpha, d, m, n, k, workspace, ws_bytes,
                       NVFP4_ALGO_AUTO, stream);
}

nvfp4_status nvfp4_gemm_swiglu_quant_ex(const uint8_t *a_fp4, const uint8_t *a_sf,
                                        const uint8_t *w_int_fp4, const uint8_t *w_int_sf,
                                        const float *alpha, const float *out_global_scale,
                                        uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n,
                                        int64_t k, void *workspace, size_t ws_bytes, nvfp4_algo algo,
                                        nvfp4_stream_t stream) {
  return swiglu_impl(a_fp4, a_sf, nullptr, w_int_fp4, w_int_sf, alpha, out_global_scale, out_fp4, out_sf, m, n,
                     k, workspace, ws_bytes, algo, stream);
}

nvfp4_status nvfp4_gemm_swiglu_quant(const uint8_t *a_fp4, const uint8_t *a_sf,
                                     const uint8_t *w_int_fp4, const uint8_t *w_int_sf,
                                     const float *alpha, const float *out_global_scale,
                                     uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n,
                                     int64_t k, void *workspace, size_t ws_bytes,
                                     nvfp4_stream_t stream) {
  return nvfp4_gemm_swiglu_quant_ex(a_fp4, a_sf, w_int_fp4, w_int_sf, alpha, out_global_scale,
                                    out_fp4, out_sf, m, n, k, workspace, ws_bytes,
                                    NVFP4_ALGO_AUTO, stream);
}

size_t nvfp4_quantize_gemm_swiglu_quant_workspace_bytes(int64_t m, int64_t n, int64_t k) {
  if (m <= 0 || n <= 0 || k <= 0) return 0;
  if (m <= 64 && swapab_supported(TC_W4A4_SWIGLU, m, n, k)) return swapab_fold_workspace_bytes(m, n, k);
  return nvfp4_workspace_bytes(m, n, k, NVFP4_ALGO_AUTO);
}

nvfp4_status nvfp4_quantize_gemm_swiglu_quant(const uint16_t *x, const float *x_global_scale, uint8_t *x_fp4,
                                              uint8_t *x_sf, const uint8_t *w_int_fp4, const uint8_t *w_int_sf,
                                              const float *alpha, const float *out_global_scale,
                                              uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n,
                                              int64_t k, void *workspace, size_t ws_bytes,
                                              nvfp4_stream_t stream) {
  if (!x || !x_global_scale || !x_fp4 || !x_sf || !w_int_fp4 || !w_int_sf || !alpha || !out_global_scale ||
      !out_fp4 || !out_sf)
    return NVFP4_ERR_INVALID_ARG;
  if (nvfp4_status s = check_gemm_shape(m, n, k)) return s;
  if (n % 128 != 0) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!aligned16(x) || !aligned16(x_fp4) || !aligned16(x_sf) || !aligned16(w_int_fp4) || !aligned16(w_int_sf) ||
      !aligned16(out_fp4) || !aligned16(out_sf))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (nvfp4_status s = check_arch()) return s;
  if (m == 0) return NVFP4_OK;
  const cudaStream_t st = (cudaStream_t)stream;
  if (m <= 64 && swapab_supported(TC_W4A4_SWIGLU, m, n, k) && workspace && aligned16(workspace) &&
      ws_bytes >= swapab_fold_workspace_bytes(m, n, k))
    return from_cuda(launch_swapab_quantize_fold(x, x_global_scale, x_fp4, x_sf, w_int_fp4, w_int_sf, alpha,
                                                 out_global_scale, out_fp4, out_sf, m, n, k, workspace, ws_bytes,
                                                 g_wait_limit.load(), st));
  // otherwise the two launches it stands for
  if (nvfp4_status s = nvfp4_quantize(x, m, k, x_global_scale, x_fp4, x_sf, NVFP4_SF_SWIZZLED_128x4, stream))
    return s;
  return nvfp4_gemm_swiglu_quant_ex(x_fp4, x_sf, w_int_fp4, w_int_sf, alpha, out_global_scale, out_fp4, out_sf,
                                    m, n, k, workspace, ws_bytes, NVFP4_ALGO_AUTO, stream);
}

}  // extern "C"

namespace {
size_t round256(size_t b) { return (b + 255) / 256 * 256; }

nvfp4_status w4a16_impl(const uint16_t *a, const uint16_t *pre_scale, const uint8_t *b_fp4, const uint8_t *b_sf,
                        const float *alpha, uint16_t *d, int64_t m, int64_t n, int64_t k, void *workspace,
                        size_t ws_bytes, nvfp4_algo algo, nvfp4_stream_t stream) {
  if (!a || !b_fp4 || !b_sf || !alpha || !d) return NVFP4_ERR_INVALID_ARG;
  if (nvfp4_status s = check_gemm_shape(m, n, k)) return s;
  if (!aligned16(a) || !aligned16(b_fp4) || !aligned16(b_sf) || !aligned16(d))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (pre_scale && !aligned16(pre_scale)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (algo < NVFP4_ALGO_AUTO || algo > NVFP4_ALGO_TC_1SM) return NVFP4_ERR_INVALID_ARG;
  if (nvfp4_status s = check_arch()) return s;
  if (m == 0) return NVFP4_OK;
  const cudaStream_t st = (cudaStream_t)stream;
  // The W4A16 tensor-core kernel always has the weight as the MMA's 128-row
  // operand and one CTA per weight tile, so NVFP4_ALGO_TC, NVFP4_ALGO_TC_SWAPAB
  // and NVFP4_ALGO_TC_1SM name the same kernel.
  if (algo == NVFP4_ALGO_AUTO)
    algo = w4a16_tc_supported(m, n, k) ? NVFP4_ALGO_TC : NVFP4_ALGO_GEMV;
  if (algo == NVFP4_ALGO_GEMV)
    return from_cuda(launch_gemv(GEMV_W4A16, a, nullptr, b_fp4, b_sf, alpha, nullptr, d, nullptr,
                                 nullptr, m, n, k, st, nullptr, pre_scale));
  if (!w4a16_tc_supported(m, n, k)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (workspace && !aligned16(workspace)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (pre_scale) {
    // Every weight tile reads the same activations: they are scaled once,
    // in a pass of their own -- by the TMEM kernel's f16 pre-pass, or else
    // into the front of the workspace by bf16_awq_prescale (the shared-memory
    // kernel's converter warps are its critical path).
    const size_t xs_bytes = round256((size_t)(m * k * 2));
    if (!workspace || ws_bytes < xs_bytes) return NVFP4_ERR_INVALID_ARG;
    uint16_t *xs = static_cast<uint16_t *>(workspace);
    workspace = static_cast<uint8_t *>(workspace) + xs_bytes;
    ws_bytes -= xs_bytes;
    if (!w4a16_uses_tmem(m, n, k, ws_bytes ? workspace : nullptr, ws_bytes)) {
      if (cudaError_t e = launch_awq_prescale(a, pre_scale, m, k, xs, st)) return from_cuda(e);
      a = xs;
      pre_scale = nullptr;
    }
  }
  if (ws_bytes == 0) workspace = nullptr;
  return from_cuda(launch_w4a16_tc(a, pre_scale, b_fp4, b_sf, alpha, d, m, n, k, workspace, ws_bytes,
                                   g_wait_limit.load(), st));
}
}  // namespace

extern "C" {

nvfp4_status bf16_fp4_gemm_ex(const uint16_t *a, const uint8_t *b_fp4, const uint8_t *b_sf,
                              const float *alpha, uint16_t *d, int64_t m, int64_t n, int64_t k,
                              void *workspace, size_t ws_bytes, nvfp4_algo algo, nvfp4_stream_t stream) {
  return w4a16_impl(a, nullptr, b_fp4, b_sf, alpha, d, m, n, k, workspace, ws_bytes, algo, stream);
}

size_t bf16_fp4_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, nvfp4_algo algo) {
  if (m <= 0 || n <= 0 || k <= 0 || algo == NVFP4_ALGO_GEMV) return 0;
  return w4a16_workspace_bytes(m, n, k);
}

nvfp4_status bf16_fp4_gemm_prescaled(const uint16_t *a, const uint16_t *pre_quant_scale,
                                     const uint8_t *b_fp4, const uint8_t *b_sf, const float *alpha,
                                     uint16_t *d, int64_t m, int64_t n, int64_t k, void *workspace,
                                     size_t ws_bytes, nvfp4_algo algo, nvfp4_stream_t stream) {
  if (!pre_quant_scale) return NVFP4_ERR_INVALID_ARG;
  return w4a16_impl(a, pre_quant_scale, b_fp4, b_sf, alpha, d, m, n, k, workspace, ws_bytes, algo, stream);
}

size_t bf16_fp4_gemm_prescaled_workspace_bytes(int64_t m, int64_t n, int64_t k, nvfp4_algo algo) {
  if (m <= 0 || n <= 0 || k <= 0 || algo == NVFP4_ALGO_GEMV) return 0;
  if (m > (int64_t(1) << 31) || k > (int64_t(1) << 31)) return 0;
  if (algo == NVFP4_ALGO_AUTO && !w4a16_tc_supported(m, n, k)) return 0;
  return round256((size_t)(m * k * 2)) + w4a16_workspace_bytes(m, n, k);
}

nvfp4_status nvfp4_mlp_decode(const uint16_t *x, const float *x_global_scale, const uint8_t *w_gate_up_int,
                              const uint8_t *w_gate_up_int_sf, const float *alpha_gate_up,
                              const float *h_global_scale, const uint8_t *w_down, const uint8_t *w_down_sf,
                              const float *alpha_down, uint8_t *x_fp4, uint8_t *x_sf, uint8_t *h_fp4,
                              uint8_t *h_sf, uint16_t *out, int64_t m, int64_t hidden, int64_t inter,
                              int round_gate_up_bf16, void *workspace, size_t ws_bytes,
                              nvfp4_stream_t stream) {
  if (!x || !x_global_scale || !w_gate_up_int || !w_gate_up_int_sf || !alpha_gate_up || !h_global_scale ||
      !w_down || !w_down_sf || !alpha_down || !x_fp4 || !x_sf || !h_fp4 || !h_sf || !out)
    return NVFP4_ERR_INVALID_ARG;
  if (m < 0 || hidden <= 0 || inter <= 0) return NVFP4_ERR_INVALID_ARG;
  if (m == 0) return NVFP4_OK;
  if (!mlp_decode_supported(m, hidden, inter)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  const void *ptrs[] = {x, w_gate_up_int, w_gate_up_int_sf, w_down, w_down_sf, x_fp4, x_sf, h_fp4, h_sf, out};
  for (const void *q : ptrs)
    if (!aligned16(q)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (!workspace || ws_bytes < mlp_decode_workspace_bytes(m, hidden, inter)) return NVFP4_ERR_INVALID_ARG;
  if (!aligned16(workspace)) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (nvfp4_status s = check_arch()) return s;
  MlpDecodeParams q{};
  q.x = x;
  q.gs_x = x_global_scale;
  q.w_gu = w_gate_up_int;
  q.w_gu_sf = w_gate_up_int_sf;
  q.alpha_gu = alpha_gate_up;
  q.gs_h = h_global_scale;
  q.w_dn = w_down;
  q.w_dn_sf = w_down_sf;
  q.alpha_dn = alpha_down;
  q.x_fp4 = x_fp4;
  q.x_sf = x_sf;
  q.h_fp4 = h_fp4;
  q.h_sf = h_sf;
  q.out = out;
  q.m = m;
  q.hidden = hidden;
  q.inter = inter;
  q.round_bf16 = round_gate_up_bf16 != 0;
  q.workspace = workspace;
  q.ws_bytes = ws_bytes;
  q.wait_limit = g_wait_limit.load();
  const cudaError_t e = launch_mlp_decode(q, (cudaStream_t)stream);
  // the device cannot hold every CTA at once (they wait on each other)
  if (e == cudaErrorCooperativeLaunchTooLarge) return NVFP4_ERR_UNSUPPORTED_SHAPE;
  return from_cuda(e);
}

size_t nvfp4_mlp_decode_workspace_bytes(int64_t m, int64_t hidden, int64_t inter) {
  return mlp_decode_workspace_bytes(m, hidden, inter);
}

nvfp4_status bf16_awq_prescale(const uint16_t *x, const uint16_t *pre_quant_scale, uint16_t *out, int64_t m,
                               int64_t k, nvfp4_stream_t stream) {
  if (!x || !pre_quant_scale || !out || m < 0 || k <= 0) return NVFP4_ERR_INVALID_ARG;
  if (k % 8 != 0 || !aligned16(x) || !aligned16(pre_quant_scale) || !aligned16(out))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (nvfp4_status s = check_arch()) return s;
  if (m == 0) return NVFP4_OK;
  return from_cuda(launch_awq_prescale(x, pre_quant_scale, m, k, out, (cudaStream_t)stream));
}

nvfp4_status bf16_fp4_gemm(const uint16_t *a, const uint8_t *b_fp4, const uint8_t *b_sf,
                           const float *alpha, uint16_t *d, int64_t m, int64_t n, int64_t k,
                           void *workspace, size_t ws_bytes, nvfp4_stream_t stream) {
  return bf16_fp4_gemm_ex(a, b_fp4, b_sf, alpha, d, m, n, k, workspace, ws_bytes, NVFP4_ALGO_AUTO,
                          stream);
}

nvfp4_status nvfp4_prepare_weights(const uint8_t *w_fp4, const uint8_t *sf_linear, int64_t n,
                                   int64_t k, uint8_t *w_out, uint8_t *sf_out,
                                   nvfp4_stream_t stream) {
  if (!w_fp4 || !sf_linear || !w_out || !sf_out || n <= 0 || k <= 0) return NVFP4_ERR_INVALID_ARG;
  if (k % 16 != 0 || !aligned16(w_fp4) || !aligned16(w_out) || !aligned16(sf_out))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (nvfp4_status s = check_arch()) return s;
  return from_cuda(launch_prepare(w_fp4, sf_linear, n, k, w_out, sf_out, false,
                                  (cudaStream_t)stream));
}

nvfp4_status nvfp4_prepare_gate_up_interleaved(const uint8_t *w_fp4, const uint8_t *sf_linear,
                                               int64_t n, int64_t k, uint8_t *w_out,
                                               uint8_t *sf_out, nvfp4_stream_t stream) {
  if (!w_fp4 || !sf_linear || !w_out || !sf_out || n <= 0 || k <= 0) return NVFP4_ERR_INVALID_ARG;
  if (w_out == w_fp4) return NVFP4_ERR_INVALID_ARG;
  if (n % 128 != 0 || k % 16 != 0 || !aligned16(w_fp4) || !aligned16(w_out) || !aligned16(sf_out))
    return NVFP4_ERR_UNSUPPORTED_SHAPE;
  if (nvfp4_status s = check_arch()) return s;
  return from_cuda(launch_prepare(w_fp4, sf_linear, n, k, w_out, sf_out, true,
                                  (cudaStream_t)stream));
}

nvfp4_status nvfp4_get_device_status(int *status_out, nvfp4_stream_t stream) {
  if (!status_out) return NVFP4_ERR_INVALID_ARG;
  if (nvfp4_status s = check_arch()) return s;
  int v = 0;
  if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return NVFP4_ERR_CUDA;
  if (read_and_clear_device_status(&v) != cudaSuccess) return NVFP4_ERR_CUDA;
  *status_out = v;
  return NVFP4_OK;
}

nvfp4_status nvfp4_set_wait_limit(uint32_t spins) {
  g_wait_limit.store(spins);
  return NVFP4_OK;
}

}  // extern "C"
