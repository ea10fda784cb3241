// Launchers shared between the C-ABI translation unit and the kernel units.
// Arguments are validated by the caller (api.cu) before any launcher runs.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "nvfp4mlp.h"

namespace nvfp4 {

// Launch with programmatic stream serialization (see pdl_wait in common.cuh).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Runs `set()` (a per-context setting such as a kernel's dynamic shared-memory
// limit) once on each device, with that device current; two host threads
// racing on the first call may both run it, which is harmless for settings.
struct PerDeviceOnce {
  std::atomic<uint8_t> done[64] = {};
  template <class F>
  cudaError_t run(F set) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (done[dev].load(std::memory_order_acquire)) return cudaSuccess;
    const cudaError_t e = set();
    if (e == cudaSuccess) done[dev].store(1, std::memory_order_release);
    return e;
  }
};

// Every split-K workspace starts with a fixed area of arrival counters (and
// other words that must start at zero); a kernel's fp32 partials follow it.
// Calls of different shapes may share one workspace in stream order: their
// counters all live in this area, which no kernel's partials overlap, and
// every complete call leaves them at zero.  A kernel that would need more
// counter slots than the area holds does not split.
constexpr size_t kCounterArea = 64 * 1024;
constexpr int64_t kCounterSlots = (int64_t)(kCounterArea / 4);

// Poll limit of the kernels' bounded waits set through nvfp4_set_wait_limit
// (0 = the kernels' wall-clock default).
uint32_t wait_limit();

cudaError_t launch_quantize(const uint16_t *x, int64_t m, int64_t k, const float *gs,
                            uint8_t *out_fp4, uint8_t *out_sf, bool swizzled, cudaStream_t st);
cudaError_t launch_quantize_per_token(const uint16_t *x, int64_t m, int64_t k, uint8_t *out_fp4,
                                      uint8_t *out_sf, bool swizzled, float *row_scale, cudaStream_t st);
cudaError_t launch_silu_mul_quantize(const uint16_t *gate_up, int64_t m, int64_t i, const float *gs,
                                     uint8_t *out_fp4, uint8_t *out_sf, cudaStream_t st);
cudaError_t launch_silu_mul_quantize_masked(const uint16_t *gate_up, const int32_t *masked_m, int64_t g,
                                            int64_t m_max, int64_t i, const float *gs, uint8_t *out_fp4,
                                            uint8_t *out_sf, cudaStream_t st);
cudaError_t launch_silu_mul_bf16(const uint16_t *gate_up, int64_t m, int64_t i, uint16_t *out,
                                 cudaStream_t st);
// out [m, k] = bf16(x * s[k]) (AWQ pre-scale); k % 8 == 0, 16-byte aligned.
cudaError_t launch_awq_prescale(const uint16_t *x, const uint16_t *s, int64_t m, int64_t k, uint16_t *out,
                                cudaStream_t st);
cudaError_t launch_prepare(const uint8_t *w, const uint8_t *sf_lin, int64_t n, int64_t k,
                           uint8_t *w_out, uint8_t *sf_out, bool interleave, cudaStream_t st);

// CUDA-core GEMV family (any M; meant for decode-sized M).
enum GemvMode { GEMV_W4A4 = 0, GEMV_W4A4_SWIGLU = 1, GEMV_W4A16 = 2 };
// a_row_scale (optional, fp32 [m]): per-row activation dequant factor that
// multiplies alpha (per-token activation scales); nullptr for none.
// pre_scale (optional, GEMV_W4A16 only, bf16 [k]): AWQ per-channel activation
// scale, the product rounded to bf16 before it meets the weight.
cudaError_t launch_gemv(GemvMode mode, const void *a, const uint8_t *a_sf, const uint8_t *b,
                        const uint8_t *b_sf, const float *alpha, const float *out_gs, uint16_t *d,
                        uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n, int64_t k,
                        cudaStream_t st, const float *a_row_scale = nullptr,
                        const uint16_t *pre_scale = nullptr);

// tcgen05 tensor-core family.  launch_tc: prefill-sized M, 128 x 256 output
// tiles; pair = 2-SM MMAs by CTA pairs (cta_group::2), else one CTA per tile.
enum TcMode { TC_W4A4 = 0, TC_W4A4_SWIGLU = 1, TC_W4A16 = 2 };
cudaError_t launch_tc(TcMode mode, bool pair, const void *a, const uint8_t *a_sf,
                      const uint8_t *b, const uint8_t *b_sf, const float *alpha,
                      const float *out_gs, uint16_t *d, uint8_t *out_fp4, uint8_t *out_sf,
                      int64_t m, int64_t n, int64_t k, uint32_t wait_limit, cudaStream_t st,
                      const float *a_row_scale = nullptr);
bool tc_supported(TcMode mode, int64_t m, int64_t n, int64_t k);

// Device status word of the current device (set by kernels that give up a
// bounded wait); reads it into *out and clears it.  Synchronous.
cudaError_t read_and_clear_device_status(int *out);
// Device address of that word, for kernels in any translation unit.
int *device_status_ptr();

// Host helpers shared by the tensor-core units.
int num_sms();
// 2-D TMA map over a row-major byte matrix [rows, row_bytes] (row stride
// row_bytes), box box_bytes x box_rows, swizzle_bytes-wide swizzle (128, 64,
// or 0 for none; the box's row must not be wider than the swizzle).
bool make_byte_map(CUtensorMap *tm, const void *ptr, int64_t rows, int64_t row_bytes,
                   uint32_t box_bytes, uint32_t box_rows, int swizzle_bytes);

// Decode-sized tensor-core path (weights as the MMA M operand).
size_t swapab_workspace_bytes(TcMode mode, int64_t m, int64_t n, int64_t k);
bool swapab_supported(TcMode mode, int64_t m, int64_t n, int64_t k);
cudaError_t launch_swapab(TcMode mode, const void *a, const uint8_t *a_sf, const uint8_t *b,
                          const uint8_t *b_sf, const float *alpha, const float *out_gs,
                          uint16_t *d, uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n,
                          int64_t k, void *workspace, size_t ws_bytes, uint32_t wait_limit,
                          cudaStream_t st, const float *a_row_scale = nullptr);
// The fused gate_up with the activation quantize folded in (bf16 x in; x's
// NVFP4 codes and swizzled scales written to x_fp4 / x_sf as nvfp4_quantize
// would).  Needs swapab_fold_workspace_bytes of workspace (zero-filled once;
// its counters are left at zero); cudaErrorNotSupported otherwise.
size_t swapab_fold_workspace_bytes(int64_t m, int64_t n, int64_t k);
cudaError_t launch_swapab_quantize_fold(const uint16_t *x, const float *gs_x, uint8_t *x_fp4, uint8_t *x_sf,
                                        const uint8_t *w_int, const uint8_t *w_int_sf, const float *alpha,
                                        const float *out_gs, uint8_t *out_fp4, uint8_t *out_sf, int64_t m,
                                        int64_t n, int64_t k, void *workspace, size_t ws_bytes,
                                        uint32_t wait_limit, cudaStream_t st);

// W4A16 on the tensor cores.  Given a workspace of w4a16_workspace_bytes
// (16-byte aligned, its counter area zero-filled once; counters left at
// zero), the TMEM kernel runs: weights dequantized to f16 into tensor memory
// (128-token tiles on CTA pairs), activations turned into f16 with a
// power-of-two scale per row by a pre-pass into the workspace (times the AWQ
// pre-scale when pre_scale is given), the swap-AB mixed split.  Without a
// workspace the shared-memory kernel runs (weights dequantized to bf16 in
// shared memory, whole tiles per CTA); it takes no pre_scale (the caller
// scales the activations first).
bool w4a16_tc_supported(int64_t m, int64_t n, int64_t k);
size_t w4a16_workspace_bytes(int64_t m, int64_t n, int64_t k);
// true when launch_w4a16_tc with this workspace runs the TMEM kernel
bool w4a16_uses_tmem(int64_t m, int64_t n, int64_t k, const void *ws, size_t ws_bytes);
cudaError_t launch_w4a16_tc(const uint16_t *x, const uint16_t *pre_scale, const uint8_t *w, const uint8_t *wsf,
                            const float *alpha, uint16_t *d, int64_t m, int64_t n, int64_t k, void *ws,
                            size_t ws_bytes, uint32_t wait_limit, cudaStream_t st);
// The TMEM kernel alone (gemm_w4a16_tmem.cu).
bool w4a16_tmem_supported(int64_t m, int64_t n, int64_t k);
size_t w4a16_tmem_workspace_bytes(int64_t m, int64_t n, int64_t k);
cudaError_t launch_w4a16_tmem(const uint16_t *x, const uint16_t *pre_scale, const uint8_t *w, const uint8_t *wsf,
                              const float *alpha, uint16_t *d, int64_t m, int64_t n, int64_t k, void *ws,
                              size_t ws_bytes, uint32_t wait_limit, cudaStream_t st);

// Whole decode MLP in one persistent kernel (mlp_decode.cu).
struct MlpDecodeParams {
  const uint16_t *x;                         // bf16 [m, hidden]
  const float *gs_x;                         // x global scale
  const uint8_t *w_gu, *w_gu_sf;             // interleaved gate_up weight, swizzled scales
  const float *alpha_gu, *gs_h;
  const uint8_t *w_dn, *w_dn_sf;             // down_proj weight [hidden, inter/2], swizzled scales
  const float *alpha_dn;
  uint8_t *x_fp4, *x_sf, *h_fp4, *h_sf;      // intermediates (outputs too)
  uint16_t *out;                             // bf16 [m, hidden]
  int64_t m, hidden, inter;
  bool round_bf16;
  void *workspace;
  size_t ws_bytes;
  uint32_t wait_limit;
};
bool mlp_decode_supported(int64_t m, int64_t hidden, int64_t inter);
size_t mlp_decode_workspace_bytes(int64_t m, int64_t hidden, int64_t inter);
cudaError_t launch_mlp_decode(const MlpDecodeParams &q, cudaStream_t st);

}  // namespace nvfp4
