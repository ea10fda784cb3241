/*
 * nvfp4mlp.h -- C ABI of the NVFP4-quantized dense MLP library (sm_103a).
 *
 * NVFP4: E2M1 4-bit values, two per byte (element 2j in the low nibble,
 * element 2j+1 in the high nibble), one unsigned E4M3 block scale per 16
 * consecutive elements along K, and an fp32 per-tensor global scale gs.  A
 * value dequantizes as E2M1(code) * E4M3(scale); the 1/gs factors of both
 * operands are folded into one fp32 GEMM alpha.
 *
 * Sources, cited by page title and section:
 *  [P1] sglang PR #34859 digest "Add Qwen3.8-27B": fused SiLU*mul + NVFP4
 *       quantize of the down_proj input; 6-D -> dense swizzled scale layout
 *       (section "关键源码片段", qwen2_moe.py excerpt).
 *  [P2] sglang PR #26626 digest "fused NVFP4 gate_up GEMM + SwiGLU + output
 *       quantize": fp4_quantize -> nvfp4_gemm_swiglu_nvfp4_quant -> down_proj
 *       call chain (deepseek_v2.py excerpt), gate/up interleave in groups of 64
 *       and the block-scale 2-D swizzle (modelopt_quant.py excerpt).
 *  [P3] sglang PR #35120 report "FlashInfer CuTe DSL NVFP4 W4A16 mode":
 *       fp4_gemm W4A4 / W4A16 entry (section "关键源码片段", fp4_gemm), linear
 *       [rows, K/16] scale view (MoE excerpt), W4A16 alpha holds only the weight
 *       dequant factor (section "实现拆解", item 3).
 *
 * Conventions shared by every call
 *  - Every pointer argument except status_out is a DEVICE pointer to memory
 *    the caller owns (allocated by the caller, e.g. through PyTorch).  The
 *    library never allocates, frees or logs, and holds no state between calls
 *    other than the device status word (nvfp4_get_device_status) and the
 *    fixed scratch array of nvfp4_gemm_decode_noalloc.
 *  - bf16 tensors are passed as uint16_t bit patterns, row-major, contiguous.
 *  - Scalars (global_scale, alpha, out_global_scale) are 1-element fp32
 *    DEVICE buffers, so a call sequence can be captured in a CUDA graph.
 *  - Calls are asynchronous and ordered on `stream` (NULL = legacy default
 *    stream); they do not synchronize, except nvfp4_get_device_status.
 *  - Kernels are launched with programmatic dependent launch ([P2]
 *    deepseek_v2.py excerpt passes enable_pdl=True to both fused-path kernels):
 *    a kernel may start while the previous kernel on the stream is finishing
 *    and stream its weights meanwhile, but it reads the previous kernel's
 *    results and writes any global memory only after that kernel completed,
 *    so stream order semantics are unchanged.
 *  - Pointers must be 16-byte aligned.  Outputs must not alias inputs.
 *  - Validation happens on the host before any launch; a call that returns
 *    anything but NVFP4_OK launched nothing and wrote nothing.
 *  - The device must be compute capability 10.3 (GB300, sm_103a); otherwise
 *    NVFP4_ERR_ARCH.  A failed launch returns NVFP4_ERR_CUDA.
 *  - m == 0 (no tokens) is valid and launches nothing.
 *
 * Block-scale layouts (nvfp4_sf_layout)
 *  - NVFP4_SF_LINEAR: uint8 [rows, K/16], row-major ([P3] MoE excerpt).
 *  - NVFP4_SF_SWIZZLED_128x4: the "dense swizzled layout fp4_gemm expects"
 *    ([P1] qwen2_moe.py excerpt, the permute of a (32, 4, m_blocks, 4, K/64)
 *    tensor).  Rows pad to Rp = ceil(rows/128)*128 and scale columns to
 *    Cp = ceil(K/16 / 4)*4; the scale of (row r, column j) sits at byte
 *        ((((r/128)*(Cp/4) + j/4)*32 + r%32)*4 + (r%128)/32)*4 + j%4
 *    i.e. 512-byte tiles of 128 rows x 4 columns, tiles ordered row block
 *    major.  Padding bytes are written as 0x00 by every producer here.
 *    Every GEMM operand scale is in this layout.
 */
#ifndef NVFP4MLP_H
#define NVFP4MLP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t. */
typedef struct CUstream_st *nvfp4_stream_t;

typedef enum {
  NVFP4_OK = 0,
  NVFP4_ERR_INVALID_ARG = 1,       /* null pointer, negative size, aliasing   */
  NVFP4_ERR_UNSUPPORTED_SHAPE = 2, /* size / alignment outside the supported set */
  NVFP4_ERR_ARCH = 3,              /* current device is not sm_103           */
  NVFP4_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed   */
  NVFP4_ERR_DEVICE_TIMEOUT = 5     /* a kernel gave up a bounded wait        */
} nvfp4_status;

typedef enum {
  NVFP4_SF_SWIZZLED_128x4 = 0,
  NVFP4_SF_LINEAR = 1
} nvfp4_sf_layout;

/* Kernel family selection for the GEMM entry points' *_ex forms.  AUTO picks
 * by M: the weight-streaming small-M kernels for decode-sized M, the
 * tcgen05 tensor-core kernels above that. */
typedef enum {
  NVFP4_ALGO_AUTO = 0,
  NVFP4_ALGO_GEMV = 1,      /* CUDA-core split-row GEMV (any M, meant for M <= 16)  */
  NVFP4_ALGO_TC = 2,        /* tcgen05 block-scaled MMA, accumulators in TMEM: CTA
                               pairs issuing 2-SM MMAs (256 x 256 per pair)        */
  NVFP4_ALGO_TC_SWAPAB = 3, /* tcgen05 with weights as the MMA M operand (small M)  */
  NVFP4_ALGO_TC_1SM = 4     /* as NVFP4_ALGO_TC with one CTA per 128 x 256 tile    */
} nvfp4_algo;

/* Human-readable name of a status code (static storage). */
const char *nvfp4_status_string(nvfp4_status s);

/* Library ABI version: (major << 16) | minor. */
int nvfp4_version(void);

/* Bytes of a block-scale buffer for `rows` rows of K elements (K % 16 == 0):
 * SWIZZLED_128x4 -> ceil(rows/128)*128 * ceil(K/64)*4; LINEAR -> rows*K/16.
 * Returns 0 for invalid arguments. */
size_t nvfp4_sf_bytes(int64_t rows, int64_t k, nvfp4_sf_layout layout);

/* Scratch bytes the GEMM entry points want for (m, n, k) with `algo` (AUTO
 * resolves as the GEMM would).  Non-zero only for the weight-streaming
 * tensor-core kernel (NVFP4_ALGO_TC_SWAPAB, AUTO for m <= 64) when it splits K
 * across CTAs: a fixed 64 KiB area of arrival counters followed by fp32
 * partial tiles.  Every workspace of this library (this one, the W4A16
 * GEMM's, nvfp4_mlp_decode's) has that layout, so calls of different shapes
 * and entry points may share one buffer sized for the largest of them.  The
 * workspace must be zero-filled once before its first use; every complete
 * call leaves the counters at zero again, so one buffer serves a whole
 * sequence of calls on one stream (not concurrent calls).  After a call
 * that reported NVFP4_ERR_DEVICE_TIMEOUT, zero it again.  A smaller or NULL
 * workspace is not an error: the kernel then runs one CTA per weight tile
 * without splitting K. */
size_t nvfp4_workspace_bytes(int64_t m, int64_t n, int64_t k, nvfp4_algo algo);

/* NVFP4 quantize of bf16 activations ([P2] deepseek_v2.py excerpt:
 * fp4_quantize(x, input_scale_inv); [P3] MoE excerpt for the linear layout).
 *   x            bf16 [m, k] row-major
 *   global_scale fp32 [1]  gs (e.g. 448*6/amax(x), static per tensor)
 *   out_fp4      uint8 [m, k/2]
 *   out_sf       uint8, nvfp4_sf_bytes(m, k, sf_layout) bytes (padding -> 0)
 * Per 16-block, in fp32 with IEEE round-to-nearest-even at each step:
 *   s = fp32(amax/6) * gs;  SF = E4M3(s) (RNE, saturating at 448);
 *   r = SF == 0 ? 0 : gs / SF;  code_i = E2M1(x_i * r) (RNE, saturating at 6,
 *   sign bit kept, so a negative value that rounds to zero is -0).
 * Requires k > 0, k % 16 == 0. */
nvfp4_status nvfp4_quantize(const uint16_t *x, int64_t m, int64_t k, const float *global_scale,
                            uint8_t *out_fp4, uint8_t *out_sf, nvfp4_sf_layout sf_layout,
                            nvfp4_stream_t stream);

/* Fused SiLU * mul + NVFP4 quantize of the down_proj input ([P1]
 * qwen2_moe.py excerpt: one kernel replaces act_fn + FP4 quantize).
 *   gate_up      bf16 [m, 2*i]: columns [0, i) gate, [i, 2i) up
 *   global_scale fp32 [1]: the down_proj input global scale
 *   out_fp4      uint8 [m, i/2];  out_sf: swizzled, nvfp4_sf_bytes(m, i, SWIZZLED)
 * h = fp32(silu(gate) * up), silu(g) = g / (1 + exp(-g)), h is not rounded
 * to bf16, then quantized exactly as nvfp4_quantize.  Requires i % 16 == 0. */
nvfp4_status silu_mul_nvfp4_quantize(const uint16_t *gate_up, int64_t m, int64_t i,
                                     const float *global_scale, uint8_t *out_fp4, uint8_t *out_sf,
                                     nvfp4_stream_t stream);

/* Masked multi-group form of silu_mul_nvfp4_quantize: the call the pages
 * make ([P1] qwen2_moe.py excerpt: silu_and_mul_scaled_nvfp4_experts_quantize
 * (gate_up[G, M, 2I], masked_m, scale), whose scale comes back as a 6-D
 * expert-grouped tensor that is permuted to the dense swizzled layout).
 *   gate_up      bf16 [g, m_max, 2*i]: per row [gate | up]
 *   masked_m     int32 [g] DEVICE: valid rows of each group (clamped to
 *                [0, m_max]); rows past it are not computed
 *   global_scale fp32 [1]: one global scale for every group
 *   out_fp4      uint8 [g, m_max, i/2]; invalid rows are left untouched
 *   out_sf       g consecutive blocks of nvfp4_sf_bytes(m_max, i, SWIZZLED)
 *                bytes: group e's scales in the dense swizzled layout over its
 *                m_max rows (the pages' permuted view, expert by expert);
 *                invalid and padding rows get 0x00.
 * Per valid row the arithmetic is exactly silu_mul_nvfp4_quantize.
 * Requires i % 16 == 0, g <= 65535. */
nvfp4_status silu_mul_nvfp4_quantize_masked(const uint16_t *gate_up, const int32_t *masked_m, int64_t g,
                                            int64_t m_max, int64_t i, const float *global_scale,
                                            uint8_t *out_fp4, uint8_t *out_sf, nvfp4_stream_t stream);

/* Unfused activation of the W4A16 chain: out = bf16(silu(gate) * up).
 *   gate_up bf16 [m, 2*i] ([gate | up]);  out bf16 [m, i].  Requires i % 8 == 0. */
nvfp4_status silu_mul_bf16(const uint16_t *gate_up, int64_t m, int64_t i, uint16_t *out,
                           nvfp4_stream_t stream);

/* W4A4 NVFP4 GEMM ([P3] fp4_gemm, quant_mode "w4a4"):
 *   d[m, n] = bf16( alpha * sum_k (E2M1(a)*SF_a)[m, k] * (E2M1(b)*SF_b)[n, k] )
 *   a_fp4 uint8 [m, k/2], a_sf swizzled over m rows (e.g. from nvfp4_quantize)
 *   b_fp4 uint8 [n, k/2], b_sf swizzled over n rows (nvfp4_prepare_weights)
 *   alpha fp32 [1] = 1 / (gs_a * gs_b);  d bf16 [m, n] row-major.
 * fp32 accumulation; d is rounded to nearest even.
 * Requires k % 64 == 0, n % 32 == 0.  workspace may be NULL when
 * nvfp4_workspace_bytes() is 0. */
nvfp4_status nvfp4_gemm(const uint8_t *a_fp4, const uint8_t *a_sf, const uint8_t *b_fp4,
                        const uint8_t *b_sf, const float *alpha, uint16_t *d, int64_t m, int64_t n,
                        int64_t k, void *workspace, size_t ws_bytes, nvfp4_stream_t stream);
nvfp4_status nvfp4_gemm_ex(const uint8_t *a_fp4, const uint8_t *a_sf, const uint8_t *b_fp4,
                           const uint8_t *b_sf, const float *alpha, uint16_t *d, int64_t m,
                           int64_t n, int64_t k, void *workspace, size_t ws_bytes,
                           nvfp4_algo algo, nvfp4_stream_t stream);

/* Fused gate_up GEMM + SwiGLU + NVFP4 requantize ([P2] "实现拆解" item 1 and
 * deepseek_v2.py excerpt: nvfp4_gemm_swiglu_nvfp4_quant).
 *   a_fp4/a_sf      activation, as nvfp4_gemm
 *   w_int_fp4/_sf   gate_up weight [n = 2I, k/2] from
 *                   nvfp4_prepare_gate_up_interleaved (rows interleaved)
 *   alpha           fp32 [1] = 1/(gs_a * gs_w), one for gate and up
 *   out_global_scale fp32 [1] = down_proj input global scale
 *   out_fp4         uint8 [m, n/4]  (I/2 bytes per row)
 *   out_sf          swizzled over m rows with I/16 columns
 * g, u = alpha * acc (fp32); h = silu(g) * u in fp32 (no bf16 rounding); h is
 * quantized as nvfp4_quantize.  W4A4 only ([P3] "实现拆解" item 5: the fused
 * kernels are guarded to quant_mode "w4a4").  Requires n % 128 == 0,
 * k % 64 == 0. */
nvfp4_status nvfp4_gemm_swiglu_quant(const uint8_t *a_fp4, const uint8_t *a_sf,
                                     const uint8_t *w_int_fp4, const uint8_t *w_int_sf,
                                     const float *alpha, const float *out_global_scale,
                                     uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n,
                                     int64_t k, void *workspace, size_t ws_bytes,
                                     nvfp4_stream_t stream);
nvfp4_status nvfp4_gemm_swiglu_quant_ex(const uint8_t *a_fp4, const uint8_t *a_sf,
                                        const uint8_t *w_int_fp4, const uint8_t *w_int_sf,
                                        const float *alpha, const float *out_global_scale,
                                        uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n,
                                        int64_t k, void *workspace, size_t ws_bytes,
                                        nvfp4_algo algo, nvfp4_stream_t stream);

/* The activation quantize folded into the fused gate_up GEMM (the decode
 * chain's nvfp4_quantize -> nvfp4_gemm_swiglu_quant; [P2] deepseek_v2.py
 * excerpt: fp4_quantize and the fused kernel, both launched with enable_pdl).
 *   x bf16 [m, k], x_global_scale fp32 [1]: quantized exactly as
 *     nvfp4_quantize(x, m, k, x_global_scale, x_fp4, x_sf,
 *     NVFP4_SF_SWIZZLED_128x4), and x_fp4 uint8 [m, k/2] / x_sf are written
 *     with that result (caller-owned, as nvfp4_quantize's outputs);
 *   then out_fp4 / out_sf = nvfp4_gemm_swiglu_quant(x_fp4, x_sf, w_int_fp4,
 *     w_int_sf, alpha, out_global_scale, ...), bit for bit.
 * For m <= 64 with nvfp4_quantize_gemm_swiglu_quant_workspace_bytes() of
 * workspace (16-byte aligned, zero-filled once before its first use; the
 * call leaves its counters at zero) this is one launch: the CTAs first
 * through the grid-dependency wait quantize x in chunks that they count in
 * the workspace, and every CTA issues its activation loads once all chunks
 * are counted, so the separate quantize launch and the grid completion
 * between the two leave the decode chain.  Otherwise (larger m, or less
 * workspace) it makes the two launches.  After NVFP4_ERR_DEVICE_TIMEOUT the
 * workspace must be zero-filled again.  Requires n % 128 == 0, k % 64 == 0,
 * 16-byte aligned x, x_fp4, x_sf, weights and outputs. */
size_t nvfp4_quantize_gemm_swiglu_quant_workspace_bytes(int64_t m, int64_t n, int64_t k);
nvfp4_status nvfp4_quantize_gemm_swiglu_quant(const uint16_t *x, const float *x_global_scale,
                                              uint8_t *x_fp4, uint8_t *x_sf, const uint8_t *w_int_fp4,
                                              const uint8_t *w_int_sf, const float *alpha,
                                              const float *out_global_scale, uint8_t *out_fp4,
                                              uint8_t *out_sf, int64_t m, int64_t n, int64_t k,
                                              void *workspace, size_t ws_bytes, nvfp4_stream_t stream);

/* Per-token dynamic activation scales ([P3] MoE excerpt: nvfp4_quantize(...,
 * per_token_activation=True) returns a per-token scale).  Each row r gets its
 * own global scale gs_r = fp32(448*6 / amax(row r)) (1 for an all-zero row)
 * and is quantized exactly as nvfp4_quantize with it; out_row_scale[r] =
 * fp32(1 / gs_r) is written for the GEMM.
 *   x bf16 [m, k];  out_fp4 uint8 [m, k/2];  out_sf as nvfp4_quantize;
 *   out_row_scale fp32 [m] DEVICE.  Requires k % 16 == 0. */
nvfp4_status nvfp4_quantize_per_token(const uint16_t *x, int64_t m, int64_t k, uint8_t *out_fp4,
                                      uint8_t *out_sf, nvfp4_sf_layout sf_layout, float *out_row_scale,
                                      nvfp4_stream_t stream);

/* nvfp4_gemm_ex / nvfp4_gemm_swiglu_quant_ex for activations quantized per
 * token: every accumulator row m is multiplied by alpha * a_row_scale[m]
 * (alpha then holds only the weight factor 1/gs_w).
 *   a_row_scale fp32 [m] DEVICE, as written by nvfp4_quantize_per_token. */
nvfp4_status nvfp4_gemm_per_token(const uint8_t *a_fp4, const uint8_t *a_sf, const float *a_row_scale,
                                  const uint8_t *b_fp4, const uint8_t *b_sf, const float *alpha,
                                  uint16_t *d, int64_t m, int64_t n, int64_t k, void *workspace,
                                  size_t ws_bytes, nvfp4_algo algo, nvfp4_stream_t stream);
nvfp4_status nvfp4_gemm_swiglu_quant_per_token(const uint8_t *a_fp4, const uint8_t *a_sf,
                                               const float *a_row_scale, const uint8_t *w_int_fp4,
                                               const uint8_t *w_int_sf, const float *alpha,
                                               const float *out_global_scale, uint8_t *out_fp4,
                                               uint8_t *out_sf, int64_t m, int64_t n, int64_t k,
                                               void *workspace, size_t ws_bytes, nvfp4_algo algo,
                                               nvfp4_stream_t stream);

/* W4A16 GEMM ([P3] fp4_gemm, quant_mode "w4a16" -> mm_bf16_fp4):
 *   d[m, n] = bf16( alpha * sum_k a[m, k] * (E2M1(b)*SF_b)[n, k] )
 *   a bf16 [m, k];  b_fp4/b_sf as nvfp4_gemm;  alpha fp32 [1] = 1/gs_b only.
 *   workspace  optional DEVICE scratch (nullptr / 0 allowed): with
 *              bf16_fp4_gemm_workspace_bytes(m, n, k, algo) bytes, 16-byte
 *              aligned and its first 64 KiB (the arrival counters)
 *              zero-filled once before first use, the tensor-core path
 *              splits the work along K over all SMs -- up to 64 tokens
 *              always, above when whole 128-row weight tiles would leave SMs
 *              idle (the counters are left at zero after every complete call;
 *              calls sharing it must be stream-ordered); with less, every SM
 *              owns whole weight tiles.  The workspace also selects the
 *              TMEM kernel: the weights are dequantized to f16 in tensor
 *              memory (128-token tiles on CTA pairs) and the activations
 *              are written into the workspace by a pre-pass as f16 times a
 *              power of two 2^e per token row (e puts the row's largest
 *              finite magnitude in [2^15, 2^16); the epilogue multiplies by
 *              2^-e).  That is exact
 *              for every activation within 2^30 of its row's largest
 *              magnitude (smaller ones are rounded by at most 2^-25 * 2^-e),
 *              so the result depends on the workspace only through the
 *              order of the fp32 accumulation.
 * Requires k % 64 == 0, n % 32 == 0. */
nvfp4_status bf16_fp4_gemm(const uint16_t *a, const uint8_t *b_fp4, const uint8_t *b_sf,
                           const float *alpha, uint16_t *d, int64_t m, int64_t n, int64_t k,
                           void *workspace, size_t ws_bytes, nvfp4_stream_t stream);
nvfp4_status bf16_fp4_gemm_ex(const uint16_t *a, const uint8_t *b_fp4, const uint8_t *b_sf,
                              const float *alpha, uint16_t *d, int64_t m, int64_t n, int64_t k,
                              void *workspace, size_t ws_bytes, nvfp4_algo algo,
                              nvfp4_stream_t stream);
/* Split-K workspace bytes for bf16_fp4_gemm(_ex) (0: none needed).  Host only. */
size_t bf16_fp4_gemm_workspace_bytes(int64_t m, int64_t n, int64_t k, nvfp4_algo algo);

/* NVFP4_AWQ activation pre-scale ([P3] "实现拆解" item 2: in W4A16 mode the
 * linear layer's apply keeps the AWQ pre_quant_scale multiply of x and then
 * runs the bf16 x FP4 GEMM on the result):
 *   out[r, c] = bf16(x[r, c] * pre_quant_scale[c])
 * the exact product rounded once to bf16 (RNE), as a bf16 tensor multiply.
 *   x, out bf16 [m, k] DEVICE (out may equal x);  pre_quant_scale bf16 [k].
 * Requires k % 8 == 0 and 16-byte aligned pointers. */
nvfp4_status bf16_awq_prescale(const uint16_t *x, const uint16_t *pre_quant_scale, uint16_t *out,
                               int64_t m, int64_t k, nvfp4_stream_t stream);

/* W4A16 GEMM on AWQ-pre-scaled activations, in one call:
 *   d[m, n] = bf16( alpha * sum_k bf16(a[m, k] * s[k]) * (E2M1(b)*SF_b)[n, k] )
 *   pre_quant_scale  bf16 [k] DEVICE, 16-byte aligned (s above; nullptr is
 *                    NVFP4_ERR_INVALID_ARG, a misaligned pointer
 *                    NVFP4_ERR_UNSUPPORTED_SHAPE).
 *   workspace        DEVICE scratch, 16-byte aligned: on the tensor cores the
 *                    scaled activations take its first m*k*2 bytes (rounded
 *                    up to 256; less: NVFP4_ERR_INVALID_ARG, nothing runs),
 *                    and the rest serves as bf16_fp4_gemm's split-K
 *                    workspace (zero-filled once before first use);
 *                    bf16_fp4_gemm_prescaled_workspace_bytes gives both.
 *   Everything else as bf16_fp4_gemm_ex (same algo choices and shape rules).
 * a * s is rounded once to bf16, the activation type, as the separate
 * multiply would.  The GEMV scales each activation as it loads it (no
 * workspace).  The tensor-core path first writes the scaled activations to
 * the workspace with bf16_awq_prescale, then runs the W4A16 GEMM on them:
 * scaling inside the GEMM would lengthen its converter warps, its critical
 * path, and repeat the work for every weight tile. */
nvfp4_status bf16_fp4_gemm_prescaled(const uint16_t *a, const uint16_t *pre_quant_scale,
                                     const uint8_t *b_fp4, const uint8_t *b_sf, const float *alpha,
                                     uint16_t *d, int64_t m, int64_t n, int64_t k, void *workspace,
                                     size_t ws_bytes, nvfp4_algo algo, nvfp4_stream_t stream);
/* Scratch bytes for bf16_fp4_gemm_prescaled: the scaled activations
 * (m*k*2 rounded up to 256) plus bf16_fp4_gemm_workspace_bytes when it runs
 * on the tensor cores (NVFP4_ALGO_AUTO on a supported shape, TC or
 * TC_SWAPAB), 0 on the GEMV.  Host only, no GPU needed. */
size_t bf16_fp4_gemm_prescaled_workspace_bytes(int64_t m, int64_t n, int64_t k, nvfp4_algo algo);

/* The whole decode MLP in one kernel launch: nvfp4_quantize of x, the gate_up
 * GEMM with the SwiGLU + NVFP4 requantize epilogue, and the down_proj GEMM
 * ([P1] "关键源码片段": quantize -> gate_up -> silu_mul_nvfp4_quantize ->
 * down_proj; [P2] "实现拆解" item 1: the fused gate_up + SwiGLU + FP4
 * quantize).  One CTA per SM streams its share of the gate_up weights and
 * then of the down_proj weights with no pause between the steps; the steps
 * that depend on each other meet at grid-wide counters in the workspace.
 *   x                bf16 [m, hidden]
 *   x_global_scale   fp32 [1] DEVICE (gs of x, as nvfp4_quantize)
 *   w_gate_up_int(_sf)  the gate/up-interleaved weight [2*inter, hidden/2]
 *                    and its swizzled scales (nvfp4_prepare_gate_up_interleaved)
 *   alpha_gate_up    fp32 [1] = 1/(gs_x * gs_w_gate_up)
 *   h_global_scale   fp32 [1]: static input scale of down_proj
 *   w_down(_sf)      [hidden, inter/2] and swizzled scales (nvfp4_prepare_weights)
 *   alpha_down       fp32 [1] = 1/(gs_h * gs_w_down)
 *   x_fp4, x_sf      OUT: quantized x, exactly as nvfp4_quantize (swizzled
 *                    scales, nvfp4_sf_bytes(m, hidden) bytes)
 *   h_fp4, h_sf      OUT: NVFP4 h [m, inter/2] + swizzled scales
 *                    (nvfp4_sf_bytes(m, inter) bytes)
 *   out              OUT: bf16 [m, hidden]
 *   round_gate_up_bf16  1: the gate_up result is rounded to bf16 before
 *                    SwiGLU, as nvfp4_gemm followed by silu_mul_nvfp4_quantize
 *                    computes it; 0: SwiGLU on the fp32 accumulators, as
 *                    nvfp4_gemm_swiglu_quant.
 *   workspace        DEVICE, >= nvfp4_mlp_decode_workspace_bytes(m, hidden,
 *                    inter), zero-filled once before first use; every
 *                    complete call leaves its counters at zero again.  Calls
 *                    sharing a workspace must not run concurrently.  After
 *                    NVFP4_ERR_DEVICE_TIMEOUT zero-fill it again.
 * Requires 1 <= m <= 64 (m == 0 is a no-op), hidden % 128 == 0,
 * inter % 64 == 0, 16-byte aligned buffers.  The kernel's CTAs wait on each
 * other: it is launched with at most one CTA per SM, and a kernel that the
 * caller runs concurrently on another stream can delay it but not block it.
 * Before launching, the call checks that the device can hold the whole grid
 * at once (occupancy per SM x SM count) and returns
 * NVFP4_ERR_UNSUPPORTED_SHAPE, launching nothing, when it cannot.
 * Tolerances as the separate calls. */
nvfp4_status nvfp4_mlp_decode(const uint16_t *x, const float *x_global_scale,
                              const uint8_t *w_gate_up_int, const uint8_t *w_gate_up_int_sf,
                              const float *alpha_gate_up, const float *h_global_scale,
                              const uint8_t *w_down, const uint8_t *w_down_sf,
                              const float *alpha_down, uint8_t *x_fp4, uint8_t *x_sf,
                              uint8_t *h_fp4, uint8_t *h_sf, uint16_t *out, int64_t m,
                              int64_t hidden, int64_t inter, int round_gate_up_bf16,
                              void *workspace, size_t ws_bytes, nvfp4_stream_t stream);
/* Workspace bytes for nvfp4_mlp_decode (0 for an unsupported shape). */
size_t nvfp4_mlp_decode_workspace_bytes(int64_t m, int64_t hidden, int64_t inter);

/* Weight prep, run once at load time ([P2] modelopt_quant.py excerpt:
 * process_weights_after_loading; [P3] "实现拆解" item 2:
 * prepare_bf16_fp4_weights).  Takes the LINEAR scales (the pages snapshot the
 * raw scales before any swizzle) and writes:
 *   w_out  uint8 [n, k/2]  copy of w_fp4 (w_out == w_fp4 is allowed: no copy)
 *   sf_out swizzled, nvfp4_sf_bytes(n, k, SWIZZLED) bytes.
 * The same prepared weight serves nvfp4_gemm and bf16_fp4_gemm.
 * Requires k % 16 == 0. */
nvfp4_status nvfp4_prepare_weights(const uint8_t *w_fp4, const uint8_t *sf_linear, int64_t n,
                                   int64_t k, uint8_t *w_out, uint8_t *sf_out,
                                   nvfp4_stream_t stream);

/* Gate/up interleave for the fused kernel ([P2] modelopt_quant.py excerpt:
 * interleave_linear_and_gate(cat(up, gate), group_size=64) on the weight and
 * on the un-swizzled scales, then swizzle_blockscale_2d on the scales).
 *   w_fp4     uint8 [n = 2I, k/2] rows [gate; up];  sf_linear uint8 [n, k/16]
 *   w_out     uint8 [n, k/2]: output row 128b + j is up row 64b + j (j < 64),
 *             gate row 64b + j - 64 (j >= 64);  must not alias w_fp4
 *   sf_out    swizzled scales of the interleaved rows.
 * Requires n % 128 == 0, k % 16 == 0. */
nvfp4_status nvfp4_prepare_gate_up_interleaved(const uint8_t *w_fp4, const uint8_t *sf_linear,
                                               int64_t n, int64_t k, uint8_t *w_out,
                                               uint8_t *sf_out, nvfp4_stream_t stream);

/* Decode W4A4 GEMM that allocates nothing (the source pages have no
 * counterpart to this call).  Same operands, result and tolerance as
 * nvfp4_gemm_ex with NVFP4_ALGO_TC_SWAPAB, for callers that cannot hand the
 * library a workspace: the split-K scratch comes from an 8 MiB array inside
 * the library (one per GPU that loads it, held until the process exits).
 *   Requires 1 <= m <= 64 (m == 0 is a no-op), k % 64 == 0, n % 32 == 0, and
 *   that the split plan for (m, n, k) fits in the 8 MiB; otherwise
 *   NVFP4_ERR_UNSUPPORTED_SHAPE and nothing runs.
 *   The first call on a device looks up the array's device address (with
 *   that device current); make that first call before any stream capture.
 *   Each call zeroes the array's arrival counters on `stream` before its
 *   kernel, and the array keeps the last call's partial sums afterwards.  All
 *   calls on a device share the one array, so calls that can run on the GPU
 *   at the same time (for instance on two streams) race on it: serialize
 *   them.  Calls no cudaMalloc/cudaFree or other allocating routine. */
nvfp4_status nvfp4_gemm_decode_noalloc(const uint8_t *a_fp4, const uint8_t *a_sf,
                                       const uint8_t *b_fp4, const uint8_t *b_sf,
                                       const float *alpha, uint16_t *d, int64_t m, int64_t n,
                                       int64_t k, nvfp4_stream_t stream);

/* Synchronizes `stream`, then returns in *status_out (HOST pointer) the
 * device status word of the current device -- NVFP4_OK, or
 * NVFP4_ERR_DEVICE_TIMEOUT if a kernel gave up a bounded pipeline wait since
 * the last call -- and clears it.  The return value reports the call itself. */
nvfp4_status nvfp4_get_device_status(int *status_out, nvfp4_stream_t stream);

/* Testing hook for the bounded waits: sets the spin limit the tensor-core
 * kernels use for every mbarrier wait (0 restores the default, about 2 s at
 * full clock).  A limit of 1 makes a wait give up at once; the kernel then
 * records NVFP4_ERR_DEVICE_TIMEOUT and returns without faulting. */
nvfp4_status nvfp4_set_wait_limit(uint32_t spins);

#ifdef __cplusplus
}
#endif
#endif /* NVFP4MLP_H */
