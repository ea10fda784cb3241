// Device helpers shared by the NVFP4 kernels: number formats, layout index
// math and the status word.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nvfp4mlp.h"

namespace nvfp4 {

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  Every kernel here is launched so that it may
// start while the previous kernel on the stream is still finishing:
// pdl_trigger() lets the next kernel's CTAs launch, pdl_wait() blocks until
// the previous kernel has completed and its memory is visible.  A kernel
// reads the previous kernel's results, and writes any global memory, only
// after pdl_wait(); without the launch attribute pdl_wait() returns at once.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// E2M1 encode of eight floats into one word (element i in nibble i), with the
// PTX conversion cvt.rn.satfinite.e2m1x2.f32: round to nearest even, magnitudes
// past 6 saturate to 6, the sign bit is kept (a negative value that rounds to
// zero gives code 0x8).  The instruction puts its first source operand in the
// high nibble.
__device__ __forceinline__ uint32_t e2m1_pack8(float v0, float v1, float v2, float v3, float v4, float v5,
                                               float v6, float v7) {
  uint32_t w;
  asm("{\n"
      ".reg .b8 b0, b1, b2, b3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b0, %2, %1;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b1, %4, %3;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b2, %6, %5;\n"
      "cvt.rn.satfinite.e2m1x2.f32 b3, %8, %7;\n"
      "mov.b32 %0, {b0, b1, b2, b3};\n"
      "}"
      : "=r"(w)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3), "f"(v4), "f"(v5), "f"(v6), "f"(v7));
  return w;
}

// E4M3 (e4m3fn) encode of a non-negative float, round to nearest even,
// saturating to 448: the PTX conversion does exactly this.
__device__ __forceinline__ uint32_t e4m3_encode_satfinite(float s) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(0.0f), "f"(s));
  return r & 0xFFu;
}

// E4M3 code (non-negative, not NaN) -> float, from the bit fields: exponent
// field e (bias 7), mantissa m (3 bits); e == 0 is subnormal m * 2^-9.
__device__ __forceinline__ float e4m3_decode(uint32_t code) {
  const uint32_t e = (code >> 3) & 0xFu, m = code & 7u;
  if (e == 0) return (float)m * 0.001953125f;  // 2^-9
  return __uint_as_float(((e + 120u) << 23) | (m << 20));
}

// bf16 bits -> float (exact).
__device__ __forceinline__ float bf16_lo(uint32_t two) { return __uint_as_float(two << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t two) { return __uint_as_float(two & 0xFFFF0000u); }

// NVFP4 quantize of one 16-element block held in registers, in the order
// the API documents: s = fp32(amax/6)*gs, SF = E4M3(s), r = gs/SF, codes of
// x*r.  Returns the scale byte; writes the 8 packed code bytes to lo/hi.
__device__ __forceinline__ uint32_t quantize_block16(const float (&x)[16], float gs, uint32_t &lo,
                                                     uint32_t &hi) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
  const float s = __fmul_rn(__fdiv_rn(amax, 6.0f), gs);
  const uint32_t sf = e4m3_encode_satfinite(s);
  const float r = (sf == 0u) ? 0.0f : __fdiv_rn(gs, e4m3_decode(sf));
  float v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __fmul_rn(x[i], r);
  lo = e2m1_pack8(v[0], v[1], v[2], v[3], v[4], v[5], v[6], v[7]);
  hi = e2m1_pack8(v[8], v[9], v[10], v[11], v[12], v[13], v[14], v[15]);
  return sf;
}

// Byte offset of block scale (row r, scale column j) in the 128x4 swizzled
// layout with cp4 = padded scale columns / 4.
__host__ __device__ __forceinline__ int64_t sf_swizzled_offset(int64_t r, int64_t j, int64_t cp4) {
  return (((r >> 7) * cp4 + (j >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (j & 3);
}

// silu(g) * u with the fast exponential and division (relative error about
// 1e-6; h feeds a quantizer whose steps are ~1e-1 apart).
__device__ __forceinline__ float silu_mul_fast(float g, float u) {
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// bf16x2 * bf16x2 rounded once to bf16x2: the fp32 product of two bf16
// values is exact, so this is the correctly rounded bf16 product.
__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t x, uint32_t s) {
  const __nv_bfloat162 r =
      __floats2bfloat162_rn(__fmul_rn(bf16_lo(x), bf16_lo(s)), __fmul_rn(bf16_hi(x), bf16_hi(s)));
  return *reinterpret_cast<const uint32_t *>(&r);
}

// silu(g) * u in fp32 with an IEEE division.
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

}  // namespace nvfp4
