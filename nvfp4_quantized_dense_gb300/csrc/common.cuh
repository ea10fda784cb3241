// Device helpers shared by the NVFP4 kernels: number formats, layout index
// math and the status word.  sm_103a only.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "nvfp4mlp.h"

namespace nvfp4 {

// ---------------------------------------------------------------------------
// E2M1 encode, round to nearest even with saturation at 6.  The magnitude
// code is the number of decision thresholds |v| lies above: a threshold is a
// midpoint between neighbouring magnitudes {0,.5,1,1.5,2,3,4,6}; at an exact
// midpoint the even code wins, which is ">" for midpoints whose lower
// neighbour has an even code and ">=" for the others.  Bit 3 copies the sign
// bit of v (so -0.1 encodes as 0x8).
__device__ __forceinline__ uint32_t e2m1_encode(float v) {
  const float a = fabsf(v);
  uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
               (a >= 3.5f) + (a > 5.0f);
  return c | ((__float_as_uint(v) >> 28) & 8u);
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
  lo = 0u;
  hi = 0u;
#pragma unroll
  for (int i = 0; i < 8; ++i) lo |= e2m1_encode(__fmul_rn(x[i], r)) << (4 * i);
#pragma unroll
  for (int i = 0; i < 8; ++i) hi |= e2m1_encode(__fmul_rn(x[8 + i], r)) << (4 * i);
  return sf;
}

// Byte offset of block scale (row r, scale column j) in the 128x4 swizzled
// layout with cp4 = padded scale columns / 4.
__host__ __device__ __forceinline__ int64_t sf_swizzled_offset(int64_t r, int64_t j, int64_t cp4) {
  return (((r >> 7) * cp4 + (j >> 2)) << 9) + ((r & 31) << 4) + (((r >> 5) & 3) << 2) + (j & 3);
}

// silu(g) * u in fp32 with an IEEE division.
__device__ __forceinline__ float silu_mul(float g, float u) {
  return __fmul_rn(__fdiv_rn(g, __fadd_rn(1.0f, expf(-g))), u);
}

}  // namespace nvfp4
