// Decode-sized GEMMs on CUDA cores: the weight stream is the roofline.
//
// Each warp owns R consecutive weight rows; its lanes split K into 32-element
// chunks (16 bytes of codes, two 16-element scale blocks), so one warp load
// instruction reads 512 contiguous bytes of a row, with streaming
// (evict-first) loads.  The partial sums are reduced across the warp by
// shuffles.  Up to MT tokens are handled per pass, reusing each decoded
// weight chunk MT times.
//
// W4A4 arithmetic: E2M1 codes of both operands convert exactly to fp16; the
// 16 products of one scale block are summed by 8 half2 FMAs, which is exact
// (each half accumulates 8 products of magnitude <= 36 on a 0.25 grid, so
// every partial sum is <= 288 and representable).  The block sum times the
// product of the two E4M3 scales is exact in fp32 too; only the fp32
// accumulation over blocks rounds.
//
// W4A16: weights decode exactly to fp16 -> fp32 and meet the bf16 activation
// in fp32 FMAs; each block's sum is scaled by the weight's E4M3 scale.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"

namespace nvfp4 {
namespace {

constexpr int kWarps = 8;

// Four packed bytes (8 E2M1 codes) -> 4 half2, element order preserved
// (the code of the lower K index lands in the lower half).
__device__ __forceinline__ void e2m1x8_to_half2x4(uint32_t w, uint32_t (&h)[4]) {
  asm("{\n"
      ".reg .b8 b0, b1, b2, b3;\n"
      "mov.b32 {b0, b1, b2, b3}, %4;\n"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n"
      "}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(w));
}

__device__ __forceinline__ void decode_chunk(const uint4 &v, uint32_t (&h)[16]) {
  uint32_t t[4];
  e2m1x8_to_half2x4(v.x, t);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[i] = t[i];
  e2m1x8_to_half2x4(v.y, t);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[4 + i] = t[i];
  e2m1x8_to_half2x4(v.z, t);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[8 + i] = t[i];
  e2m1x8_to_half2x4(v.w, t);
#pragma unroll
  for (int i = 0; i < 4; ++i) h[12 + i] = t[i];
}

// L2 policy for the weight stream: read once per call, evict first.
__device__ __forceinline__ uint64_t evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint4 ld_stream16(const uint8_t *p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}

// Two adjacent scale bytes (scale columns j, j+1 with j even) of row r.
__device__ __forceinline__ uint32_t ld_sf_pair(const uint8_t *sf, int64_t r, int64_t j, int64_t cp4) {
  return *reinterpret_cast<const uint16_t *>(sf + sf_swizzled_offset(r, j, cp4));
}

__device__ __forceinline__ float half2_sum(uint32_t h) {
  const __half2 v = *reinterpret_cast<const __half2 *>(&h);
  return __low2float(v) + __high2float(v);
}

__device__ __forceinline__ uint32_t hfma2(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct GemvArgs {
  const uint8_t *a;    // W4A4: codes [M, K/2]; W4A16: bf16 [M, K]
  const uint8_t *a_sf; // W4A4: swizzled scales over M rows
  const uint8_t *b;    // codes [N, K/2]
  const uint8_t *b_sf; // swizzled scales over N rows
  const float *alpha;
  const float *out_gs;
  uint16_t *d;         // bf16 [M, N]
  uint8_t *out_fp4;    // fused: [M, N/4]
  uint8_t *out_sf;     // fused: swizzled over M rows, N/32 columns
  int64_t m, n, k;
  int64_t m0;          // first token of this pass
  const float *rs;     // optional per-token dequant factor [M]
  const uint16_t *pqs; // W4A16: optional AWQ pre_quant_scale, bf16 [K]
};

// Weight row handled by warp `w`, sub-row `r` of CTA `cta`.  Plain mode: rows
// are consecutive.  SwiGLU mode (R = 4, 8 warps): the CTA owns 16 output
// features f0 = 16*cta; warps 0-3 take their up rows, warps 4-7 their gate
// rows, in the interleaved weight order (blocks of 128 = [64 up ; 64 gate]).
template <int R, bool SWIGLU>
__device__ __forceinline__ int64_t weight_row(int64_t cta, int w, int r) {
  if (!SWIGLU) return (cta * kWarps + w) * R + r;
  const int64_t blk = cta >> 2, q = cta & 3;
  const int64_t base = blk * 128 + q * 16 + (w >= 4 ? 64 : 0);
  return base + (w & 3) * R + r;
}

// SwiGLU epilogue of the GEMV: the CTA's 16 up and 16 gate sums per token
// meet in shared memory; one thread per token forms h = silu(gate)*up and
// quantizes the 16-feature block.
template <int MT, int R>
__device__ __forceinline__ void swiglu_epilogue(const GemvArgs &p, float (&acc)[MT][R], float alpha,
                                                int warp, int lane, int64_t cta, int mt) {
  __shared__ float s_up[MT][16], s_gate[MT][16];
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float v = warp_sum(acc[t][r]);
      if (lane == 0) {
        const int f = (warp & 3) * R + r;
        const float at = (p.rs && t < mt) ? alpha * p.rs[p.m0 + t] : alpha;
        if (warp < 4) s_up[t][f] = at * v;
        else s_gate[t][f] = at * v;
      }
    }
  __syncthreads();
  const int64_t inter = p.n >> 1;
  const int64_t f0 = 16 * cta;                    // first output feature
  const int64_t ocols = inter >> 4, ocp4 = (ocols + 3) >> 2;
  const int64_t mpad = (p.m + 127) & ~(int64_t)127;
  const int64_t jcol = f0 >> 4;
  if ((int)threadIdx.x < MT) {
    const int t = threadIdx.x;
    if (t < mt) {
      float h[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) h[i] = silu_mul(s_gate[t][i], s_up[t][i]);
      uint32_t lo, hi;
      const uint32_t sf = quantize_block16(h, __ldg(p.out_gs), lo, hi);
      const int64_t tok = p.m0 + t;
      *reinterpret_cast<uint2 *>(p.out_fp4 + tok * (inter >> 1) + f0 / 2) = make_uint2(lo, hi);
      p.out_sf[sf_swizzled_offset(tok, jcol, ocp4)] = (uint8_t)sf;
    }
  }
  // the pass that handles the last tokens also zeroes the padding rows
  if (p.m0 + MT >= p.m) {
    for (int64_t r = p.m + threadIdx.x; r < mpad; r += blockDim.x)
      p.out_sf[sf_swizzled_offset(r, jcol, ocp4)] = 0;
  }
}

template <int MT, int R, bool SWIGLU>
__global__ void __launch_bounds__(kWarps * 32) gemv_w4a4_kernel(GemvArgs p) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t cta = blockIdx.x;
  const int64_t kb = p.k >> 1;                  // bytes per row
  const int64_t cp4 = ((p.k >> 4) + 3) >> 2;    // scale column groups
  const int mt = (int)min((int64_t)MT, p.m - p.m0);
  const int64_t nchunks = p.k >> 5;
  const uint64_t pol = evict_first_policy();

  int64_t rows[R];
#pragma unroll
  for (int r = 0; r < R; ++r) rows[r] = weight_row<R, SWIGLU>(cta, warp, r);

  float acc[MT][R];
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int r = 0; r < R; ++r) acc[t][r] = 0.0f;

  for (int64_t c = lane; c < nchunks; c += 32) {
    uint4 wv[R];
    uint32_t wsf[R];
#pragma unroll
    for (int r = 0; r < R; ++r) {
      wv[r] = ld_stream16(p.b + rows[r] * kb + c * 16, pol);
      wsf[r] = ld_sf_pair(p.b_sf, rows[r], 2 * c, cp4);
    }
    uint32_t wh[R][16];
#pragma unroll
    for (int r = 0; r < R; ++r) decode_chunk(wv[r], wh[r]);
#pragma unroll
    for (int t = 0; t < MT; ++t) {
      if (t < mt) {
        const int64_t tok = p.m0 + t;
        const uint4 av = __ldg(reinterpret_cast<const uint4 *>(p.a + tok * kb + c * 16));
        const uint32_t asf = ld_sf_pair(p.a_sf, tok, 2 * c, cp4);
        uint32_t ah[16];
        decode_chunk(av, ah);
        const float sa0 = e4m3_decode(asf & 0xFF), sa1 = e4m3_decode((asf >> 8) & 0xFF);
#pragma unroll
        for (int r = 0; r < R; ++r) {
          uint32_t p0 = 0u, p1 = 0u;
#pragma unroll
          for (int i = 0; i < 8; ++i) p0 = hfma2(ah[i], wh[r][i], p0);
#pragma unroll
          for (int i = 8; i < 16; ++i) p1 = hfma2(ah[i], wh[r][i], p1);
          const float s0 = sa0 * e4m3_decode(wsf[r] & 0xFF);
          const float s1 = sa1 * e4m3_decode((wsf[r] >> 8) & 0xFF);
          acc[t][r] = fmaf(half2_sum(p0), s0, acc[t][r]);
          acc[t][r] = fmaf(half2_sum(p1), s1, acc[t][r]);
        }
      }
    }
  }

  const float alpha = __ldg(p.alpha);
  if constexpr (!SWIGLU) {
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
      for (int r = 0; r < R; ++r) {
        const float v = warp_sum(acc[t][r]);
        if (lane == 0 && t < mt) {
          const float at = p.rs ? alpha * p.rs[p.m0 + t] : alpha;
          const __nv_bfloat16 o = __float2bfloat16_rn(at * v);
          p.d[(p.m0 + t) * p.n + rows[r]] = *reinterpret_cast<const uint16_t *>(&o);
        }
      }
  } else {
    swiglu_epilogue<MT, R>(p, acc, alpha, warp, lane, cta, mt);
  }
}


// W4A16: each warp takes R consecutive weight rows; its lanes split K into
// 32-element chunks and put B chunks of every row in flight (B*R 16-byte
// evict-first loads per lane before the first is used), so that an SM holds
// ~100 KB of the weight stream in flight.  Each chunk is consumed 8 elements
// at a time: the activations (bf16, read through L1: every warp reads the
// same token rows) are converted to fp32 once and used for the R rows.
template <int MT, int R, int B>
__global__ void __launch_bounds__(kWarps * 32, 2) gemv_w4a16_kernel(GemvArgs p) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row0 = ((int64_t)blockIdx.x * kWarps + warp) * R;
  const int64_t kb = p.k >> 1;
  const int64_t cp4 = ((p.k >> 4) + 3) >> 2;
  const int mt = (int)min((int64_t)MT, p.m - p.m0);
  const int64_t nchunks = p.k >> 5;
  const uint16_t *a = reinterpret_cast<const uint16_t *>(p.a);
  const uint64_t pol = evict_first_policy();

  float acc[MT][R];
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int r = 0; r < R; ++r) acc[t][r] = 0.0f;

  for (int64_t c0 = lane; c0 < nchunks; c0 += 32 * B) {
    uint4 wv[B][R];
    uint32_t wsf[B][R];
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int64_t c = c0 + 32 * b;
#pragma unroll
      for (int r = 0; r < R; ++r) {
        if (c < nchunks) {
          wv[b][r] = ld_stream16(p.b + (row0 + r) * kb + c * 16, pol);
          wsf[b][r] = ld_sf_pair(p.b_sf, row0 + r, 2 * c, cp4);
        } else {
          wv[b][r] = make_uint4(0u, 0u, 0u, 0u);
          wsf[b][r] = 0u;
        }
      }
    }
#pragma unroll
    for (int b = 0; b < B; ++b) {
      const int64_t c = c0 + 32 * b;
      if (c >= nchunks) continue;
#pragma unroll
      for (int t = 0; t < MT; ++t) {
        if (t >= mt) continue;
        const uint4 *ap = reinterpret_cast<const uint4 *>(a + (p.m0 + t) * p.k + c * 32);
        const uint4 *sp = reinterpret_cast<const uint4 *>(p.pqs ? p.pqs + c * 32 : nullptr);
        float bs[R][2];
#pragma unroll
        for (int r = 0; r < R; ++r) bs[r][0] = bs[r][1] = 0.0f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {            // elements 8q .. 8q+7 (scale block q >> 1)
          const uint4 v = __ldg(ap + q);
          const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
          uint32_t s4[4] = {0u, 0u, 0u, 0u};
          if (sp) {
            const uint4 sv = __ldg(sp + q);
            s4[0] = sv.x; s4[1] = sv.y; s4[2] = sv.z; s4[3] = sv.w;
          }
          float x[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            float x0 = bf16_lo(w4[e]), x1 = bf16_hi(w4[e]);
            if (sp) {                            // bf16(x * s): the fp32 product is exact, one rounding
              x0 = __bfloat162float(__float2bfloat16_rn(__fmul_rn(x0, bf16_lo(s4[e]))));
              x1 = __bfloat162float(__float2bfloat16_rn(__fmul_rn(x1, bf16_hi(s4[e]))));
            }
            x[2 * e] = x0;
            x[2 * e + 1] = x1;
          }
#pragma unroll
          for (int r = 0; r < R; ++r) {
            const uint32_t codes = q == 0 ? wv[b][r].x : q == 1 ? wv[b][r].y : q == 2 ? wv[b][r].z : wv[b][r].w;
            uint32_t wh[4];
            e2m1x8_to_half2x4(codes, wh);
            float &sum = bs[r][q >> 1];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const __half2 h = *reinterpret_cast<const __half2 *>(&wh[i]);
              sum = fmaf(x[2 * i], __low2float(h), sum);
              sum = fmaf(x[2 * i + 1], __high2float(h), sum);
            }
          }
        }
#pragma unroll
        for (int r = 0; r < R; ++r) {
          acc[t][r] = fmaf(bs[r][0], e4m3_decode(wsf[b][r] & 0xFF), acc[t][r]);
          acc[t][r] = fmaf(bs[r][1], e4m3_decode((wsf[b][r] >> 8) & 0xFF), acc[t][r]);
        }
      }
    }
  }
  const float alpha = __ldg(p.alpha);
#pragma unroll
  for (int t = 0; t < MT; ++t)
#pragma unroll
    for (int r = 0; r < R; ++r) {
      const float v = warp_sum(acc[t][r]);
      if (lane == 0 && t < mt) {
        const __nv_bfloat16 o = __float2bfloat16_rn(alpha * v);
        p.d[(p.m0 + t) * p.n + row0 + r] = *reinterpret_cast<const uint16_t *>(&o);
      }
    }
}

template <int MT>
cudaError_t launch_mt(GemvMode mode, const GemvArgs &a, cudaStream_t st) {
  const dim3 block(kWarps * 32);
  switch (mode) {
    case GEMV_W4A4:
      return launch_pdl(gemv_w4a4_kernel<MT, 2, false>, dim3((unsigned)(a.n / (kWarps * 2))), block, 0, st, a);
    case GEMV_W4A4_SWIGLU:
      return launch_pdl(gemv_w4a4_kernel<MT, 4, true>, dim3((unsigned)(a.n / 32)), block, 0, st, a);
    case GEMV_W4A16:
      if constexpr (MT > 4) {
        return cudaErrorInvalidValue;   // W4A16 passes hold at most 4 tokens
      } else {
        // two rows a warp (the activation chunk converted once for both) when
        // that still leaves 16 warps an SM; one row with twice the chunks in
        // flight otherwise
        if (a.n >= (int64_t)num_sms() * kWarps * 2 * 2 * 2)
          return launch_pdl(gemv_w4a16_kernel<MT, 2, 4>, dim3((unsigned)(a.n / (kWarps * 2))), block, 0, st, a);
        return launch_pdl(gemv_w4a16_kernel<MT, 1, 8>, dim3((unsigned)(a.n / kWarps)), block, 0, st, a);
      }
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_gemv(GemvMode mode, const void *a, const uint8_t *a_sf, const uint8_t *b,
                        const uint8_t *b_sf, const float *alpha, const float *out_gs, uint16_t *d,
                        uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n, int64_t k,
                        cudaStream_t st, const float *a_row_scale, const uint16_t *pre_scale) {
  GemvArgs args{static_cast<const uint8_t *>(a), a_sf, b, b_sf, alpha, out_gs, d, out_fp4, out_sf,
                m, n, k, 0, a_row_scale, pre_scale};
  // passes of 16, 8, 4, 2 or 1 tokens (W4A16: at most 4) until every token is covered
  for (int64_t m0 = 0; m0 < m;) {
    const int64_t left = m - m0;
    int mt = left >= 16 ? 16 : left > 4 ? 8 : left > 2 ? 4 : (int)left;
    if (mode == GEMV_W4A16 && mt > 4) mt = 4;
    args.m0 = m0;
    cudaError_t e;
    switch (mt) {
      case 16: e = launch_mt<16>(mode, args, st); break;
      case 8: e = launch_mt<8>(mode, args, st); break;
      case 4: e = launch_mt<4>(mode, args, st); break;
      case 2: e = launch_mt<2>(mode, args, st); break;
      default: e = launch_mt<1>(mode, args, st); break;
    }
    if (e != cudaSuccess) return e;
    m0 += left < mt ? left : mt;
  }
  return cudaSuccess;
}

}  // namespace nvfp4
