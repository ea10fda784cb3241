// Elementwise kernels of the NVFP4 MLP: activation quantize, fused
// SiLU*mul + quantize, SiLU*mul to bf16, and the load-time weight prep.
// All HBM-bound: one pass over the input, vector loads, coalesced stores.
#include "common.cuh"
#include "internal.h"

namespace nvfp4 {

namespace {

// The tiled kernels map a 512-byte tile of the swizzled scale layout (128
// rows x 4 scale columns, 64 elements of K) onto one CTA's threads: thread t
// owns the block (row, column) whose scale byte sits at offset t of the tile,
// so each tile's scale stores are one contiguous 512-byte write, and each
// group of 4 threads reads 128 contiguous bytes of one input row.  The
// quantize kernel takes two consecutive tiles along K a CTA, the fused
// SiLU*mul quantize one.
constexpr int kTileThreads = 512;

__device__ __forceinline__ void tile_coords(int t, int64_t &row, int64_t &col) {
  const int c4 = t & 3, r4 = (t >> 2) & 3, r32 = t >> 4;
  row = (int64_t)blockIdx.y * 128 + r4 * 32 + r32;
  col = (int64_t)blockIdx.x * 4 + c4;
}

__device__ __forceinline__ void load16_bf16(const uint16_t *p, float (&x)[16]) {
  const uint4 *q = reinterpret_cast<const uint4 *>(p);
  const uint4 v0 = __ldcs(q), v1 = __ldcs(q + 1);
  const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16_lo(w[i]);
    x[2 * i + 1] = bf16_hi(w[i]);
  }
}

// x [m, k] bf16 -> codes [m, k/2] + scales.  Grid (ceil(k/128), ceil(m/128)):
// a CTA takes two consecutive scale tiles along K, thread t the block at
// offset t of each; both blocks' loads are issued before either is
// quantized, so an SM (three CTAs of 512 threads) keeps twice the bytes in
// flight that one block a thread would (HBM-bound: 96 % of the measured copy
// bandwidth at [8192, 7168], against 83 % with one).
__global__ void __launch_bounds__(kTileThreads, 3) quantize_kernel(
    const uint16_t *__restrict__ x, int64_t m, int64_t k, const float *__restrict__ gs_ptr,
    uint8_t *__restrict__ out_fp4, uint8_t *__restrict__ out_sf, bool swizzled) {
  pdl_trigger();
  pdl_wait();
  constexpr int TPC = 2;
  const int t = threadIdx.x;
  const int64_t row = (int64_t)blockIdx.y * 128 + ((t >> 2) & 3) * 32 + (t >> 4);
  const int64_t cols = k >> 4;
  const int64_t cp4 = (cols + 3) >> 2;
  uint4 raw[TPC][2];
#pragma unroll
  for (int i = 0; i < TPC; ++i) {
    const int64_t col = ((int64_t)blockIdx.x * TPC + i) * 4 + (t & 3);
    if (row < m && col < cols) {
      const uint4 *q = reinterpret_cast<const uint4 *>(x + row * k + col * 16);
      raw[i][0] = __ldcs(q);
      raw[i][1] = __ldcs(q + 1);
    }
  }
  const float gs = __ldg(gs_ptr);
#pragma unroll
  for (int i = 0; i < TPC; ++i) {
    const int64_t tile = (int64_t)blockIdx.x * TPC + i;
    const int64_t col = tile * 4 + (t & 3);
    const bool valid = row < m && col < cols;
    uint32_t sf = 0;
    if (valid) {
      const uint32_t w[8] = {raw[i][0].x, raw[i][0].y, raw[i][0].z, raw[i][0].w,
                             raw[i][1].x, raw[i][1].y, raw[i][1].z, raw[i][1].w};
      float v[16];
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        v[2 * j] = bf16_lo(w[j]);
        v[2 * j + 1] = bf16_hi(w[j]);
      }
      uint32_t lo, hi;
      sf = quantize_block16(v, gs, lo, hi);
      *reinterpret_cast<uint2 *>(out_fp4 + row * (k >> 1) + col * 8) = make_uint2(lo, hi);
    }
    if (swizzled) {
      if (tile < cp4) out_sf[(((int64_t)blockIdx.y * cp4 + tile) << 9) + t] = (uint8_t)sf;
    } else if (valid) {
      out_sf[row * cols + col] = (uint8_t)sf;
    }
  }
}

// Per-token quantize: one CTA per row (rows past m only zero their padding
// scales).  Pass 1 reduces the row's amax, gs = fp32(448*6 / amax) (1 for an
// all-zero row); pass 2 quantizes every 16-block with gs exactly as
// quantize_kernel; row_scale[row] = fp32(1 / gs) is the dequant factor a GEMM
// folds into that row.
__global__ void __launch_bounds__(256) quantize_per_token_kernel(
    const uint16_t *__restrict__ x, int64_t m, int64_t k, uint8_t *__restrict__ out_fp4,
    uint8_t *__restrict__ out_sf, bool swizzled, float *__restrict__ row_scale) {
  pdl_trigger();
  pdl_wait();
  const int64_t row = blockIdx.x;
  const int64_t cols = k >> 4, cp4 = (cols + 3) >> 2;
  const int64_t cols_pad = swizzled ? cp4 * 4 : cols;
  if (row >= m) {        // padding rows of the swizzled layout
    for (int64_t j = threadIdx.x; j < cols_pad; j += blockDim.x) out_sf[sf_swizzled_offset(row, j, cp4)] = 0;
    return;
  }
  __shared__ float s_red[8];
  float amax = 0.0f;
  for (int64_t j = threadIdx.x; j < cols; j += blockDim.x) {
    float v[16];
    load16_bf16(x + row * k + j * 16, v);
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = 0.0f;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) amax = fmaxf(amax, s_red[w]);
  const float gs = amax > 0.0f ? __fdiv_rn(2688.0f, amax) : 1.0f;    // 448 * 6
  for (int64_t j = threadIdx.x; j < cols_pad; j += blockDim.x) {
    uint32_t sf = 0;
    if (j < cols) {
      float v[16];
      load16_bf16(x + row * k + j * 16, v);
      uint32_t lo, hi;
      sf = quantize_block16(v, gs, lo, hi);
      *reinterpret_cast<uint2 *>(out_fp4 + row * (k >> 1) + j * 8) = make_uint2(lo, hi);
    }
    if (swizzled) out_sf[sf_swizzled_offset(row, j, cp4)] = (uint8_t)sf;
    else out_sf[row * cols + j] = (uint8_t)sf;
  }
  if (threadIdx.x == 0) row_scale[row] = __fdiv_rn(1.0f, gs);
}

// gate_up [m, 2i] bf16 ([gate | up]) -> h = silu(gate)*up (fp32) -> NVFP4
// with swizzled scales.  Same tiling as quantize_kernel over h [m, i].  With
// groups (blockIdx.z), group e's rows start at e * m rows of every tensor, its
// scales at e * sf_group bytes, and only its first masked_m[e] rows are valid
// (the rest get zero scales and untouched codes).
__global__ void __launch_bounds__(kTileThreads) silu_mul_quantize_kernel(
    const uint16_t *__restrict__ gate_up, int64_t m, int64_t inter, const float *__restrict__ gs_ptr,
    uint8_t *__restrict__ out_fp4, uint8_t *__restrict__ out_sf, const int32_t *__restrict__ masked_m,
    int64_t sf_group) {
  pdl_trigger();
  pdl_wait();
  int64_t row, col;
  tile_coords(threadIdx.x, row, col);
  const int64_t e = blockIdx.z;
  const int64_t rows_valid = masked_m ? min((int64_t)max(masked_m[e], 0), m) : m;
  gate_up += e * m * 2 * inter;
  out_fp4 += e * m * (inter >> 1);
  out_sf += e * sf_group;
  const int64_t cols = inter >> 4;
  const int64_t cp4 = (cols + 3) >> 2;
  uint32_t sf = 0;
  if (row < rows_valid && col < cols) {
    const float gs = __ldg(gs_ptr);
    float g[16], u[16], h[16];
    load16_bf16(gate_up + row * 2 * inter + col * 16, g);
    load16_bf16(gate_up + row * 2 * inter + inter + col * 16, u);
    // the fast exponential and division, as the fused GEMM epilogues: h is
    // within ~1e-6 relative of the correctly rounded one, far inside the
    // requantize tolerance, and the kernel stays bound by HBM, not the ALUs
#pragma unroll
    for (int i = 0; i < 16; ++i) h[i] = silu_mul_fast(g[i], u[i]);
    uint32_t lo, hi;
    sf = quantize_block16(h, gs, lo, hi);
    *reinterpret_cast<uint2 *>(out_fp4 + row * (inter >> 1) + col * 8) = make_uint2(lo, hi);
  }
  out_sf[(((int64_t)blockIdx.y * cp4 + blockIdx.x) << 9) + threadIdx.x] = (uint8_t)sf;
}

// out [m, i] = bf16(silu(gate) * up); 8 outputs per thread on a 2-D grid
// (x: groups of 8 columns, y: rows), so that no thread divides an index: the
// kernel's ALU work (the correctly rounded exponential and division) is what
// it shares the HBM time with.
__global__ void __launch_bounds__(256) silu_mul_bf16_kernel(const uint16_t *__restrict__ gate_up,
                                                            int64_t m, int64_t inter,
                                                            uint16_t *__restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int64_t c8 = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t row = blockIdx.y;
  if (c8 >= (inter >> 3) || row >= m) return;
  const uint4 g = __ldcs(reinterpret_cast<const uint4 *>(gate_up + row * 2 * inter + c8 * 8));
  const uint4 u = __ldcs(reinterpret_cast<const uint4 *>(gate_up + row * 2 * inter + inter + c8 * 8));
  const uint32_t gw[4] = {g.x, g.y, g.z, g.w}, uw[4] = {u.x, u.y, u.z, u.w};
  uint32_t o[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float h0 = silu_mul(bf16_lo(gw[i]), bf16_lo(uw[i]));
    const float h1 = silu_mul(bf16_hi(gw[i]), bf16_hi(uw[i]));
    const __nv_bfloat162 b = __floats2bfloat162_rn(h0, h1);  // .x = h0 -> low half
    o[i] = *reinterpret_cast<const uint32_t *>(&b);
  }
  *reinterpret_cast<uint4 *>(out + row * inter + c8 * 8) = make_uint4(o[0], o[1], o[2], o[3]);
}

// NVFP4_AWQ activation pre-scale: out[r, c] = bf16(x[r, c] * s[c]); the fp32
// product of two bf16 values is exact, so the result is rounded once.  Eight
// elements per thread, grid-stride.
__global__ void __launch_bounds__(256) awq_prescale_kernel(const uint16_t *__restrict__ x,
                                                           const uint16_t *__restrict__ s, int64_t m,
                                                           int64_t k, uint16_t *__restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int64_t per_row = k >> 3;
  const int64_t total = m * per_row;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t row = idx / per_row, c8 = idx - row * per_row;
    const uint4 xv = __ldcs(reinterpret_cast<const uint4 *>(x + row * k + c8 * 8));
    const uint4 sv = __ldg(reinterpret_cast<const uint4 *>(s + c8 * 8));
    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w}, sw[4] = {sv.x, sv.y, sv.z, sv.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = bf16x2_mul(xw[i], sw[i]);
    *reinterpret_cast<uint4 *>(out + row * k + c8 * 8) = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// Output row -> source row of the gate/up interleave: blocks of 128 rows are
// [up 64b..64b+63 ; gate 64b..64b+63], with [gate; up] source rows.
__device__ __forceinline__ int64_t interleave_src(int64_t o, int64_t n) {
  const int64_t b = o >> 7, j = o & 127;
  return j < 64 ? (n >> 1) + 64 * b + j : 64 * b + (j - 64);
}

// Row copy (8 bytes per thread), with the optional interleave row map.
__global__ void __launch_bounds__(256) prep_rows_kernel(const uint8_t *__restrict__ w, int64_t n,
                                                        int64_t row_bytes, uint8_t *__restrict__ w_out,
                                                        bool interleave) {
  const int64_t per_row = row_bytes >> 3;
  const int64_t total = n * per_row;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t o = idx / per_row, c = idx - o * per_row;
    const int64_t src = interleave ? interleave_src(o, n) : o;
    reinterpret_cast<uint2 *>(w_out + o * row_bytes)[c] =
        reinterpret_cast<const uint2 *>(w + src * row_bytes)[c];
  }
}

// Linear scales [n, cols] -> swizzled; 4 output bytes (one row, 4 scale
// columns) per thread; padding rows and columns get 0.
__global__ void __launch_bounds__(256) prep_sf_kernel(const uint8_t *__restrict__ sf_lin, int64_t n,
                                                      int64_t cols, uint8_t *__restrict__ sf_out,
                                                      bool interleave) {
  const int64_t cp4 = (cols + 3) >> 2;
  const int64_t rp = (n + 127) & ~(int64_t)127;
  const int64_t words = rp * cp4;
  for (int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < words;
       idx += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tile = idx >> 7, within = idx & 127;  // 128 words per 512-byte tile
    const int64_t rb = tile / cp4, kb = tile - rb * cp4;
    const int64_t r = rb * 128 + ((within & 3) << 5) + (within >> 2);
    uint32_t word = 0;
    if (r < n) {
      const int64_t src = interleave ? interleave_src(r, n) : r;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int64_t j = kb * 4 + c;
        if (j < cols) word |= (uint32_t)sf_lin[src * cols + j] << (8 * c);
      }
    }
    reinterpret_cast<uint32_t *>(sf_out)[idx] = word;
  }
}

inline unsigned grid_for(int64_t work, int threads) {
  int64_t blocks = (work + threads - 1) / threads;
  const int64_t cap = 152 * 16;
  return (unsigned)(blocks < 1 ? 1 : (blocks > cap ? cap : blocks));
}

}  // namespace

cudaError_t launch_quantize(const uint16_t *x, int64_t m, int64_t k, const float *gs,
                            uint8_t *out_fp4, uint8_t *out_sf, bool swizzled, cudaStream_t st) {
  const dim3 grid((unsigned)(((k / 16 + 3) / 4 + 1) / 2), (unsigned)((m + 127) / 128));
  return launch_pdl(quantize_kernel, grid, dim3(kTileThreads), 0, st, x, m, k, gs, out_fp4, out_sf, swizzled);
}

cudaError_t launch_quantize_per_token(const uint16_t *x, int64_t m, int64_t k, uint8_t *out_fp4,
                                      uint8_t *out_sf, bool swizzled, float *row_scale, cudaStream_t st) {
  const int64_t rows = swizzled ? (m + 127) / 128 * 128 : m;
  return launch_pdl(quantize_per_token_kernel, dim3((unsigned)rows), dim3(256), 0, st, x, m, k, out_fp4, out_sf,
                    swizzled, row_scale);
}

cudaError_t launch_silu_mul_quantize(const uint16_t *gate_up, int64_t m, int64_t i, const float *gs,
                                     uint8_t *out_fp4, uint8_t *out_sf, cudaStream_t st) {
  const dim3 grid((unsigned)((i / 16 + 3) / 4), (unsigned)((m + 127) / 128));
  return launch_pdl(silu_mul_quantize_kernel, grid, dim3(kTileThreads), 0, st, gate_up, m, i, gs, out_fp4,
                    out_sf, (const int32_t *)nullptr, (int64_t)0);
}

cudaError_t launch_silu_mul_quantize_masked(const uint16_t *gate_up, const int32_t *masked_m, int64_t g,
                                            int64_t m_max, int64_t i, const float *gs, uint8_t *out_fp4,
                                            uint8_t *out_sf, cudaStream_t st) {
  const int64_t sf_group = ((m_max + 127) / 128 * 128) * ((i / 16 + 3) / 4 * 4);
  const dim3 grid((unsigned)((i / 16 + 3) / 4), (unsigned)((m_max + 127) / 128), (unsigned)g);
  return launch_pdl(silu_mul_quantize_kernel, grid, dim3(kTileThreads), 0, st, gate_up, m_max, i, gs, out_fp4,
                    out_sf, masked_m, sf_group);
}

cudaError_t launch_silu_mul_bf16(const uint16_t *gate_up, int64_t m, int64_t i, uint16_t *out,
                                 cudaStream_t st) {
  if (m > 65535) {      // (the grid's y extent) in slices of rows
    for (int64_t r0 = 0; r0 < m; r0 += 65535) {
      const int64_t rows = m - r0 < 65535 ? m - r0 : 65535;
      if (cudaError_t e = launch_silu_mul_bf16(gate_up + r0 * 2 * i, rows, i, out + r0 * i, st)) return e;
    }
    return cudaSuccess;
  }
  const dim3 grid((unsigned)((i / 8 + 255) / 256), (unsigned)m);
  return launch_pdl(silu_mul_bf16_kernel, grid, dim3(256), 0, st, gate_up, m, i, out);
}

cudaError_t launch_awq_prescale(const uint16_t *x, const uint16_t *s, int64_t m, int64_t k, uint16_t *out,
                                cudaStream_t st) {
  return launch_pdl(awq_prescale_kernel, dim3(grid_for(m * (k / 8), 256)), dim3(256), 0, st, x, s, m, k, out);
}

cudaError_t launch_prepare(const uint8_t *w, const uint8_t *sf_lin, int64_t n, int64_t k,
                           uint8_t *w_out, uint8_t *sf_out, bool interleave, cudaStream_t st) {
  if (w_out != w || interleave) {
    prep_rows_kernel<<<grid_for(n * (k / 16), 256), 256, 0, st>>>(w, n, k / 2, w_out, interleave);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  const int64_t cols = k / 16;
  const int64_t words = ((n + 127) / 128 * 128) * ((cols + 3) / 4);
  prep_sf_kernel<<<grid_for(words, 256), 256, 0, st>>>(sf_lin, n, cols, sf_out, interleave);
  return cudaGetLastError();
}

}  // namespace nvfp4
