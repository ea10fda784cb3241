// W4A16 GEMM on the tensor cores: bf16 activations x NVFP4 weights
// ([P3] fp4_gemm with quant_mode "w4a16": the activation is not quantized,
// alpha holds only the weight dequant factor).
//
// The tensor cores need both operands of a kind::f16 MMA in the same type,
// so the weight is dequantized to bf16 in shared memory: converter warps read
// the stage's E2M1 codes and E4M3 scales (TMA / bulk copies) and write
// E2M1 * scale -- exact in bf16, at most 5 significant bits -- into a
// 128-byte-swizzled K-major tile that the MMA reads directly.  The weight is
// the MMA's 128-row operand and the tokens its N (16..256), so each weight
// element is dequantized once per 256-token tile; D^T[n, t] accumulates in
// TMEM (two buffers) and the epilogue writes D[t, n] with the 32 lanes of a
// warp on 32 consecutive n.
//
// Roles (320 threads, one CTA per SM, persistent over (weight tile, token
// tile) pairs, token tile fastest): warp 0 TMA producer, warp 1 TMEM owner +
// MMA issuer, warps 2..5 converters, warps 6..9 epilogue.  Bounded waits as
// in gemm_tc.cu.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int BK = 64;                      // K per stage: 128 bytes of bf16 per row
constexpr uint32_t WC_BYTES = 128 * BK / 2; // weight codes, 4 KB
constexpr uint32_t WS_BYTES = 512;          // one 128x4 scale tile
constexpr uint32_t WB_BYTES = 128 * BK * 2; // dequantized weight tile, 16 KB
constexpr int kThreads = 320;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint32_t kDrainPolls = 1u << 22;

template <int NT>
struct Cfg {
  static constexpr uint32_t X_BYTES = NT * BK * 2;                       // NT rows x 128 B
  static constexpr uint32_t RAW = X_BYTES + WB_BYTES + WC_BYTES + WS_BYTES;
  static constexpr uint32_t STAGE_BYTES = (RAW + 1023) / 1024 * 1024;
  static constexpr int STAGES = (220 * 1024) / STAGE_BYTES > 8 ? 8 : (220 * 1024) / STAGE_BYTES;
  static constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
  static constexpr uint32_t TMEM_COLS = 2 * NT <= 32 ? 32 : 2 * NT <= 64 ? 64 : 2 * NT <= 128 ? 128 : 2 * NT <= 256 ? 256 : 512;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(STAGES >= 3, "pipeline depth");
};

struct W4A16Args {
  const uint8_t *w;        // codes [N, K/2]
  const uint8_t *wsf;      // swizzled scales over N rows
  const float *alpha;
  uint16_t *d;             // bf16 [M, N]
  int32_t m, n, k;
  int32_t wtiles, ttiles;
  uint32_t wait_limit;
  int *status;
};

__device__ __forceinline__ void conv_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Eight codes (one 32-bit word) times one E4M3 scale -> four bf16x2, exact:
// E2M1 -> f16x2, times the scale in f16 (product within f16's normal range and
// precision), widened to f32 and rounded to bf16 (no rounding happens: the
// values have at most 5 significant bits).
__device__ __forceinline__ void dequant8(uint32_t codes, uint32_t scale_h2, uint32_t (&out)[4]) {
  uint32_t h[4];
  asm("{\n"
      ".reg .b8 b0, b1, b2, b3;\n"
      "mov.b32 {b0, b1, b2, b3}, %4;\n"
      "cvt.rn.f16x2.e2m1x2 %0, b0;\n"
      "cvt.rn.f16x2.e2m1x2 %1, b1;\n"
      "cvt.rn.f16x2.e2m1x2 %2, b2;\n"
      "cvt.rn.f16x2.e2m1x2 %3, b3;\n"
      "}"
      : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3])
      : "r"(codes));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t p;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(p) : "r"(h[i]), "r"(scale_h2));
    const __half2 ph = *reinterpret_cast<const __half2 *>(&p);
    const __nv_bfloat162 b = __floats2bfloat162_rn(__low2float(ph), __high2float(ph));
    out[i] = *reinterpret_cast<const uint32_t *>(&b);
  }
}

// E4M3 scale byte -> f16 duplicated in both halves (exact).
__device__ __forceinline__ uint32_t e4m3_to_h2(uint32_t byte) {
  uint32_t r;
  const uint16_t two = (uint16_t)(byte | (byte << 8));
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(two));
  return r;
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                 const W4A16Args p) {
  using C = Cfg<NT>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t *full = reinterpret_cast<uint64_t *>(base + STAGES * C::STAGE_BYTES);
  uint64_t *conv = full + STAGES;
  uint64_t *empty = conv + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
  auto st_x = [&](int s) { return base + s * C::STAGE_BYTES; };
  auto st_wb = [&](int s) { return st_x(s) + C::X_BYTES; };
  auto st_wc = [&](int s) { return st_wb(s) + WB_BYTES; };
  auto st_ws = [&](int s) { return st_wc(s) + WC_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&conv[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&tfull[b], 1);
      ptx::mbar_init(&tempty[b], 128);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tm_x);
    ptx::prefetch_tensormap(&tm_w);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tslot, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;

  const int tiles = p.wtiles * p.ttiles;
  const int nkb = p.k / BK;
  const int cp4 = p.k >> 6;              // 512-byte scale tiles per 128-row block
  const uint32_t limit = p.wait_limit;
  uint32_t issued_mask = 0, issued_parity = 0;
  bool mma_issued = false;
  auto give_up = [&]() {
    *abort_flag = 1;
    atomicCAS(p.status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
  };

  if (warp == 0) {
    if (ptx::elect_one()) {
      const uint64_t pol_w = ptx::l2_policy_evict_first();
      const uint64_t pol_x = ptx::l2_policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      // The first STAGES stages get their weight codes and scales before the
      // previous kernel on the stream has finished; their activation tiles
      // follow once it has.
      int pend_s[STAGES], pend_kb[STAGES], pend_tt[STAGES];
      int npend = 0, c = 0;
      bool flushed = false;
      auto load_x = [&](int st, int kb, int tt) {
        ptx::tma_load_2d(st_x(st), &tm_x, &full[st], kb * (BK * 2), tt * NT, pol_x);
      };
      auto flush = [&]() {
        pdl_wait();
        for (int i = 0; i < npend; ++i) load_x(pend_s[i], pend_kb[i], pend_tt[i]);
        flushed = true;
      };
      for (int tile = blockIdx.x; tile < tiles && !*abort_flag; tile += gridDim.x) {
        const int wt = tile / p.ttiles, tt = tile % p.ttiles;
        for (int kb = 0; kb < nkb; ++kb, ++c) {
          if (c == STAGES && !flushed) flush();
          if (!ptx::mbar_wait_bounded(&empty[s], ph ^ 1u, limit, kTimeoutNs, abort_flag)) {
            give_up();
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[s], C::X_BYTES + WC_BYTES + WS_BYTES);
          ptx::tma_load_2d(st_wc(s), &tm_w, &full[s], kb * (BK / 2), wt * 128, pol_w);
          ptx::bulk_load(st_ws(s), p.wsf + ((size_t)wt * cp4 + kb) * 512, WS_BYTES, &full[s], pol_w);
          if (c < STAGES) {
            pend_s[npend] = s;
            pend_kb[npend] = kb;
            pend_tt[npend] = tt;
            ++npend;
          } else {
            load_x(s, kb, tt);
          }
          issued_mask |= 1u << s;
          issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
      if (!flushed) flush();
    }
  } else if (warp == 1) {
    pdl_wait();
    if (ptx::elect_one()) {
      // kind::f16: F32 accumulator (bits 4-5 = 1), A = B = BF16 (1), K-major,
      // N >> 3 in bits 17-22, M = 128 >> 4 in bits 24-28
      constexpr uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NT >> 3) << 17) | (8u << 24);
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      for (int tile = blockIdx.x; tile < tiles && !*abort_flag; tile += gridDim.x, ++it) {
        const int ab = it & 1;
        if (!ptx::mbar_wait_bounded(&tempty[ab], (uint32_t)((it >> 1) & 1) ^ 1u, limit, kTimeoutNs, abort_flag)) {
          give_up();
          break;
        }
        ptx::tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!ptx::mbar_wait_bounded(&full[s], ph, limit, kTimeoutNs, abort_flag) ||
              !ptx::mbar_wait_bounded(&conv[s], ph, limit, kTimeoutNs, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t wb = ptx::smem_u32(st_wb(s)), xs = ptx::smem_u32(st_x(s));
#pragma unroll
          for (int j = 0; j < BK / 16; ++j)
            ptx::mma_bf16(tmem + ab * NT, ptx::smem_desc(wb + 32 * j, 16, 1024, 2),
                          ptx::smem_desc(xs + 32 * j, 16, 1024, 2), idesc, (kb | j) != 0);
          mma_issued = true;
          ptx::tc_commit(&empty[s]);
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        ptx::tc_commit(&tfull[ab]);
      }
    }
  } else if (warp < 6) {
    // ---------------------------------------------------------- converters
    pdl_wait();
    const int r = threadIdx.x - 64;             // weight row of the tile, 0..127
    const int swz = r & 7;
    int s = 0;
    uint32_t ph = 0;
    bool ok = true;
    for (int tile = blockIdx.x; tile < tiles && ok; tile += gridDim.x) {
      for (int kb = 0; kb < nkb; ++kb) {
        const bool got = ptx::mbar_wait_bounded(&full[s], ph, limit, kTimeoutNs, abort_flag);
        if (!got) give_up();
        if (ptx::bar_any(1, 128, !got || *abort_flag)) {   // the four warps leave together
          ok = false;
          break;
        }
        const uint4 *codes = reinterpret_cast<const uint4 *>(st_wc(s) + r * (BK / 2));
        const uint4 c0 = codes[0], c1 = codes[1];
        const uint32_t sfw =
            *reinterpret_cast<const uint32_t *>(st_ws(s) + ((r & 31) << 4) + (((r >> 5) & 3) << 2));
        const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        uint8_t *rowp = st_wb(s) + (r >> 3) * 1024 + (r & 7) * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c) {           // 16-byte chunk c = elements 8c .. 8c+7
          uint32_t o[4];
          dequant8(cw[c], e4m3_to_h2((sfw >> (8 * (c >> 1))) & 0xFFu), o);
          *reinterpret_cast<uint4 *>(rowp + ((c ^ swz) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
        }
        fence_proxy_async();                     // generic-proxy writes -> tensor-core reads
        conv_bar();
        if (r == 0) ptx::mbar_arrive(&conv[s]);
        if (++s == STAGES) { s = 0; ph ^= 1u; }
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
    const float alpha = __ldg(p.alpha);
    int it = 0;
    for (int tile = blockIdx.x; tile < tiles; tile += gridDim.x, ++it) {
      const int ab = it & 1;
      if (!ptx::mbar_wait_bounded(&tfull[ab], (uint32_t)((it >> 1) & 1), limit, kTimeoutNs, abort_flag)) {
        give_up();
        break;
      }
      ptx::tc_fence_after();
      const int wt = tile / p.ttiles, tt = tile % p.ttiles;
      const int n = wt * 128 + row;
      const int t0 = tt * NT;
#pragma unroll 1
      for (int c = 0; c < NT / 16; ++c) {
        uint32_t v[16];
        ptx::tmem_ld16(t_row + ab * NT + 16 * c, v);
        ptx::tmem_wait_ld();
        if (n < p.n) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int t = t0 + 16 * c + i;
            if (t < p.m) {
              const __nv_bfloat16 o = __float2bfloat16_rn(alpha * __uint_as_float(v[i]));
              p.d[(size_t)t * p.n + n] = *reinterpret_cast<const uint16_t *>(&o);
            }
          }
        }
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&tempty[ab]);
    }
  }

  __syncthreads();
  if (*abort_flag) {
    if (warp == 0 && issued_mask) {
      for (int s = 0; s < STAGES; ++s)
        if (issued_mask & (1u << s)) {
          volatile int no_abort = 0;
          ptx::mbar_wait_bounded(&full[s], (issued_parity >> s) & 1u, kDrainPolls, 0, &no_abort);
        }
    }
    if (warp == 1 && mma_issued) {
      volatile int no_abort = 0;
      ptx::tc_commit(drain);
      ptx::mbar_wait_bounded(drain, 0, kDrainPolls, 0, &no_abort);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, C::TMEM_COLS);
}

template <int NT>
cudaError_t launch_nt(const uint16_t *x, const uint8_t *w, const uint8_t *wsf, const float *alpha, uint16_t *d,
                      int64_t m, int64_t n, int64_t k, uint32_t wait_limit, cudaStream_t st) {
  using C = Cfg<NT>;
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(w4a16_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  CUtensorMap tm_x, tm_w;
  // activations bf16 [m, k]: box 128 bytes (64 elements) x NT rows, 128-byte swizzle
  // weight codes [n, k/2]: box 32 bytes (64 codes) x 128 rows, no swizzle
  if (!make_byte_map(&tm_x, x, m, k * 2, 128, NT, true) || !make_byte_map(&tm_w, w, n, k / 2, 32, 128, false))
    return cudaErrorInvalidValue;
  W4A16Args a{};
  a.w = w;
  a.wsf = wsf;
  a.alpha = alpha;
  a.d = d;
  a.m = (int32_t)m;
  a.n = (int32_t)n;
  a.k = (int32_t)k;
  a.wtiles = (int32_t)((n + 127) / 128);
  a.ttiles = (int32_t)((m + NT - 1) / NT);
  a.wait_limit = wait_limit;
  a.status = device_status_ptr();
  if (!a.status) return cudaErrorInvalidValue;
  const int tiles = a.wtiles * a.ttiles;
  const int grid = tiles < num_sms() ? tiles : num_sms();
  return launch_pdl(w4a16_kernel<NT>, dim3(grid), dim3(kThreads), C::SMEM_BYTES, st, tm_x, tm_w, a);
}

}  // namespace

bool w4a16_tc_supported(int64_t m, int64_t n, int64_t k) {
  return m > 0 && n > 0 && k > 0 && k % 64 == 0 && n % 32 == 0 && m < (1 << 30) && n < (1 << 30) &&
         k < (1 << 29);
}

cudaError_t launch_w4a16_tc(const uint16_t *x, const uint8_t *w, const uint8_t *wsf, const float *alpha,
                            uint16_t *d, int64_t m, int64_t n, int64_t k, uint32_t wait_limit, cudaStream_t st) {
  if (!w4a16_tc_supported(m, n, k)) return cudaErrorNotSupported;
  if (m <= 16) return launch_nt<16>(x, w, wsf, alpha, d, m, n, k, wait_limit, st);
  if (m <= 32) return launch_nt<32>(x, w, wsf, alpha, d, m, n, k, wait_limit, st);
  if (m <= 64) return launch_nt<64>(x, w, wsf, alpha, d, m, n, k, wait_limit, st);
  if (m <= 128) return launch_nt<128>(x, w, wsf, alpha, d, m, n, k, wait_limit, st);
  return launch_nt<256>(x, w, wsf, alpha, d, m, n, k, wait_limit, st);
}

}  // namespace nvfp4
