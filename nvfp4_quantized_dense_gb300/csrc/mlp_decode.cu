// The whole decode MLP in one persistent kernel: bf16 x -> NVFP4 quantize ->
// gate_up GEMM with the SwiGLU + NVFP4 requantize epilogue -> down_proj GEMM
// -> bf16 ([P1] "关键源码片段", the silu_mul_nvfp4_quantize chain; [P2]
// "实现拆解" item 1, the fused gate_up + SwiGLU + FP4 quantize kernel).
//
// At decode sizes (M <= 64) every step of the chain is bound by the weight
// bytes it streams from HBM; as separate kernels each step pays its own
// launch, pipeline fill and split-K tail, and the weights stop flowing
// between them.  Here one CTA per SM streams its share of the gate_up weights
// and then, without a pause, its share of the down_proj weights, while the
// data-dependent steps meet at arrival counters in the workspace:
//   phase A  every CTA quantizes a slice of x (codes + swizzled scales) and
//            arrives on the x counter;
//   phase B  gate_up as in the swap-AB kernel (weights as the MMA's 128 rows,
//            tokens as its N).  Each CTA first takes a contiguous run of
//            (tile, k-block) pairs of the tiles that are split across CTAs,
//            then whole tiles of its own; the CTA finishing a tile applies
//            SwiGLU, writes that tile's 64 features of h as NVFP4 and counts
//            the tile on its 256-feature slice of h;
//   phase C  down_proj the same way on h, bf16 output.  A stage's h half is
//            issued once the four gate_up tiles of its slice are counted;
//            the slices fed by split gate_up tiles are ready halfway through
//            phase B, and every CTA takes those k-blocks first.
// The producer issues the weight half of every stage at once and defers the
// activation half until its slice is written, so the weight stream runs
// ahead by the whole stage ring across both phase boundaries.
//
// The CTAs must all be resident at once (they wait on each other): the grid
// is at most one CTA per SM and every CTA needs more than half an SM's shared
// memory.  Dependent launches are released only after the x counter is
// complete (every CTA has started), so a following kernel cannot take the SM
// of a CTA that has not started yet.  Every wait is bounded: on a timeout the kernel
// records NVFP4_ERR_DEVICE_TIMEOUT and returns; the workspace then holds
// stale counters and must be zero-filled again before the next call.
//
// Roles per CTA (192 threads): warp 0 TMA producer, warp 1 TMEM owner + MMA
// issuer, warps 2..5 quantize (phase A) and epilogues (TMEM lane = weight
// row).
#include "common.cuh"
#include "internal.h"
#include "splitk.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int BK = 256, KSTEPS = 4;
constexpr uint32_t W_BYTES = 128 * BK / 2;
constexpr uint32_t SFW_BYTES = KSTEPS * 512, SFX_BYTES = KSTEPS * 512;
constexpr int kThreads = 192;
constexpr int ACC_BUFS = 2;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint32_t kDrainPolls = 1u << 22;

template <int NT>
struct Cfg {
  static constexpr uint32_t X_BYTES = NT * BK / 2;
  static constexpr uint32_t STAGE_BYTES = W_BYTES + X_BYTES + SFW_BYTES + SFX_BYTES;
  static constexpr int STAGES = NT == 64 ? 6 : 8;
  static constexpr int PITCH = NT + 1;                      // floats per staged row
  static constexpr uint32_t OUT_BYTES = 128 * PITCH * 4;
  static constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + OUT_BYTES + 1024 + 256;
  static constexpr uint32_t SFW_COL = ACC_BUFS * NT;
  static constexpr uint32_t SFX_COL = SFW_COL + 4 * KSTEPS;
  static constexpr uint32_t USED_COLS = SFX_COL + 4 * KSTEPS;
  static constexpr uint32_t TMEM_COLS = USED_COLS <= 64 ? 64 : USED_COLS <= 128 ? 128 : 256;
  static_assert(STAGE_BYTES % 1024 == 0, "stages must keep 1024-byte alignment");
  static_assert(SMEM_BYTES <= 227 * 1024 && SMEM_BYTES > 116 * 1024, "one CTA per SM");
};

// One GEMM of the chain.
struct Gemm {
  const uint8_t *sfw;   // weight scales, swizzled over the weight rows
  const uint8_t *sfx;   // activation scales, swizzled (one 128-row block)
  float *partials;      // [grid][maxfrag][NT][128] fp32
  int *counters;        // [tiles] split-K arrival counters
  int32_t tiles, kbt, maxfrag, ksteps;   // 128-row tiles, 256-wide k-blocks per tile, K / 64
  int32_t whole, split_tiles;            // work split (MixedPartition)
  int32_t early;                         // k-blocks per tile whose activation slice is written early
};

// Order of a tile's k-blocks within the CTA runs: the `early` k-blocks (those
// whose activation slice is ready first) spread evenly among the others, so
// that every CTA's run holds some of them; a CTA takes the early units of a
// fragment first.
struct KOrder {
  int32_t kbt, early;
};

// Walks the units [u0, u1) of a fragment, the early ones first, giving the
// k-block of each.  Unit u is early when floor((u+1)*early/kbt) exceeds
// floor(u*early/kbt); both counts advance incrementally (one division per
// pass, none per unit: the producer and MMA threads pace the pipeline).
struct KWalk {
  int32_t kbt, early, u0, u1;
  int32_t pass = 0, u = 0, eb = 0, r = 0;
  __device__ __forceinline__ KWalk(const KOrder &ko, int a, int b) : kbt(ko.kbt), early(ko.early), u0(a), u1(b) {
    start();
  }
  __device__ __forceinline__ void start() {
    u = u0;
    eb = u0 * early / kbt;          // early units before u
    r = u0 * early - eb * kbt;      // (u * early) mod kbt
  }
  __device__ __forceinline__ bool next(int &kb) {
    for (;;) {
      if (u >= u1) {
        if (pass == 1) return false;
        pass = 1;
        start();
        continue;
      }
      const bool is_early = r + early >= kbt;
      const int e = eb, cur = u;
      if (is_early) {
        ++eb;
        r += early - kbt;
      } else {
        r += early;
      }
      ++u;
      if (is_early != (pass == 0)) continue;
      kb = is_early ? e : early + (cur - e);
      return true;
    }
  }
};

struct MlpArgs {
  Gemm g[2];            // 0: gate_up (K = hidden), 1: down_proj (K = inter)
  const uint16_t *x;    // bf16 [m, hid]
  const float *gs_x;    // x global scale
  uint8_t *xq, *xs;     // quantized x: codes [m, hid/2], swizzled scales
  const float *alpha_gu, *gs_h;
  uint8_t *h, *hs;      // NVFP4 h: codes [m, inter/2], swizzled scales
  const float *alpha_dn;
  uint16_t *out;        // bf16 [m, hid]
  int32_t m, hid, inter, grid;
  int32_t round_bf16;   // 1: gate_up rounded to bf16 before SwiGLU (the unfused chain)
  uint32_t *sync;       // [0] phase-A arrivals, [1] producers done with every wait
  uint32_t *slice_ready;  // per 256-feature slice of h: gate_up tiles written (of 4)
  uint32_t wait_limit;
  int *status;
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }
__device__ __forceinline__ void named_bar(uint32_t id, uint32_t n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}
__device__ __forceinline__ void red_release_add(uint32_t *p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

template <int NT>
__global__ void __launch_bounds__(kThreads, 1)
    mlp_decode_kernel(const __grid_constant__ CUtensorMap tm_wgu, const __grid_constant__ CUtensorMap tm_xq,
                      const __grid_constant__ CUtensorMap tm_wdn, const __grid_constant__ CUtensorMap tm_h,
                      const MlpArgs p) {
  using C = Cfg<NT>;
  constexpr int STAGES = C::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float *s_out = reinterpret_cast<float *>(base + STAGES * C::STAGE_BYTES);
  uint64_t *full = reinterpret_cast<uint64_t *>(base + STAGES * C::STAGE_BYTES + C::OUT_BYTES);
  uint64_t *empty = full + STAGES;
  uint64_t *tfull = empty + STAGES;
  uint64_t *tempty = tfull + ACC_BUFS;
  uint64_t *drain = tempty + ACC_BUFS;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(drain + 1);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
  volatile int *last_flag = abort_flag + 1;
  auto st_w = [&](int s) { return base + s * C::STAGE_BYTES; };
  auto st_x = [&](int s) { return st_w(s) + W_BYTES; };
  auto st_sfw = [&](int s) { return st_x(s) + C::X_BYTES; };
  auto st_sfx = [&](int s) { return st_sfw(s) + SFW_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < ACC_BUFS; ++b) {
      ptx::mbar_init(&tfull[b], 1);
      ptx::mbar_init(&tempty[b], 128);
    }
    ptx::mbar_init(drain, 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tm_wgu);
    ptx::prefetch_tensormap(&tm_xq);
    ptx::prefetch_tensormap(&tm_wdn);
    ptx::prefetch_tensormap(&tm_h);
  }
  // The producer starts once the barriers exist; the TMEM allocation is
  // waited for only by the MMA and epilogue warps.
  named_bar(2, kThreads);
  uint32_t tmem = 0;
  if (warp != 0) {
    if (warp == 1) {
      ptx::tmem_alloc(tslot, C::TMEM_COLS);
      ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    named_bar(3, kThreads - 32);
    ptx::tc_fence_after();
    tmem = *tslot;
  }

  const MixedPartition part[2] = {{p.g[0].kbt, p.grid, p.g[0].whole, p.g[0].split_tiles},
                                   {p.g[1].kbt, p.grid, p.g[1].whole, p.g[1].split_tiles}};
  const KOrder korder[2] = {{p.g[0].kbt, p.g[0].early}, {p.g[1].kbt, p.g[1].early}};
  // gate_up tiles writing the h slice of down_proj k-block kb
  auto slice_target = [&](int kb) { return (uint32_t)min(4, (p.inter >> 6) - 4 * kb); };
  const uint32_t limit = p.wait_limit;
  uint32_t issued_mask = 0, issued_parity = 0;
  bool mma_issued = false;
  auto give_up = [&]() {
    *abort_flag = 1;
    atomicCAS(p.status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (ptx::elect_one()) {
      const uint64_t pol_w = ptx::l2_policy_evict_first();
      const uint64_t pol_x = ptx::l2_policy_evict_last();
      int s = 0, c = 0;
      uint32_t ph = 0;
      // stages whose activation half waits for the step writing it (FIFO)
      int pend_s[STAGES], pend_kb[STAGES], pend_g[STAGES];
      int head = 0, npend = 0;
      bool x_ready = false, waited_pdl = false, ok = true;
      auto issue_x = [&](int st, int gi, int kb) {
        const Gemm &G = p.g[gi];
        const int nk = min(KSTEPS, G.ksteps - kb * KSTEPS);
        ptx::tma_load_2d(st_x(st), gi == 0 ? &tm_xq : &tm_h, &full[st], kb * (BK / 2), 0, pol_x);
        ptx::bulk_load(st_sfx(st), G.sfx + (size_t)kb * KSTEPS * 512, nk * 512u, &full[st], pol_x);
      };
      // the counter and count that make the activation slice of (gi, kb) ready
      auto ready_ctr = [&](int gi, int kb, uint32_t &target) -> const uint32_t * {
        if (gi == 0) {
          target = (uint32_t)p.grid;
          return &p.sync[0];
        }
        target = slice_target(kb);
        return &p.slice_ready[kb];
      };
      // Is (gi, kb)'s slice written?  (Blocking: wait, bounded; false if that
      // wait gave up.)
      auto check = [&](int gi, int kb, bool block) -> bool {
        if (gi == 0 && x_ready) return true;
        // Before the previous kernel on the stream has completed, its own
        // counts may still sit in the workspace (its last CTAs reset them).
        if (!waited_pdl) return false;
        uint32_t target;
        const uint32_t *ctr = ready_ctr(gi, kb, target);
        bool done = ptx::ld_acquire_gpu(ctr) >= target;
        if (!done && block) done = ptx::counter_wait_bounded(ctr, target, limit, kTimeoutNs, abort_flag);
        if (!done) return false;
        // (each writing thread fenced its generic stores for the async proxy
        // before the release that this acquire observed)
        if (gi == 0) {
          x_ready = true;
          pdl_trigger();                    // every CTA of the grid has started
        }
        return true;
      };
      // Issue the pending activation halves whose slice is written, oldest
      // first; with `block`, wait (bounded) for the oldest.  Returns false
      // only when that wait gave up.
      auto flush = [&](bool block) -> bool {
        for (bool first = true; npend > 0; first = false) {
          if (!check(pend_g[head], pend_kb[head], block && first)) return !(block && first);
          issue_x(pend_s[head], pend_g[head], pend_kb[head]);
          head = head + 1 == STAGES ? 0 : head + 1;
          --npend;
        }
        return true;
      };
      for (int gi = 0; gi < 2 && ok; ++gi) {
        const Gemm &G = p.g[gi];
        const KOrder &ko = korder[gi];
        const CUtensorMap *tm_w = gi == 0 ? &tm_wgu : &tm_wdn;
        MixedIter fi(part[gi], blockIdx.x);
        int tile, u0, u1;
        while (ok && !*abort_flag && fi.next(tile, u0, u1)) {
          KWalk walk(ko, u0, u1);
          for (int kb; ok && walk.next(kb); ++c) {
            // the first STAGES weight stages go out before the previous
            // kernel on the stream has finished
            if (c == STAGES && !waited_pdl) {
              pdl_wait();
              waited_pdl = true;
            }
            flush(false);
            // reusing the stage of a still-pending one needs that one issued
            if (npend == STAGES && !flush(true)) {
              give_up();
              ok = false;
              break;
            }
            if (!ptx::mbar_wait_bounded(&empty[s], ph ^ 1u, limit, kTimeoutNs, abort_flag)) {
              give_up();
              ok = false;
              break;
            }
            const int nk = min(KSTEPS, G.ksteps - kb * KSTEPS);
            ptx::mbar_arrive_expect_tx(&full[s], W_BYTES + C::X_BYTES + 2u * (uint32_t)nk * 512u);
            ptx::tma_load_2d(st_w(s), tm_w, &full[s], kb * (BK / 2), tile * 128, pol_w);
            ptx::bulk_load(st_sfw(s), G.sfw + ((size_t)tile * G.ksteps + kb * KSTEPS) * 512, nk * 512u,
                           &full[s], pol_w);
            if (npend == 0 && check(gi, kb, false)) {
              issue_x(s, gi, kb);
            } else {
              const int e = head + npend < STAGES ? head + npend : head + npend - STAGES;
              pend_s[e] = s;
              pend_kb[e] = kb;
              pend_g[e] = gi;
              ++npend;
            }
            issued_mask |= 1u << s;
            issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
            if (++s == STAGES) { s = 0; ph ^= 1u; }
          }
        }
      }
      if (!waited_pdl) {
        pdl_wait();
        waited_pdl = true;
      }
      while (ok && npend > 0 && !*abort_flag)
        if (!flush(true)) {
          give_up();
          ok = false;
        }
      // After a give-up, still issue the deferred halves (reading whatever
      // the buffers hold): every issued stage's barrier then completes and
      // the drain below is short.
      while (npend > 0) {
        issue_x(pend_s[head], pend_g[head], pend_kb[head]);
        head = head + 1 == STAGES ? 0 : head + 1;
        --npend;
      }
      // This CTA reads no counter any more.  The last CTA to get here resets
      // the phase and slice counters for the next call (every slice count is
      // complete by now: each slice is read by some CTA's producer).
      if (ok && !*abort_flag &&
          atom_add_acq_rel_gpu(reinterpret_cast<int *>(&p.sync[1]), 1) == (uint32_t)p.grid - 1) {
        p.sync[0] = 0;
        for (int kb = 0; kb < p.g[1].kbt; ++kb) p.slice_ready[kb] = 0;
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        p.sync[1] = 0;
      }
    }
  } else if (warp == 1) {
    // ----------------------------------------------------------------- MMA
    pdl_wait();
    if (ptx::elect_one()) {
      // kind::mxf4nvf4, E2M1 x E2M1, UE4M3 scales, M = 128 (weights), N = NT (tokens)
      constexpr uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(NT >> 3) << 17) | (8u << 24);
      int s = 0, it = 0;
      uint32_t ph = 0;
      bool ok = true;
      for (int gi = 0; gi < 2 && ok; ++gi) {
        const Gemm &G = p.g[gi];
        const KOrder &ko = korder[gi];
        MixedIter fi(part[gi], blockIdx.x);
        int tile, u0, u1;
        for (; ok && !*abort_flag && fi.next(tile, u0, u1); ++it) {
          const int ab = it & 1;
          if (!ptx::mbar_wait_bounded(&tempty[ab], (uint32_t)((it >> 1) & 1) ^ 1u, limit, kTimeoutNs,
                                      abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          bool accumulate = false;
          KWalk walk(ko, u0, u1);
          for (int kb; walk.next(kb);) {
            if (!ptx::mbar_wait_bounded(&full[s], ph, limit, kTimeoutNs, abort_flag)) {
              give_up();
              ok = false;
              break;
            }
            ptx::tc_fence_after();
            const int nk = min(KSTEPS, G.ksteps - kb * KSTEPS);
            const uint32_t sfw_s = ptx::smem_u32(st_sfw(s)), sfx_s = ptx::smem_u32(st_sfx(s));
            for (int j = 0; j < nk; ++j) {
              ptx::tmem_cp_32x128b_x4(tmem + C::SFW_COL + 4 * j, ptx::smem_desc(sfw_s + 512 * j, 0, 128, 0));
              ptx::tmem_cp_32x128b_x4(tmem + C::SFX_COL + 4 * j, ptx::smem_desc(sfx_s + 512 * j, 0, 128, 0));
            }
            const uint32_t w_s = ptx::smem_u32(st_w(s)), x_s = ptx::smem_u32(st_x(s));
            for (int j = 0; j < nk; ++j)
              ptx::mma_nvfp4(tmem + ab * NT, ptx::smem_desc(w_s + 32 * j, 16, 1024, 2),
                             ptx::smem_desc(x_s + 32 * j, 16, 1024, 2), idesc, tmem + C::SFW_COL + 4 * j,
                             tmem + C::SFX_COL + 4 * j, accumulate || (j != 0));
            accumulate = true;
            mma_issued = true;
            ptx::tc_commit(&empty[s]);
            if (++s == STAGES) { s = 0; ph ^= 1u; }
          }
          if (!ok) break;
          ptx::tc_commit(&tfull[ab]);
        }
      }
    }
  } else {
    // ------------------------------------------ quantize, then epilogues
    pdl_wait();
    const int q = warp & 3;
    const int r = q * 32 + lane;                 // weight row within the tile
    const int et = threadIdx.x - 64;             // 0..127 across these warps
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
    const int mt = min(p.m, NT);
    bool ok = true;

    // phase A: this CTA's share of x's 16-element blocks, then the padding
    // rows m..127 of the scale block (zero)
    {
      const int cols = p.hid >> 4, cp4 = cols >> 2;
      const float gs = __ldg(p.gs_x);
      const int64_t stride = (int64_t)p.grid * 128;
      for (int64_t b = (int64_t)blockIdx.x * 128 + et; b < (int64_t)p.m * cols; b += stride) {
        const int row = (int)(b / cols), j = (int)(b - (int64_t)row * cols);
        const uint4 *src = reinterpret_cast<const uint4 *>(p.x + (size_t)row * p.hid + 16 * j);
        const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
        float v[16];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[2 * i] = bf16_lo(w[i]);
          v[2 * i + 1] = bf16_hi(w[i]);
        }
        uint32_t lo, hi;
        const uint32_t sf = quantize_block16(v, gs, lo, hi);
        *reinterpret_cast<uint2 *>(p.xq + (size_t)row * (p.hid >> 1) + 8 * j) = make_uint2(lo, hi);
        p.xs[sf_swizzled_offset(row, j, cp4)] = (uint8_t)sf;
      }
      for (int64_t w = (int64_t)blockIdx.x * 128 + et; w < (int64_t)(128 - p.m) * cp4; w += stride) {
        const int row = p.m + (int)(w / cp4), j4 = (int)(w % cp4);
        *reinterpret_cast<uint32_t *>(p.xs + sf_swizzled_offset(row, 4 * j4, cp4)) = 0u;
      }
      ptx::fence_proxy_async_global();
      epi_bar();
      if (et == 0) {
        asm volatile("fence.acq_rel.gpu;" ::: "memory");
        atomicAdd(&p.sync[0], 1u);
      }
    }

    const float alpha_gu = __ldg(p.alpha_gu), alpha_dn = __ldg(p.alpha_dn);
    int it = 0;
    for (int gi = 0; gi < 2 && ok; ++gi) {
      const Gemm &G = p.g[gi];
      const MixedPartition &pt = part[gi];
      MixedIter fi(pt, blockIdx.x);
      int tile, u0, u1;
      for (; fi.next(tile, u0, u1); ++it) {
        const int ab = it & 1;
        const bool got = ptx::mbar_wait_bounded(&tfull[ab], (uint32_t)((it >> 1) & 1), limit, kTimeoutNs,
                                                abort_flag);
        if (!got) give_up();
        if (ptx::bar_any(1, 128, !got || *abort_flag)) {   // the four warps leave together
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        float v[NT];
#pragma unroll
        for (int c = 0; c < NT / 16; ++c) {
          uint32_t raw[16];
          ptx::tmem_ld16(t_row + ab * NT + 16 * c, raw);
          ptx::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) v[16 * c + i] = __uint_as_float(raw[i]);
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&tempty[ab]);

        // split-K: the CTAs sharing this tile meet as in the swap-AB kernel
        const bool split = pt.is_split(tile);
        const int64_t c_first = split ? pt.cta_of((int64_t)tile * G.kbt) : 0;
        const int64_t c_last = split ? pt.cta_of((int64_t)tile * G.kbt + G.kbt - 1) : 0;
        if (c_last > c_first) {
          // partial slot of contributor c: its fragment index is 0 except for
          // c_first (every later contributor's run starts inside this tile)
          const int f_first = tile - (int)(pt.start(c_first) / G.kbt);
          auto slot = [&](int64_t c) {
            return G.partials + ((size_t)c * G.maxfrag + (c == c_first ? f_first : 0)) * NT * 128;
          };
          float *mine = slot(blockIdx.x);
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t < mt) mine[t * 128 + r] = v[t];
          epi_bar();
          if (et == 0)
            *last_flag = atom_add_acq_rel_gpu(&G.counters[tile], 1) == (uint32_t)(c_last - c_first);
          epi_bar();
          if (!*last_flag) continue;
          sum_partials_in_k_order<NT>(v, c_first, c_last, mt, r, slot);
          if (et == 0) G.counters[tile] = 0;
        }

        if (gi == 0) {
          // rows 0..63 of the tile are up, 64..127 gate, for features
          // 64*tile + (0..63) (the gate/up interleave of the weight prep)
#pragma unroll
          for (int t = 0; t < NT; ++t) {
            const float y = alpha_gu * v[t];
            s_out[r * C::PITCH + t] = p.round_bf16 ? __bfloat162float(__float2bfloat16_rn(y)) : y;
          }
          epi_bar();
          // SwiGLU one element per thread; h replaces the up value in s_out
          for (int idx = et; idx < mt * 64; idx += 128) {
            const int t = idx >> 6, i = idx & 63;
            const float g = s_out[(64 + i) * C::PITCH + t], u = s_out[i * C::PITCH + t];
            s_out[i * C::PITCH + t] = p.round_bf16 ? silu_mul(g, u) : silu_mul_fast(g, u);
          }
          epi_bar();
          const int ocp4 = p.inter >> 6;
          const float gs = __ldg(p.gs_h);
          for (int idx = et; idx < mt * 4; idx += 128) {
            const int t = idx >> 2, qb = idx & 3;
            float hv[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) hv[i] = s_out[(16 * qb + i) * C::PITCH + t];
            uint32_t lo, hi;
            const uint32_t sf = quantize_block16(hv, gs, lo, hi);
            const int f = 64 * tile + 16 * qb;
            *reinterpret_cast<uint2 *>(p.h + (size_t)t * (p.inter >> 1) + f / 2) = make_uint2(lo, hi);
            p.hs[sf_swizzled_offset(t, f >> 4, ocp4)] = (uint8_t)sf;
          }
          // padding rows of the 128-row scale block: zero this tile's 4 columns
          for (int t = p.m + et; t < 128; t += 128)
            *reinterpret_cast<uint32_t *>(p.hs + sf_swizzled_offset(t, tile * 4, ocp4)) = 0u;
          ptx::fence_proxy_async_global();     // these stores -> down_proj's TMA reads
          epi_bar();
          if (et == 0) red_release_add(&p.slice_ready[tile >> 2], 1u);
        } else {
          const int n = tile * 128 + r;
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t < mt) {
              const __nv_bfloat16 o = __float2bfloat16_rn(alpha_dn * v[t]);
              p.out[(size_t)t * p.hid + n] = *reinterpret_cast<const uint16_t *>(&o);
            }
        }
      }
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

struct Plan {
  int nt, grid;
  int tiles[2], kbt[2], maxfrag[2], whole[2], split_tiles[2];
  size_t part_bytes[2], counter_bytes, ws_bytes;
};

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

Plan make_plan(int64_t m, int64_t hid, int64_t inter) {
  Plan pl{};
  pl.nt = m <= 16 ? 16 : m <= 32 ? 32 : 64;
  pl.tiles[0] = (int)(2 * inter / 128);
  pl.kbt[0] = (int)((hid + BK - 1) / BK);
  pl.tiles[1] = (int)(hid / 128);
  pl.kbt[1] = (int)((inter + BK - 1) / BK);
  const int64_t w0 = (int64_t)pl.tiles[0] * pl.kbt[0], w1 = (int64_t)pl.tiles[1] * pl.kbt[1];
  int64_t grid = num_sms();
  if (w0 < grid) grid = w0;
  if (w1 < grid) grid = w1;
  pl.grid = (int)grid;
  // sync words, then the h slice counters, then the split-K tile counters
  pl.counter_bytes = kCounterArea;   // sync words, h-slice counters and tile counters fit in it
  pl.ws_bytes = pl.counter_bytes;
  for (int g = 0; g < 2; ++g) {
    pl.whole[g] = (int)(pl.tiles[g] / grid);
    pl.split_tiles[g] = pl.tiles[g] - pl.whole[g] * (int)grid;
    // a shared tile counts every CTA between its first and last owner as a
    // contributor: each CTA must own at least one shared k-block
    if (pl.whole[g] > 0 && pl.split_tiles[g] > 0 && (int64_t)pl.split_tiles[g] * pl.kbt[g] < grid) {
      --pl.whole[g];
      pl.split_tiles[g] += (int)grid;
    }
    const int64_t w = (int64_t)pl.split_tiles[g] * pl.kbt[g];
    const int64_t per = (w + grid - 1) / grid;
    pl.maxfrag[g] = (int)((per + pl.kbt[g] - 1) / pl.kbt[g] + 1);
    pl.part_bytes[g] = round256((size_t)grid * pl.maxfrag[g] * pl.nt * 128 * 4);
    pl.ws_bytes += pl.part_bytes[g];
  }
  return pl;
}

template <int NT>
cudaError_t launch_nt(const Plan &pl, const MlpDecodeParams &q, cudaStream_t st) {
  using C = Cfg<NT>;
  // the shared-memory limit is a setting of each device's context
  static PerDeviceOnce smem_attr;
  if (cudaError_t e = smem_attr.run([] {
        return cudaFuncSetAttribute(mlp_decode_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES);
      }))
    return e;
  // The CTAs wait on each other, so all of them must be resident at once:
  // refuse up front (rather than time out) when the device cannot hold the
  // grid, e.g. when other work or a partition leaves fewer SMs to this kernel.
  int per_sm = 0;
  if (cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, mlp_decode_kernel<NT>, kThreads,
                                                                    C::SMEM_BYTES))
    return e;
  if ((int64_t)per_sm * num_sms() < pl.grid) return cudaErrorCooperativeLaunchTooLarge;
  const int64_t m = q.m, hid = q.hidden, inter = q.inter;
  CUtensorMap tm_wgu, tm_xq, tm_wdn, tm_h;
  // codes [rows, K/2] bytes; box 128 bytes of K x (128 weight rows | NT token rows), 128-byte swizzle
  if (!make_byte_map(&tm_wgu, q.w_gu, 2 * inter, hid / 2, 128, 128, 128) ||
      !make_byte_map(&tm_xq, q.x_fp4, m, hid / 2, 128, NT, 128) ||
      !make_byte_map(&tm_wdn, q.w_dn, hid, inter / 2, 128, 128, 128) ||
      !make_byte_map(&tm_h, q.h_fp4, m, inter / 2, 128, NT, 128))
    return cudaErrorInvalidValue;
  MlpArgs a{};
  uint8_t *ws = static_cast<uint8_t *>(q.workspace);
  a.sync = reinterpret_cast<uint32_t *>(ws);
  a.slice_ready = reinterpret_cast<uint32_t *>(ws + 256);
  int *counters = reinterpret_cast<int *>(ws + 256) + pl.kbt[1];
  uint8_t *parts = ws + pl.counter_bytes;
  for (int g = 0; g < 2; ++g) {
    a.g[g].tiles = pl.tiles[g];
    a.g[g].kbt = pl.kbt[g];
    a.g[g].maxfrag = pl.maxfrag[g];
    a.g[g].whole = pl.whole[g];
    a.g[g].split_tiles = pl.split_tiles[g];
    a.g[g].early = 0;
    a.g[g].counters = counters + (g == 0 ? 0 : pl.tiles[0]);
    a.g[g].partials = reinterpret_cast<float *>(parts + (g == 0 ? 0 : pl.part_bytes[0]));
  }
  a.g[0].sfw = q.w_gu_sf;
  a.g[0].sfx = q.x_sf;
  a.g[0].ksteps = (int32_t)(hid / 64);
  a.g[1].sfw = q.w_dn_sf;
  a.g[1].sfx = q.h_sf;
  a.g[1].ksteps = (int32_t)(inter / 64);
  // down_proj k-blocks whose h slice comes only from split gate_up tiles
  // (tiles [0, split_tiles), finished halfway through the gate_up stream)
  a.g[1].early = pl.split_tiles[0] / 4 < pl.kbt[1] ? pl.split_tiles[0] / 4 : pl.kbt[1];
  a.x = q.x;
  a.gs_x = q.gs_x;
  a.xq = q.x_fp4;
  a.xs = q.x_sf;
  a.alpha_gu = q.alpha_gu;
  a.gs_h = q.gs_h;
  a.h = q.h_fp4;
  a.hs = q.h_sf;
  a.alpha_dn = q.alpha_dn;
  a.out = q.out;
  a.m = (int32_t)m;
  a.hid = (int32_t)hid;
  a.inter = (int32_t)inter;
  a.grid = pl.grid;
  a.round_bf16 = q.round_bf16 ? 1 : 0;
  a.wait_limit = q.wait_limit;
  a.status = device_status_ptr();
  if (!a.status) return cudaErrorInvalidValue;
  return launch_pdl(mlp_decode_kernel<NT>, dim3(pl.grid), dim3(kThreads), C::SMEM_BYTES, st, tm_wgu, tm_xq,
                    tm_wdn, tm_h, a);
}

}  // namespace

bool mlp_decode_supported(int64_t m, int64_t hidden, int64_t inter) {
  if (!(m >= 1 && m <= 64 && hidden >= 128 && hidden % 128 == 0 && inter >= 64 && inter % 64 == 0 &&
        hidden < (1 << 24) && inter < (1 << 24)))
    return false;
  // sync words, then one counter per down_proj k-block (h slice) and per tile of both GEMMs
  const int64_t words = 64 + (inter + BK - 1) / BK + 2 * inter / 128 + hidden / 128;
  return words <= kCounterSlots;
}

size_t mlp_decode_workspace_bytes(int64_t m, int64_t hidden, int64_t inter) {
  if (!mlp_decode_supported(m, hidden, inter)) return 0;
  return make_plan(m, hidden, inter).ws_bytes;
}

cudaError_t launch_mlp_decode(const MlpDecodeParams &q, cudaStream_t st) {
  if (!mlp_decode_supported(q.m, q.hidden, q.inter)) return cudaErrorNotSupported;
  const Plan pl = make_plan(q.m, q.hidden, q.inter);
  if (q.ws_bytes < pl.ws_bytes) return cudaErrorInvalidValue;
  if (pl.nt == 16) return launch_nt<16>(pl, q, st);
  if (pl.nt == 32) return launch_nt<32>(pl, q, st);
  return launch_nt<64>(pl, q, st);
}

}  // namespace nvfp4
