// W4A16 GEMM on the tensor cores: bf16 activations x NVFP4 weights
// ([P3] fp4_gemm with quant_mode "w4a16": the activation is not quantized,
// alpha holds only the weight dequant factor).  This is the kernel for
// calls without a workspace; with one the TMEM kernel (gemm_w4a16_tmem.cu)
// runs instead.  (Its split-K planning below still serves that case's
// whole-tile grid.)
//
// The tensor cores need both operands of a kind::f16 MMA in the same type,
// so the weight is dequantized to bf16 in shared memory: converter warps read
// a k-block's E2M1 codes and E4M3 scales and write E2M1 * scale -- exact in
// bf16, at most 6 significant bits -- into 128-byte-swizzled K-major tiles
// (one per 64-wide sub-block) that the MMA reads directly.  The weight is the MMA's 128-row operand and
// the tokens its N (16..256); D^T[n, t] accumulates in TMEM (two buffers) and
// the epilogue writes D[t, n] with the 32 lanes of a warp on 32 consecutive n.
//
// Two rings: raw k-blocks (weight codes and scales from HBM plus the
// k-block's activation tile) and dequantized weight tiles.  A raw stage is
// released by the MMA (it reads the activation tile there), a dequantized
// tile likewise.  A k-block is 128 wide up to 32 tokens (9 KB of weight
// codes and scales, a 32 KB dequantized tile filled by a pair of converter
// warps) and 64 wide above: at decode sizes every k-block costs each role a
// barrier round, so wider k-blocks halve that cost per weight byte.
//
// Work split: as in the swap-AB kernel, the (weight tile, k-block)
// pairs are cut into one contiguous run per CTA when the caller gives a
// workspace -- always up to 64 tokens, and for more tokens when whole tiles
// would leave more than 20 % of the SMs' rounds idle (e.g. 40 weight tiles of
// a 5120-row down_proj on 152 SMs: measured 104 -> 60 us at 128 tokens; at
// 89 % fill the reductions cost more than they save); a tile shared by CTAs
// is finished by the
// last to arrive, which sums the fp32 partials in K order.  Otherwise every
// CTA owns whole tiles.
//
// Roles (512 threads, one CTA per SM): warp 0 TMA producer, warp 1 TMEM owner
// + MMA issuer, warps 2..9 converters, warps 10..13 epilogue, warp 14 second
// MMA issuer, warp 15 second producer.  At decode sizes a single thread that
// loads, or issues the MMAs of, every k-block is the bound (a barrier wait
// costs ~170 cycles even when the phase is complete, a small MMA ~50, a
// commit ~45), so up to 128 tokens the k-blocks of the CTA's sequence
// alternate between two producers and two issuers; each issuer accumulates
// into its own TMEM columns and the epilogue adds the two.  Bounded waits as
// in gemm_tc.cu.
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "splitk.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {
namespace {

constexpr uint32_t SUB_WB = 128 * 64 * 2;  // dequantized 64-wide sub-block of a tile, 16 KB
constexpr int kConvWarps = 8;               // converter warps
constexpr int kConvThreads = 32 * kConvWarps;
constexpr int kWarpMma2 = 2 + kConvWarps + 4;   // second MMA issuer
constexpr int kWarpProd2 = kWarpMma2 + 1;       // second producer
constexpr int kThreads = 64 + kConvThreads + 128 + 64;
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint32_t kDrainPolls = 1u << 22;

template <int NT>
struct Cfg {
  // K per k-block (the unit of the work split and of every barrier round):
  // 128 up to 32 tokens, where the barrier waits, copies, commits and MMA
  // issues of each k-block bound the kernel; 64 above.  A k-block is SUB
  // 64-wide sub-blocks, each one 128-byte-swizzle atom column of the
  // dequantized tile and of the activation tile.
  static constexpr int BK = NT <= 32 ? 128 : 64;
  static constexpr int SUB = BK / 64;
  static constexpr uint32_t WC_BYTES = 128 * BK / 2;                     // weight codes, 64-byte rows
  static constexpr uint32_t WS_BYTES = SUB * 512;                        // 128x4 scale tiles
  static constexpr uint32_t WB_BYTES = SUB * SUB_WB;                     // dequantized tile
  static constexpr uint32_t SUB_X = NT * 128;                            // NT rows x 128 B
  static constexpr uint32_t X_BYTES = SUB * SUB_X;
  static constexpr uint32_t RAW_BYTES = (X_BYTES + WC_BYTES + WS_BYTES + 1023) / 1024 * 1024;
  // Up to 64 tokens the converter warps dequantize whole k-blocks, WPT warps
  // per tile (k-block j -> tile j % DSTAGES): many k-blocks in flight for the
  // weight stream.  Above, every warp takes 16 rows of every k-block: short
  // latency per k-block for the compute-bound MMA.
  static constexpr bool WHOLE_KB = NT <= 64;
  static constexpr int WPT = !WHOLE_KB ? kConvWarps : SUB == 2 ? 2 : 1;   // converter warps per tile
  static constexpr int DSTAGES = NT <= 32 ? 4 : NT == 64 ? 6 : 4;         // dequantized tiles
  static_assert(!WHOLE_KB || DSTAGES * WPT <= kConvWarps, "converter warps per dequantized tile");
  static constexpr int NI = NT <= 128 ? 2 : 1;                             // MMA issuers
  static constexpr int RSTAGES_FIT = (int)((220u * 1024 - DSTAGES * WB_BYTES) / RAW_BYTES) / NI * NI;
  static constexpr int RSTAGES = RSTAGES_FIT > 32 ? 32 : RSTAGES_FIT;   // raw k-blocks in flight
  // issuer i takes the k-blocks j with j % NI == i: with both ring depths
  // multiples of NI every ring barrier serves one issuer, in order
  static_assert(RSTAGES % NI == 0 && DSTAGES % NI == 0, "ring barriers per issuer");
  static_assert(RSTAGES >= DSTAGES, "raw ring at least as deep as the dequantized one");
  static constexpr uint32_t BAR_BYTES = 1024;
  static constexpr uint32_t SMEM_BYTES = DSTAGES * WB_BYTES + RSTAGES * RAW_BYTES + BAR_BYTES + 1024;
  static constexpr uint32_t ACC_COLS = 2 * NI * NT;                       // two tiles x NI issuers
  static constexpr uint32_t TMEM_COLS = ACC_COLS <= 32 ? 32 : ACC_COLS <= 64 ? 64 : ACC_COLS <= 128 ? 128 : ACC_COLS <= 256 ? 256 : 512;
  static_assert(ACC_COLS <= 512, "TMEM columns");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert(RSTAGES >= 4, "pipeline depth");
  static_assert((2 * RSTAGES + 2 * DSTAGES + 6) * 8 + 16 <= BAR_BYTES, "barrier area");
};

struct W4A16Args {
  const uint8_t *wsf;      // swizzled scales over N rows
  const float *alpha;
  uint16_t *d;             // bf16 [M, N]
  float *partials;         // [grid][maxfrag][NT][128] fp32 (tiles shared by CTAs)
  int *counters;           // [tiles] arrival counters
  int32_t m, n, k;
  int32_t wtiles, ttiles, nkb;
  int32_t grid, maxfrag, split_ok;
  uint32_t wait_limit;
  int *status;
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Eight codes (one 32-bit word) times one E4M3 scale -> four bf16x2, exact:
// E2M1 -> f16x2, times the scale in f16 (product within f16's normal range and
// precision), widened to f32 and rounded to bf16 (no rounding happens: the
// values have at most 6 significant bits).
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
__global__ void __launch_bounds__(kThreads, 1)   // 16 warps: at most 128 registers
    w4a16_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                 const W4A16Args p) {
  using C = Cfg<NT>;
  constexpr int RST = C::RSTAGES;
  constexpr int DSTAGES = C::DSTAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  constexpr int BK = C::BK, SUB = C::SUB;
  auto st_wb = [&](int d) { return base + d * C::WB_BYTES; };
  auto st_x = [&](int r) { return base + DSTAGES * C::WB_BYTES + r * C::RAW_BYTES; };
  auto st_wc = [&](int r) { return st_x(r) + C::X_BYTES; };
  auto st_ws = [&](int r) { return st_wc(r) + C::WC_BYTES; };
  uint64_t *rfull = reinterpret_cast<uint64_t *>(base + DSTAGES * C::WB_BYTES + RST * C::RAW_BYTES);
  uint64_t *rempty = rfull + RST;
  uint64_t *dfull = rempty + RST;
  uint64_t *dempty = dfull + DSTAGES;
  uint64_t *tfull = dempty + DSTAGES;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(drain + 2);   // drain: one per issuer
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
  volatile int *last_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int r = 0; r < RST; ++r) {
      ptx::mbar_init(&rfull[r], 1);
      ptx::mbar_init(&rempty[r], 1);
    }
    for (int d = 0; d < DSTAGES; ++d) {
      ptx::mbar_init(&dfull[d], C::WPT);   // arrivals of the warps filling it
      ptx::mbar_init(&dempty[d], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&tfull[b], C::NI);      // one commit per issuer
      ptx::mbar_init(&tempty[b], 128);
      ptx::mbar_init(&drain[b], 1);
    }
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
  const int cp4 = p.k >> 6;              // 512-byte scale tiles per 128-row block
  // 64-wide sub-blocks of k-block kb (the last k-block may hold fewer)
  auto nsub_of = [&](int kb) { return min(SUB, cp4 - kb * SUB); };
  const Partition part{(int64_t)tiles * p.nkb, p.grid, p.nkb, p.split_ok == 0, tiles};
  const int64_t my_start = part.start(blockIdx.x), my_end = part.start(blockIdx.x + 1);
  const uint32_t limit = p.wait_limit;
  uint32_t issued_mask = 0, issued_parity = 0;
  bool mma_issued = false;
  auto give_up = [&]() {
    *abort_flag = 1;
    atomicCAS(p.status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
  };

  if (warp == 0 || warp == kWarpProd2) {
    // ----------------------------------------------------------- producers
    // producer p fills the raw stages of the k-blocks j with j % NI == p
    const int prod = warp == 0 ? 0 : 1;
    if (prod < C::NI && ptx::elect_one()) {
      const uint64_t pol_w = ptx::l2_policy_evict_first();
      const uint64_t pol_x = ptx::l2_policy_evict_last();
      int r = 0, j = 0;
      uint32_t ph = 0;
      // The raw stages of the first RST k-blocks get their weight codes and
      // scales before the previous kernel on the stream has finished; their
      // activation tiles follow once it has.
      int pend_r[RST], pend_kb[RST], pend_tt[RST];
      int npend = 0;
      bool flushed = false;
      auto load_x = [&](int st, int kb, int tt) {
        // one 128-byte-swizzled NT x 128 B tile per sub-block (a sub-block
        // past K reads zeros)
#pragma unroll
        for (int sb = 0; sb < SUB; ++sb)
          ptx::tma_load_2d(st_x(st) + sb * C::SUB_X, &tm_x, &rfull[st], (kb * SUB + sb) * 128, tt * NT, pol_x);
      };
      auto flush = [&]() {
        pdl_wait();
        for (int i = 0; i < npend; ++i) load_x(pend_r[i], pend_kb[i], pend_tt[i]);
        flushed = true;
      };
      FragIter fi{my_start, my_end, p.nkb};
      int tile, kb0, kb1;
      bool ok = true;
      while (ok && !*abort_flag && fi.next(tile, kb0, kb1)) {
        const int wt = tile / p.ttiles, tt = tile - wt * p.ttiles;
        for (int kb = kb0; kb < kb1; ++kb, ++j) {
          if (C::NI == 1 || (j & 1) == prod) {
            // a stage is reused only after this producer's own earlier
            // activation tiles are in flight
            if (j >= RST && !flushed) flush();
            if (!ptx::mbar_wait_bounded(&rempty[r], ph ^ 1u, limit, kTimeoutNs, abort_flag)) {
              give_up();
              ok = false;
              break;
            }
            const uint32_t sfb = (uint32_t)nsub_of(kb) * 512u;   // scales only of the sub-blocks K has
            ptx::mbar_arrive_expect_tx(&rfull[r], C::X_BYTES + C::WC_BYTES + sfb);
            ptx::tma_load_2d(st_wc(r), &tm_w, &rfull[r], kb * (BK / 2), wt * 128, pol_w);
            ptx::bulk_load(st_ws(r), p.wsf + ((size_t)wt * cp4 + kb * SUB) * 512, sfb, &rfull[r], pol_w);
            if (j < RST) {
              pend_r[npend] = r;
              pend_kb[npend] = kb;
              pend_tt[npend] = tt;
              ++npend;
            } else {
              load_x(r, kb, tt);
            }
            issued_mask |= 1u << r;
            issued_parity = (issued_parity & ~(1u << r)) | (ph << r);
          }
          if (++r == RST) { r = 0; ph ^= 1u; }
        }
      }
      if (!flushed) flush();
    }
  } else if (warp == 1 || warp == kWarpMma2) {
    // ----------------------------------------------------------------- MMA
    const int issuer = warp == 1 ? 0 : 1;
    pdl_wait();
    if (issuer < C::NI && ptx::elect_one()) {
      // kind::f16: F32 accumulator (bits 4-5 = 1), A = B = BF16 (1), K-major,
      // N >> 3 in bits 17-22, M = 128 >> 4 in bits 24-28
      constexpr uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(NT >> 3) << 17) | (8u << 24);
      int r = 0, d = 0, it = 0, j = 0;
      uint32_t dph = 0;
      auto advance = [&]() {
        ++j;
        if (++d == DSTAGES) { d = 0; dph ^= 1u; }
        if (++r == RST) r = 0;
      };
      FragIter fi{my_start, my_end, p.nkb};
      int tile, kb0, kb1;
      bool ok = true;
      for (; ok && !*abort_flag && fi.next(tile, kb0, kb1); ++it) {
        const int ab = it & 1;
        if (!ptx::mbar_wait_bounded(&tempty[ab], (uint32_t)((it >> 1) & 1) ^ 1u, limit, kTimeoutNs, abort_flag)) {
          give_up();
          break;
        }
        ptx::tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)((ab * C::NI + issuer) * NT);
        bool first = true;
        for (int kb = kb0; kb < kb1; ++kb, advance()) {
          if (C::NI > 1 && (j & 1) != issuer) continue;
          // the converters filled the tile after they saw the raw stage,
          // activation tile included, complete: no wait on the stage here
          if (!ptx::mbar_wait_bounded(&dfull[d], dph, limit, kTimeoutNs, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t wb = ptx::smem_u32(st_wb(d)), xs = ptx::smem_u32(st_x(r));
          const int nsub = nsub_of(kb);
          for (int sb = 0; sb < nsub; ++sb)
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
              ptx::mma_bf16(acc, ptx::smem_desc(wb + sb * SUB_WB + 32 * jj, 16, 1024, 2),
                            ptx::smem_desc(xs + sb * C::SUB_X + 32 * jj, 16, 1024, 2), idesc,
                            !first || sb != 0 || jj != 0);
          first = false;
          mma_issued = true;
          ptx::tc_commit(&dempty[d]);
          ptx::tc_commit(&rempty[r]);
        }
        if (!ok) break;
        ptx::tc_commit(&tfull[ab]);          // also when this issuer had no k-block of the tile
      }
    }
  } else if (warp < 2 + kConvWarps) {
    // ---------------------------------------------------------- converters
    pdl_wait();
    const int cw = warp - 2;
    // whole k-blocks: warp cw fills tile cw / WPT, rows [part*RPW, (part+1)*RPW)
    constexpr int RPW = 128 / (C::WHOLE_KB ? C::WPT : 1);
    const int dt = cw / C::WPT, part = cw % C::WPT;
    FragIter fi{my_start, my_end, p.nkb};
    int tile, kb0, kb1;
    int j = 0;                                  // index of the k-block in this CTA's sequence
    bool ok = !C::WHOLE_KB || dt < DSTAGES;     // spare warps have no tile
    // A warp walks its k-blocks in order and waits for its tile's release
    // before the raw stage (RSTAGES >= DSTAGES), so no barrier parity is
    // ambiguous; no barrier joins the converter warps.
    while (ok && fi.next(tile, kb0, kb1)) {
      for (int kb = kb0; kb < kb1; ++kb, ++j) {
        if (C::WHOLE_KB && j % DSTAGES != dt) continue;
        const int r = j % RST, d = j % DSTAGES;
        const uint32_t rph = (uint32_t)((j / RST) & 1), dph = (uint32_t)((j / DSTAGES) & 1);
        bool got = ptx::mbar_wait_bounded(&dempty[d], dph ^ 1u, limit, kTimeoutNs, abort_flag);
        if (got) got = ptx::mbar_wait_bounded(&rfull[r], rph, limit, kTimeoutNs, abort_flag);
        if (__any_sync(0xffffffffu, !got)) {   // the warp leaves together
          give_up();
          ok = false;
          break;
        }
        const int nsub = nsub_of(kb);
        if constexpr (C::WHOLE_KB) {
          // the warp's RPW rows of each 64-wide sub-block, in steps of 16
          // rows; lane pair (2i, 2i+1) takes the two 32-code halves of row
          // part*RPW + 16s + i, so that every load instruction reads 512
          // contiguous bytes.  All loads of a sub-block first (the compiler
          // cannot move them past the tile stores); the 16-byte scale row q
          // holds the scales of rows q, q+32, q+64, q+96.
          constexpr int STEPS = RPW / 16;
          const int hf = lane & 1, i = lane >> 1;
          for (int sb = 0; sb < nsub; ++sb) {
            uint4 cv[STEPS];
#pragma unroll
            for (int s8 = 0; s8 < STEPS; ++s8)
              cv[s8] = *reinterpret_cast<const uint4 *>(st_wc(r) + (part * RPW + 16 * s8 + i) * (BK / 2) + sb * 32 +
                                                        hf * 16);
            const uint4 sa = *reinterpret_cast<const uint4 *>(st_ws(r) + sb * 512 + i * 16);
            const uint4 sz = *reinterpret_cast<const uint4 *>(st_ws(r) + sb * 512 + (16 + i) * 16);
#pragma unroll
            for (int s8 = 0; s8 < STEPS; ++s8) {
              const int row = part * RPW + 16 * s8 + i;
              const uint4 &sv = (s8 & 1) ? sz : sa;          // row & 31 is i or 16 + i
              const int comp = (row >> 5) & 3;
              const uint32_t sfw = comp == 0 ? sv.x : comp == 1 ? sv.y : comp == 2 ? sv.z : sv.w;
              const uint32_t cwd[4] = {cv[s8].x, cv[s8].y, cv[s8].z, cv[s8].w};
              uint8_t *rowp = st_wb(d) + sb * SUB_WB + (row >> 3) * 1024 + (row & 7) * 128;
              const int swz = row & 7;
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int c = 4 * hf + u;       // 16-byte chunk c = elements 8c .. 8c+7
                uint32_t o[4];
                dequant8(cwd[u], e4m3_to_h2((sfw >> (8 * (c >> 1))) & 0xFFu), o);
                *reinterpret_cast<uint4 *>(rowp + ((c ^ swz) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
              }
            }
          }
        } else {
          // 16 rows of the tile (one 64-wide sub-block: BK = 64 here): two
          // lanes per row, 32 elements each
          static_assert(C::WHOLE_KB || SUB == 1, "row-split converters take 64-wide k-blocks");
          const int row = 16 * cw + (lane >> 1), hf = lane & 1;
          const uint4 cv = *reinterpret_cast<const uint4 *>(st_wc(r) + row * (BK / 2) + hf * 16);
          const uint32_t sfw =
              *reinterpret_cast<const uint32_t *>(st_ws(r) + ((row & 31) << 4) + (((row >> 5) & 3) << 2));
          const uint32_t cwd[4] = {cv.x, cv.y, cv.z, cv.w};
          uint8_t *rowp = st_wb(d) + (row >> 3) * 1024 + (row & 7) * 128;
          const int swz = row & 7;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int c = 4 * hf + i;
            uint32_t o[4];
            dequant8(cwd[i], e4m3_to_h2((sfw >> (8 * (c >> 1))) & 0xFFu), o);
            *reinterpret_cast<uint4 *>(rowp + ((c ^ swz) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          }
        }
        fence_proxy_async();                     // generic-proxy writes -> tensor-core reads
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&dfull[d]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int et = threadIdx.x - (64 + kConvThreads);
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
    const float alpha = __ldg(p.alpha);
    constexpr int TG = 16;                       // tokens summed per pass of the reduction
    int it = 0, j0 = 0;                          // j0: index of the fragment's first k-block
    // 16 accumulator columns of tile buffer ab, summed over the issuers that
    // had a k-block of the fragment (warp-uniform)
    auto load_acc = [&](int ab, int c, bool p0, bool p1, float (&o)[16]) {
      uint32_t v[16], w[16];
      const uint32_t a0 = t_row + (uint32_t)(ab * C::NI * NT + 16 * c);
      if (p0) ptx::tmem_ld16(a0, v);
      if (C::NI > 1 && p1) ptx::tmem_ld16(a0 + NT, w);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 16; ++i)
        o[i] = (p0 ? __uint_as_float(v[i]) : 0.0f) + ((C::NI > 1 && p1) ? __uint_as_float(w[i]) : 0.0f);
    };
    FragIter fi{my_start, my_end, p.nkb};
    int tile, kb0, kb1;
    for (; fi.next(tile, kb0, kb1); ++it, j0 += kb1 - kb0) {
      const int ab = it & 1;
      const bool got = ptx::mbar_wait_bounded(&tfull[ab], (uint32_t)((it >> 1) & 1), limit, kTimeoutNs, abort_flag);
      if (!got) give_up();
      if (ptx::bar_any(2, 128, !got || *abort_flag)) break;   // the four warps leave together
      ptx::tc_fence_after();
      const int wt = tile / p.ttiles, tt = tile - wt * p.ttiles;
      const int n = wt * 128 + row;
      const int t0 = tt * NT;
      const int mt = min(p.m - t0, NT);
      const int64_t c_first = part.cta_of((int64_t)tile * p.nkb);
      const int64_t c_last = part.cta_of((int64_t)tile * p.nkb + p.nkb - 1);
      const bool p0 = C::NI == 1 || (j0 & 1) == 0 || kb1 - kb0 >= 2;
      const bool p1 = C::NI > 1 && ((j0 & 1) == 1 || kb1 - kb0 >= 2);
      if (c_last == c_first) {
        // the whole tile is this CTA's: straight to the output
#pragma unroll 1
        for (int c = 0; c < NT / 16; ++c) {
          float v[16];
          load_acc(ab, c, p0, p1, v);
          if (n < p.n) {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const int tk = 16 * c + i;
              if (tk < mt) {
                const __nv_bfloat16 o = __float2bfloat16_rn(alpha * v[i]);
                p.d[(size_t)(t0 + tk) * p.n + n] = *reinterpret_cast<const uint16_t *>(&o);
              }
            }
          }
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&tempty[ab]);
        continue;
      }
      // shared tile: this CTA's fp32 partial to the workspace; the last
      // contributor to arrive sums all of them in K order
      // partial slot of contributor cc: its fragment index is 0 except for
      // c_first (every later contributor's run starts inside this tile)
      const int f_first = tile - (int)(part.start(c_first) / p.nkb);
      auto slot = [&](int64_t cc) {
        return p.partials + ((size_t)cc * p.maxfrag + (cc == c_first ? f_first : 0)) * NT * 128;
      };
      float *mine = slot(blockIdx.x);
#pragma unroll 1
      for (int c = 0; c < NT / 16; ++c) {
        float v[16];
        load_acc(ab, c, p0, p1, v);
#pragma unroll
        for (int i = 0; i < 16; ++i)
          if (16 * c + i < mt) mine[(16 * c + i) * 128 + row] = v[i];
      }
      ptx::tc_fence_before();
      ptx::mbar_arrive(&tempty[ab]);
      epi_bar();                    // every partial write of the CTA precedes the release below
      if (et == 0)
        *last_flag = atom_add_acq_rel_gpu(&p.counters[tile], 1) == (uint32_t)(c_last - c_first);
      epi_bar();
      if (!*last_flag) continue;
      if (et == 0) p.counters[tile] = 0;
#pragma unroll 1
      for (int g0 = 0; g0 < mt; g0 += TG) {
        float acc[TG];
#pragma unroll
        for (int i = 0; i < TG; ++i) acc[i] = 0.0f;
        for (int64_t cc = c_first; cc <= c_last; ++cc) {       // K order
          const float *pc = slot(cc) + (size_t)g0 * 128 + row;
          float tmp[TG];
#pragma unroll
          for (int i = 0; i < TG; ++i) tmp[i] = (g0 + i < mt) ? __ldcg(pc + i * 128) : 0.0f;
#pragma unroll
          for (int i = 0; i < TG; ++i) acc[i] += tmp[i];
        }
        if (n < p.n) {
#pragma unroll
          for (int i = 0; i < TG; ++i)
            if (g0 + i < mt) {
              const __nv_bfloat16 o = __float2bfloat16_rn(alpha * acc[i]);
              p.d[(size_t)(t0 + g0 + i) * p.n + n] = *reinterpret_cast<const uint16_t *>(&o);
            }
        }
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    if ((warp == 0 || warp == kWarpProd2) && issued_mask) {
      for (int r = 0; r < RST; ++r)
        if (issued_mask & (1u << r)) {
          volatile int no_abort = 0;
          ptx::mbar_wait_bounded(&rfull[r], (issued_parity >> r) & 1u, kDrainPolls, 0, &no_abort);
        }
    }
    if ((warp == 1 || warp == kWarpMma2) && mma_issued) {
      volatile int no_abort = 0;
      uint64_t *dr = &drain[warp == 1 ? 0 : 1];
      ptx::tc_commit(dr);
      ptx::mbar_wait_bounded(dr, 0, kDrainPolls, 0, &no_abort);
    }
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, C::TMEM_COLS);
}

int pick_nt(int64_t m) { return m <= 16 ? 16 : m <= 32 ? 32 : m <= 64 ? 64 : m <= 128 ? 128 : 256; }

// Work split of one call: split-K over (tile, k-block) pairs for up to 64
// tokens (one token tile), and above when whole tiles fill less than 80 % of
// the rounds of one CTA per SM; whole tiles otherwise.
struct Plan {
  int nt, wtiles, ttiles, nkb, grid, maxfrag;
  bool can_split;
  size_t ws_bytes;   // workspace the split needs (0: none)
};

Plan make_plan(int64_t m, int64_t n, int64_t k) {
  Plan pl{};
  pl.nt = pick_nt(m);
  pl.wtiles = (int)((n + 127) / 128);
  pl.ttiles = (int)((m + pl.nt - 1) / pl.nt);
  const int bk = pl.nt <= 32 ? Cfg<16>::BK : Cfg<64>::BK;   // k-block width of the token tile
  pl.nkb = (int)((k + bk - 1) / bk);                         // the last one may be 64 wide
  const int tiles = pl.wtiles * pl.ttiles;
  const int sms = num_sms();
  const int64_t rounds = (tiles + sms - 1) / sms;
  pl.can_split = (pl.nt <= 64 || (int64_t)tiles * 100 < rounds * sms * 80) && tiles <= kCounterSlots;
  if (pl.can_split) {
    const int64_t w = (int64_t)tiles * pl.nkb;
    pl.grid = (int)(w < num_sms() ? w : num_sms());
    const int64_t per = (w + pl.grid - 1) / pl.grid;
    pl.maxfrag = (int)((per + pl.nkb - 1) / pl.nkb + 1);
    const bool shared = (w % pl.grid != 0) || ((w / pl.grid) % pl.nkb != 0);
    pl.ws_bytes = shared ? kCounterArea + (size_t)pl.grid * pl.maxfrag * pl.nt * 128 * 4 : 0;
  } else {
    pl.grid = tiles < num_sms() ? tiles : num_sms();
  }
  return pl;
}

template <int NT>
cudaError_t launch_nt(const Plan &pl, const uint16_t *x, const uint8_t *w, const uint8_t *wsf, const float *alpha,
                      uint16_t *d, int64_t m, int64_t n, int64_t k, void *ws, size_t ws_bytes, uint32_t wait_limit,
                      cudaStream_t st) {
  using C = Cfg<NT>;
  // the shared-memory limit is a setting of each device's context
  static PerDeviceOnce smem_attr;
  if (cudaError_t e = smem_attr.run([] {
        return cudaFuncSetAttribute(w4a16_kernel<NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES);
      }))
    return e;
  CUtensorMap tm_x, tm_w;
  // activations bf16 [m, k]: box 128 bytes (64 elements) x NT rows, 128-byte swizzle
  // weight codes [n, k/2]: box BK/2 bytes x 128 rows, no swizzle
  if (!make_byte_map(&tm_x, x, m, k * 2, 128, NT, 128) || !make_byte_map(&tm_w, w, n, k / 2, C::BK / 2, 128, 0))
    return cudaErrorInvalidValue;
  W4A16Args a{};
  a.wsf = wsf;
  a.alpha = alpha;
  a.d = d;
  a.m = (int32_t)m;
  a.n = (int32_t)n;
  a.k = (int32_t)k;
  a.wtiles = pl.wtiles;
  a.ttiles = pl.ttiles;
  a.nkb = pl.nkb;
  const bool split = pl.can_split && (pl.ws_bytes == 0 || (ws != nullptr && ws_bytes >= pl.ws_bytes));
  if (split) {
    a.grid = pl.grid;
    a.maxfrag = pl.maxfrag;
    a.split_ok = 1;
    if (pl.ws_bytes) {
      a.counters = static_cast<int *>(ws);
      a.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + kCounterArea);
    }
  } else {
    const int tiles = pl.wtiles * pl.ttiles;
    a.grid = tiles < num_sms() ? tiles : num_sms();
    a.maxfrag = 1;
    a.split_ok = 0;
  }
  a.wait_limit = wait_limit;
  a.status = device_status_ptr();
  if (!a.status) return cudaErrorInvalidValue;
  return launch_pdl(w4a16_kernel<NT>, dim3(a.grid), dim3(kThreads), C::SMEM_BYTES, st, tm_x, tm_w, a);
}

}  // namespace

bool w4a16_tc_supported(int64_t m, int64_t n, int64_t k) {
  return m > 0 && n > 0 && k > 0 && k % 64 == 0 && n % 32 == 0 && m < (1 << 30) && n < (1 << 30) &&
         k < (1 << 29);
}

size_t w4a16_workspace_bytes(int64_t m, int64_t n, int64_t k) {
  if (!w4a16_tc_supported(m, n, k)) return 0;
  if (w4a16_tmem_supported(m, n, k)) return w4a16_tmem_workspace_bytes(m, n, k);
  return make_plan(m, n, k).ws_bytes;
}

bool w4a16_uses_tmem(int64_t m, int64_t n, int64_t k, const void *ws, size_t ws_bytes) {
  return w4a16_tmem_supported(m, n, k) && ws != nullptr && ws_bytes >= w4a16_tmem_workspace_bytes(m, n, k);
}

cudaError_t launch_w4a16_tc(const uint16_t *x, const uint16_t *pre_scale, const uint8_t *w, const uint8_t *wsf,
                            const float *alpha, uint16_t *d, int64_t m, int64_t n, int64_t k, void *ws,
                            size_t ws_bytes, uint32_t wait_limit, cudaStream_t st) {
  if (!w4a16_tc_supported(m, n, k)) return cudaErrorNotSupported;
  if (w4a16_uses_tmem(m, n, k, ws, ws_bytes))
    return launch_w4a16_tmem(x, pre_scale, w, wsf, alpha, d, m, n, k, ws, ws_bytes, wait_limit, st);
  if (pre_scale) return cudaErrorInvalidValue;   // the caller scales the activations for this kernel
  const Plan pl = make_plan(m, n, k);
  switch (pl.nt) {
    case 16: return launch_nt<16>(pl, x, w, wsf, alpha, d, m, n, k, ws, ws_bytes, wait_limit, st);
    case 32: return launch_nt<32>(pl, x, w, wsf, alpha, d, m, n, k, ws, ws_bytes, wait_limit, st);
    case 64: return launch_nt<64>(pl, x, w, wsf, alpha, d, m, n, k, ws, ws_bytes, wait_limit, st);
    case 128: return launch_nt<128>(pl, x, w, wsf, alpha, d, m, n, k, ws, ws_bytes, wait_limit, st);
    default: return launch_nt<256>(pl, x, w, wsf, alpha, d, m, n, k, ws, ws_bytes, wait_limit, st);
  }
}

}  // namespace nvfp4
