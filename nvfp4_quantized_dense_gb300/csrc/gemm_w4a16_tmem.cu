// W4A16 GEMM on the tensor cores: bf16 activations x NVFP4 weights ([P3]
// fp4_gemm with quant_mode "w4a16"), the dequantized weight tiles held in
// tensor memory; 16/32/64-token tiles on one CTA (decode), 128-token tiles on
// CTA pairs.
//
// Why TMEM.  A 128-row x 128-wide block of weights is 9 KB of codes and
// scales in HBM but 32 KB once dequantized to 16 bits.  Written to shared
// memory and read back by the MMA it costs 64 KB of shared-memory traffic per
// 9 KB streamed, more than an SM's shared memory carries at its share of the
// HBM bandwidth.  Here each converter thread dequantizes one weight row into
// registers and stores it with tcgen05.st into TMEM, and the MMA takes its A
// operand (the weights, M = 128) from there; only the activations (B, N = the
// token tile) come from shared memory.
//
// Operand type f16.  E2M1 -> f16 is one conversion per two codes and the
// UE4M3 scale one f16x2 multiply, both exact: the product has at most 6
// significant bits and lies in f16's normal range (2^-11 .. 2688).  A
// pre-pass turns each token row of the bf16 activations into f16 times a
// power of two 2^e that brings the row's largest finite magnitude into
// [2^15, 2^16): every element within 2^30 of that magnitude converts
// exactly (smaller ones are f16 subnormals, rounded by at most 2^-25 in the
// scaled units).  The MMA's products and fp32 sums are then those of the bf16
// operands times 2^e, and the epilogue applies alpha and then 2^-e, so the
// output is the bf16 computation's (a power-of-two scale commutes with every
// rounding, barring underflow).
//
// Pipeline.  A k-block is 256 wide: the weight codes arrive as 128-byte rows
// (whole 128-byte lines per weight row and request; 64-byte rows measured
// about 72 % of the copy bandwidth in steady state), 128-byte swizzled so
// that a thread reads its own row without bank conflicts.  Weights (codes and
// the 128x4 scale tiles) and the f16 activation tiles travel in rings of
// their own: a weight stage is released as soon as the converters hold its
// codes in registers, so nearly the whole weight ring is in flight from HBM,
// and the weights stream (and are dequantized into TMEM) while the
// activation pre-pass is still running.  A k-block is dequantized in two
// 128-wide halves into 64-column TMEM slots after the accumulators.
//
// Work split (as the swap-AB kernel's mixed split): every CTA owns `whole`
// whole weight tiles, done last so that no CTA ends its run with a
// reduction; the other tiles are cut into one contiguous run of (tile,
// k-block) pairs per CTA, a tile shared by CTAs finished by the last to
// arrive, which sums the fp32 partials in K order.
//
// Roles (768 threads, one CTA per SM): warp 0 weight producer, warp 3
// activation producer, warps 1 (also TMEM owner) and 2 the MMA issuers of
// halves 0 and 1 at decode sizes (one thread issuing every MMA would bound
// the kernel; 128-token tiles: warp 1 alone), each accumulating into its own
// TMEM columns; warps 4..19
// converters, one per (half, 64-wide quarter, TMEM lane quarter): warp w
// writes TMEM lanes 32(w%4) .. 32(w%4)+31 (the lanes a warp may access), one
// weight row per thread, and every converter warp visits every k-block, so
// no ring barrier's phase is ambiguous (conversion is latency-bound: four
// converter warps per SM sub-partition hide what two cannot); warps 20..23
// epilogue, adding the two issuers' accumulators.  Every wait is bounded as
// in the other tensor-core kernels.
#include <cfloat>
#include <cuda_fp16.h>

#include "common.cuh"
#include "internal.h"
#include "splitk.cuh"
#include "tc_ptx.cuh"

namespace nvfp4 {
namespace {

constexpr int kThreads = 768;
constexpr int kWarpProdW = 0, kWarpMma0 = 1, kWarpMma1 = 2, kWarpProdX = 3;
constexpr int kFirstConv = 4;
constexpr int kFirstEpi = kFirstConv + 16;   // warps 20..23
constexpr uint64_t kTimeoutNs = 2000000000ull;
constexpr uint32_t kDrainPolls = 1u << 22;
constexpr uint64_t kSettleNs = 20000;      // abort path of a pair: the partner's copies land meanwhile

// Two configurations, both with 256-wide k-blocks of 128-byte code rows,
// each dequantized in two halves into TMEM slots of 64 columns by 16
// converter warps, one per (half, 64-wide quarter, TMEM lane quarter).  Up to
// 64 tokens (weight streaming) two MMA issuers take the halves, with a
// full/empty barrier pair per half.  128-token tiles run on CTA pairs (256
// weight rows, the tokens split 64/64 between the two CTAs' shared memory)
// with one issuer and one barrier pair per k-block: a barrier wait or a
// commit of the issuing thread costs about as much as an MMA at N = 128, and
// the tensor pipe idles while it runs, so the fewer per MMA the better.
template <int NT, bool PAIR = false>
struct TCfg {
  static_assert(!PAIR || NT == 128, "CTA pairs take 128-token tiles");
  static constexpr int CL = PAIR ? 2 : 1;                       // CTAs per tile
  static constexpr bool DECODE = NT <= 64;
  static constexpr int BK = 256;                                // K per k-block
  static constexpr int SUB = BK / 64;                           // 64-wide sub-blocks (one scale tile each)
  static constexpr int CPQ = BK / 128;                          // 32-element code chunks per quarter
  static constexpr int NI = DECODE ? 2 : 1;                     // MMA issuers
  static constexpr uint32_t CODE_ROW = BK / 2;                  // code bytes of a weight row per k-block
  static constexpr int XROWS = NT / CL;                         // token rows staged by one CTA
  static constexpr uint32_t SUB_X = XROWS * 128;                // XROWS rows x 64 f16, 128-byte swizzle
  static constexpr uint32_t X_BYTES = SUB * SUB_X;              // one activation stage
  static constexpr uint32_t WC_BYTES = 128 * CODE_ROW;
  static constexpr uint32_t WS_BYTES = SUB * 512;               // 128x4 scale tiles
  static constexpr uint32_t W_BYTES = WC_BYTES + WS_BYTES;      // one weight stage (a multiple of 1024)
  static constexpr int XSTAGES = NT <= 32 ? 4 : NT == 64 ? 3 : PAIR ? 4 : 2;
  static constexpr uint32_t BAR_BYTES = 1024;
  static constexpr int WSTAGES_FIT = (int)((224u * 1024 - XSTAGES * X_BYTES - BAR_BYTES - 1024) / W_BYTES);
  static constexpr int WSTAGES = WSTAGES_FIT > 16 ? 16 : WSTAGES_FIT;
  static constexpr uint32_t ACC_COLS = 2 * NI * NT;             // two tile buffers x the issuers
  static constexpr uint32_t A_COLS = BK / 4;                    // f16 pairs of one half k-block row
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr int DSTAGES = (int)((TMEM_COLS - ACC_COLS) / A_COLS) / 2 * 2;
  static constexpr uint32_t SMEM_BYTES = XSTAGES * X_BYTES + WSTAGES * W_BYTES + BAR_BYTES + 1024;
  static_assert(W_BYTES % 1024 == 0 && X_BYTES % 1024 == 0, "stage alignment for the swizzles");
  static_assert(DSTAGES >= 2 && DSTAGES % 2 == 0, "dequantized halves: slot parity = half");
  static_assert(WSTAGES >= 4, "weight ring depth");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
  static_assert((2 * WSTAGES + 2 * XSTAGES + 2 * DSTAGES + 6) * 8 + 16 <= BAR_BYTES, "barrier area");
  static_assert(ACC_COLS + 2 * A_COLS <= TMEM_COLS, "TMEM columns");
};

struct TArgs {
  const uint8_t *wsf;      // swizzled scales over N rows
  const float *alpha;
  const float *rs;         // [m] 2^-e of each token row
  uint16_t *d;             // bf16 [M, N]
  float *partials;         // [grid][maxfrag][NT][128] fp32 (tiles shared by CTAs)
  int *counters;           // [split tiles] arrival counters
  int32_t m, n, k;
  int32_t wtiles, ttiles, nkb;   // tile t = weight tile t / ttiles, token tile t % ttiles
  int32_t grid, maxfrag, whole, split_tiles;
  uint32_t wait_limit;
  int *status;
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// A split tile's sum handed out in chunks (128-token tiles): chunk c covers
// token rows 8 (c >> 2) .. +7 and weight rows 32 (c & 3) .. +31 of the
// tile.  The epilogue posts the task; its own warps and every converter warp
// that has finished dequantizing take chunks through `word` = generation
// (bits 16-31) | chunk count (8-15) | chunks handed out (0-7), so one atomic
// returns a chunk index together with the post it belongs to.
struct SumTask {
  int64_t c_first, c_last;
  int32_t tile, t0, mt, f_first;
  uint32_t word;
  int32_t done;          // chunks finished
  int32_t stop;          // the epilogue has no more tiles
  int32_t idle;          // converter warps done dequantizing (taking chunks)
  int32_t use;           // this sum is posted in chunks (else the epilogue sums alone)
};

// Eight E2M1 codes (one word, element i in nibble i) times an f16x2 scale ->
// four f16x2 (elements 2i, 2i+1 in word i, the lower index in the low half).
__device__ __forceinline__ void dequant8_f16(uint32_t codes, uint32_t scale_h2, uint32_t *out) {
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
  for (int i = 0; i < 4; ++i) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[i]) : "r"(h[i]), "r"(scale_h2));
}

// Two UE4M3 scale bytes (low byte first) -> each one as f16 in both halves.
__device__ __forceinline__ void scales_to_h2(uint32_t two, uint32_t &s0, uint32_t &s1) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"((uint16_t)two));
  s0 = __byte_perm(r, 0, 0x1010);
  s1 = __byte_perm(r, 0, 0x3232);
}

template <int NT, bool PAIR>
__global__ void __launch_bounds__(kThreads, 1)
    w4a16_tmem_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_w,
                      const TArgs p) {
  using C = TCfg<NT, PAIR>;
  constexpr int WST = C::WSTAGES, XST = C::XSTAGES, DST = C::DSTAGES;
  constexpr int BK = C::BK, SUB = C::SUB, NI = C::NI, CPQ = C::CPQ, CL = C::CL;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *base = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  auto st_x = [&](int r) { return base + r * C::X_BYTES; };
  auto st_wc = [&](int r) { return base + XST * C::X_BYTES + r * C::W_BYTES; };
  auto st_ws = [&](int r) { return st_wc(r) + C::WC_BYTES; };
  uint64_t *wfull = reinterpret_cast<uint64_t *>(base + XST * C::X_BYTES + WST * C::W_BYTES);
  uint64_t *wempty = wfull + WST;
  uint64_t *xfull = wempty + WST;
  uint64_t *xempty = xfull + XST;
  uint64_t *dfull = xempty + XST;
  uint64_t *dempty = dfull + DST;
  uint64_t *tfull = dempty + DST;
  uint64_t *tempty = tfull + 2;
  uint64_t *drain = tempty + 2;
  uint32_t *tslot = reinterpret_cast<uint32_t *>(drain + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
  volatile int *last_flag = abort_flag + 1;
  SumTask *task = reinterpret_cast<SumTask *>((reinterpret_cast<uintptr_t>(last_flag + 1) + 15) & ~uintptr_t(15));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // In a pair, rank 0 (the leader) issues the pair's MMAs and owns the
  // barriers that both CTAs' activation copies and dequantized slots
  // complete on; the leader's commits release both CTAs' stages.
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  auto in_cta = [&](const void *v, uint32_t r) { return ptx::map_to_cta(ptx::smem_u32(v), r); };
  const int cluster = blockIdx.x / CL;
  // One chunk of the posted split-tile sum (128-token tiles): thread `lane`
  // of the calling warp adds weight row 32 (ch & 3) + lane of token rows
  // 8 (ch >> 2) .. +7 over the tile's contributors in K order and stores
  // them as bf16(alpha * v * 2^-e).
  auto sum_chunk = [&](int ch) {
    constexpr int TGC = 8, MAXC = 2;
    const int row = 32 * (ch & 3) + (int)(threadIdx.x & 31), g0 = TGC * (ch >> 2);
    const int64_t c_first = task->c_first, c_last = task->c_last;
    const int tl = task->tile, t0 = task->t0, mt = task->mt, f_first = task->f_first;
    const int n = ((tl / p.ttiles) * CL + (int)rank) * 128 + row;
    auto slot = [&](int64_t cc) {
      return p.partials + (((size_t)cc * p.maxfrag + (cc == c_first ? f_first : 0)) * CL + rank) * NT * 128;
    };
    float acc[TGC];
#pragma unroll
    for (int x = 0; x < TGC; ++x) acc[x] = 0.0f;
    for (int64_t c0 = c_first; c0 <= c_last; c0 += MAXC) {
      float pv[MAXC][TGC];
#pragma unroll
      for (int u = 0; u < MAXC; ++u) {
        const bool have = c0 + u <= c_last;
        const float *pc = slot(have ? c0 + u : c0) + (size_t)g0 * 128 + row;
#pragma unroll
        for (int x = 0; x < TGC; ++x) pv[u][x] = (have && g0 + x < mt) ? __ldcg(pc + x * 128) : 0.0f;
      }
#pragma unroll
      for (int u = 0; u < MAXC; ++u)
        if (c0 + u <= c_last) {
#pragma unroll
          for (int x = 0; x < TGC; ++x) acc[x] += pv[u][x];
        }
    }
    if (n < p.n) {
      const float alpha = __ldg(p.alpha);
#pragma unroll
      for (int x = 0; x < TGC; ++x)
        if (g0 + x < mt) {
          const __nv_bfloat16 o = __float2bfloat16_rn(alpha * acc[x] * __ldg(p.rs + t0 + g0 + x));
          p.d[(size_t)(t0 + g0 + x) * p.n + n] = *reinterpret_cast<const uint16_t *>(&o);
        }
    }
  };
  // Take chunks of the current post until none is left; returns the
  // generation of the post the last grab belonged to.
  auto take_chunks = [&]() {
    for (;;) {
      uint32_t old = 0;
      if ((threadIdx.x & 31) == 0) old = atomicAdd(&task->word, 1u);
      old = __shfl_sync(0xffffffffu, old, 0);
      if ((old & 0xFFu) >= ((old >> 8) & 0xFFu)) return old >> 16;
      __threadfence_block();                 // the fields of that post
      sum_chunk((int)(old & 0xFFu));
      __syncwarp();
      if ((threadIdx.x & 31) == 0) atomicAdd(&task->done, 1);
    }
  };
  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int r = 0; r < WST; ++r) {
      ptx::mbar_init(&wfull[r], 1);
      ptx::mbar_init(&wempty[r], 16);      // every converter warp, once it holds its codes
    }
    for (int r = 0; r < XST; ++r) {
      ptx::mbar_init(&xfull[r], 1);
      ptx::mbar_init(&xempty[r], NI);      // one commit per issuer
    }
    for (int d = 0; d < DST; ++d) {
      // per half (two issuers): its eight converter warps; per k-block (one
      // issuer): all sixteen (of both CTAs of a pair)
      ptx::mbar_init(&dfull[d], (NI == 2 ? 8 : 16) * CL);
      ptx::mbar_init(&dempty[d], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&tfull[b], NI);       // one commit per issuer
      ptx::mbar_init(&tempty[b], 4 * CL);  // one arrival per epilogue warp (of the pair)
      ptx::mbar_init(&drain[b], 1);
    }
    *abort_flag = 0;
    task->word = 0;
    task->done = 0;
    task->stop = 0;
    task->idle = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tm_x);
    ptx::prefetch_tensormap(&tm_w);
  }
  // The weight producer (warp 0, whose thread 0 initialized the barriers)
  // starts streaming at once; the others wait until the barriers and the
  // TMEM allocation are in place.
  uint32_t tmem = 0;
  if constexpr (PAIR) {
    // both CTAs' barriers and the pair's TMEM exist before any remote arrival
    if (warp == kWarpMma0) {
      ptx::tmem_alloc_pair(tslot, C::TMEM_COLS);
      ptx::tmem_relinquish_pair();
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    tmem = *tslot;
  } else if (warp == kWarpProdW) {
    __syncwarp();
    asm volatile("bar.arrive 1, %0;" ::"r"(kThreads) : "memory");
  } else {
    if (warp == kWarpMma0) {
      ptx::tmem_alloc(tslot, C::TMEM_COLS);
      ptx::tmem_relinquish();
    }
    ptx::tc_fence_before();
    asm volatile("bar.sync 1, %0;" ::"r"(kThreads) : "memory");
    ptx::tc_fence_after();
    tmem = *tslot;
  }
  auto a_col = [&](int d) { return C::ACC_COLS + (uint32_t)d * C::A_COLS; };

  const int cp4 = p.k >> 6;              // 512-byte scale tiles per 128-row block
  auto nsub_of = [&](int kb) { return min(SUB, cp4 - kb * SUB); };
  // 64-wide sub-blocks of half h of k-block kb (0 .. SUB/2)
  auto nsub_half = [&](int kb, int h) { return min(SUB / 2, max(0, nsub_of(kb) - (SUB / 2) * h)); };
  const MixedPartition mixed{p.nkb, p.grid, p.whole, p.split_tiles};
  const uint32_t limit = p.wait_limit;
  uint32_t issued_w = 0, issued_w_par = 0, issued_x = 0, issued_x_par = 0;
  bool mma_issued = false;
  auto give_up = [&]() {
    *abort_flag = 1;
    atomicCAS(p.status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
    if constexpr (PAIR) ptx::st_cluster_u32(in_cta(const_cast<const int *>(abort_flag), rank ^ 1u), 1u);
  };

  if (warp == kWarpProdW) {
    // ---------------------------------------------------- weight producer
    if (ptx::elect_one()) {
      // a weight tile read once (one token tile) need not stay in L2; with
      // several token tiles the cluster reads it again for each, back to back
      const uint64_t pol_w = p.ttiles == 1 ? ptx::l2_policy_evict_first() : ptx::l2_policy_evict_normal();
      int r = 0;
      uint32_t ph = 0;
      MixedIter mi(mixed, cluster);
      int tile, kb0, kb1;
      bool ok = true;
      while (ok && !*abort_flag && mi.next(tile, kb0, kb1)) {
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_bounded(&wempty[r], ph ^ 1u, limit, kTimeoutNs, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          const uint32_t sfb = (uint32_t)nsub_of(kb) * 512u;   // scales only of the sub-blocks K has
          const int rb = (tile / p.ttiles) * CL + (int)rank;      // this CTA's 128-row weight block
          if (rb * 128 < p.n) {
            ptx::mbar_arrive_expect_tx(&wfull[r], C::WC_BYTES + sfb);
            ptx::tma_load_2d(st_wc(r), &tm_w, &wfull[r], kb * (BK / 2), rb * 128, pol_w);
            ptx::bulk_load(st_ws(r), p.wsf + ((size_t)rb * cp4 + kb * SUB) * 512, sfb, &wfull[r], pol_w);
          } else {
            ptx::mbar_arrive(&wfull[r]);   // rows past N (the pair's second half): nothing to load
          }
          issued_w |= 1u << r;
          issued_w_par = (issued_w_par & ~(1u << r)) | (ph << r);
          if (++r == WST) { r = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp == kWarpProdX) {
    // ------------------------------------------------ activation producer
    pdl_wait();                          // the pre-pass wrote the f16 activations
    if (ptx::elect_one()) {
      const uint64_t pol_x = ptx::l2_policy_evict_last();
      int r = 0;
      uint32_t ph = 0;
      MixedIter mi(mixed, cluster);
      int tile, kb0, kb1;
      bool ok = true;
      while (ok && !*abort_flag && mi.next(tile, kb0, kb1)) {
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_bounded(&xempty[r], ph ^ 1u, limit, kTimeoutNs, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          // this CTA's XROWS token rows; in a pair both halves land on the leader's barrier
          if (leader) ptx::mbar_arrive_expect_tx(&xfull[r], CL * C::X_BYTES);
          const int x_row = (tile % p.ttiles) * NT + (int)rank * C::XROWS;
#pragma unroll
          for (int sb = 0; sb < SUB; ++sb) {  // a sub-block past K reads zeros
            if (PAIR && !leader)
              ptx::tma_load_2d_to_pair_bar(st_x(r) + sb * C::SUB_X, &tm_x, in_cta(&xfull[r], 0),
                                           (kb * SUB + sb) * 128, x_row, pol_x);
            else
              ptx::tma_load_2d(st_x(r) + sb * C::SUB_X, &tm_x, &xfull[r], (kb * SUB + sb) * 128, x_row, pol_x);
          }
          if (leader) {   // (a pair partner's copies complete on the leader's barrier)
            issued_x |= 1u << r;
            issued_x_par = (issued_x_par & ~(1u << r)) | (ph << r);
          }
          if (++r == XST) { r = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp == kWarpMma0 || warp == kWarpMma1) {
    // ----------------------------------------------------------------- MMA
    // issuer hi issues the halves h of every k-block with h % NI == hi
    const int hi = warp == kWarpMma0 ? 0 : 1;
    // commit: the MMAs so far have completed -> arrive on this barrier (of both CTAs of a pair)
    auto commit = [&](uint64_t *bar) {
      if constexpr (PAIR) {
        ptx::tc_commit_pair(ptx::smem_u32(bar));
        ptx::tc_commit_pair(in_cta(bar, 1));
      } else {
        ptx::tc_commit(bar);
      }
    };
    if (leader && hi < NI && ptx::elect_one()) {
      // kind::f16: F32 accumulator (bits 4-5 = 1), A = B = F16 (0), K-major,
      // N >> 3 in bits 17-22, M (128 per CTA) >> 4 in bits 24-28
      constexpr uint32_t idesc = (1u << 4) | ((uint32_t)(NT >> 3) << 17) | ((uint32_t)(8 * CL) << 24);
      int xr = 0, it = 0, i = 0;
      uint32_t xph = 0;
      MixedIter mi(mixed, cluster);
      int tile, kb0, kb1;
      bool ok = true;
      for (; ok && !*abort_flag && mi.next(tile, kb0, kb1); ++it) {
        const int ab = it & 1;
        if (!ptx::mbar_wait_bounded(&tempty[ab], (uint32_t)((it >> 1) & 1) ^ 1u, limit, kTimeoutNs, abort_flag)) {
          give_up();
          break;
        }
        ptx::tc_fence_after();
        const uint32_t acc = tmem + (uint32_t)((ab * NI + hi) * NT);
        bool first = true;
        for (int kb = kb0; kb < kb1 && ok; ++kb, ++i) {
          if (!ptx::mbar_wait_bounded(&xfull[xr], xph, limit, kTimeoutNs, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          // one issuer: both halves' slots are ready together (one barrier per k-block)
          const int ek = (2 * i) % DST;
          const uint32_t eph = (uint32_t)(((2 * i) / DST) & 1);
          if (NI == 1) {
            if (!ptx::mbar_wait_bounded(&dfull[ek >> 1], eph, limit, kTimeoutNs, abort_flag)) {
              give_up();
              ok = false;
              break;
            }
            ptx::tc_fence_after();
          }
#pragma unroll
          for (int h = hi; h < 2; h += NI) {
            const int j = 2 * i + h, d = j % DST;
            const uint32_t dph = (uint32_t)((j / DST) & 1);
            if (NI == 2) {
              if (!ptx::mbar_wait_bounded(&dfull[d], dph, limit, kTimeoutNs, abort_flag)) {
                give_up();
                ok = false;
                break;
              }
              ptx::tc_fence_after();
            }
            const uint32_t xs = ptx::smem_u32(st_x(xr)) + (uint32_t)(h * (SUB / 2)) * C::SUB_X;
            const uint32_t wa = tmem + a_col(d);
            const int ns = nsub_half(kb, h);
            for (int sb = 0; sb < ns; ++sb)
#pragma unroll
              for (int jj = 0; jj < 4; ++jj) {
                const uint64_t bd = ptx::smem_desc(xs + sb * C::SUB_X + 32 * jj, 16, 1024, 2);
                if constexpr (PAIR)
                  ptx::mma_f16_tmem_a_pair(acc, wa + 8 * (4 * sb + jj), bd, idesc, !first);
                else
                  ptx::mma_f16_tmem_a(acc, wa + 8 * (4 * sb + jj), bd, idesc, !first);
                first = false;
              }
            mma_issued = true;
            if (NI == 2) commit(&dempty[d]);
          }
          if (!ok) break;
          if (NI == 1) commit(&dempty[ek >> 1]);
          commit(&xempty[xr]);
          if (++xr == XST) { xr = 0; xph ^= 1u; }
        }
        if (!ok) break;
        commit(&tfull[ab]);                  // also when this issuer had nothing to add
      }
    }
  } else if (warp < kFirstEpi) {
    // ---------------------------------------------------------- converters
    // warp (h, qt, q): half h, its quarter qt (CPQ 32-element chunks starting
    // at chunk (2h + qt) * CPQ of the k-block; TMEM columns (A_COLS / 2) * qt
    // .. of the half's slot), TMEM lanes 32 q ..  A half's slot has the
    // half's parity (DST is even).
    const int cg = (warp - kFirstConv) >> 2;
    const int h = cg >> 1, qt = cg & 1, q = warp & 3;
    const int chunk0 = (2 * h + qt) * CPQ;    // first code chunk of the quarter
    const int sb = chunk0 >> 1;               // its 64-wide sub-block
    const int row = 32 * q + lane;
    const uint32_t t_lane = tmem + ((uint32_t)(32 * q) << 16) + (C::A_COLS / 2) * qt;
    // chunk c of the row sits at c ^ swz: 128-byte swizzle (128-byte rows) or 64-byte (64-byte rows)
    const int swz = C::CODE_ROW == 128 ? (row & 7) : ((row >> 1) & 3);
    const uint32_t sf_off = (uint32_t)(sb * 512 + (row & 31) * 16 + (row >> 5) * 4);
    const uint32_t c_off = (uint32_t)(row * C::CODE_ROW);
    MixedIter mi(mixed, cluster);
    int tile, kb0, kb1;
    int i = 0, wr = 0;
    uint32_t wph = 0;
    bool ok = true;
    while (ok && mi.next(tile, kb0, kb1)) {
      for (int kb = kb0; kb < kb1; ++kb, ++i) {
        const int j = 2 * i + h, d = j % DST;
        const uint32_t dph = (uint32_t)((j / DST) & 1);
        const int bi = NI == 2 ? d : d >> 1;   // its slot's barriers: per half, or per k-block
        bool got = ptx::mbar_wait_bounded(&dempty[bi], dph ^ 1u, limit, kTimeoutNs, abort_flag);
        if (got) got = ptx::mbar_wait_bounded(&wfull[wr], wph, limit, kTimeoutNs, abort_flag);
        if (__any_sync(0xffffffffu, !got)) {   // the warp leaves together
          give_up();
          ok = false;
          break;
        }
        const bool have = sb < nsub_of(kb);    // this quarter holds some of K
        const uint8_t *crow = st_wc(wr) + c_off;
        uint4 cv[CPQ];
#pragma unroll
        for (int c = 0; c < CPQ; ++c)
          cv[c] = *reinterpret_cast<const uint4 *>(crow + (((chunk0 + c) ^ swz) << 4));
        const uint32_t sw = *reinterpret_cast<const uint32_t *>(st_ws(wr) + sf_off);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&wempty[wr]);   // the stage's codes are read (release)
        if (++wr == WST) { wr = 0; wph ^= 1u; }
        if (have) {
#pragma unroll
          for (int c = 0; c < CPQ; ++c) {
            // chunk chunk0 + c: 32 elements, scales 2 (chunk & 1) and 2 (chunk & 1) + 1 of the sub-block
            uint32_t s0, s1;
            scales_to_h2(sw >> (16 * ((chunk0 + c) & 1)), s0, s1);
            uint32_t o[16];
            dequant8_f16(cv[c].x, s0, o);
            dequant8_f16(cv[c].y, s0, o + 4);
            dequant8_f16(cv[c].z, s1, o + 8);
            dequant8_f16(cv[c].w, s1, o + 12);
            ptx::tmem_st16(t_lane + a_col(d) + 16 * c, o);
          }
          ptx::tmem_wait_st();
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if (PAIR && !leader) ptx::mbar_arrive_remote(in_cta(&dfull[bi], 0));
          else ptx::mbar_arrive(&dfull[bi]);
        }
      }
    }
    if constexpr (NT == 128) {
      // Done dequantizing: take chunks of the split-tile sums the epilogue
      // posts from now on, until it has no more tiles (bounded wait).
      if (lane == 0) atomicAdd(&task->idle, 1);
      uint32_t seen = 0, polls = 0;
      uint64_t w0 = 0;
      while (ok) {
        if ((*reinterpret_cast<volatile uint32_t *>(&task->word) >> 16) != seen) {
          seen = take_chunks();
          polls = 0;
          w0 = 0;
          continue;
        }
        if (*reinterpret_cast<volatile int *>(&task->stop) || *abort_flag) break;
        ++polls;
        bool late = limit && polls >= limit;
        if (!limit && (polls & 63u) == 0) {
          const uint64_t now = ptx::globaltimer();
          if (w0 == 0) w0 = now;
          else late = now - w0 > kTimeoutNs;
        }
        if (__any_sync(0xffffffffu, late)) {   // the warp leaves together
          give_up();
          break;
        }
        __nanosleep(128);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();
    const int q = warp & 3;
    const int row = q * 32 + lane;
    const int et = threadIdx.x - 32 * kFirstEpi;
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
    const float alpha = __ldg(p.alpha);
    constexpr int TG = 16;                   // tokens per pass
    constexpr int MAXC = 2;                  // contributors' partials loaded together
    int it = 0;
    auto load_acc = [&](int ab, int c, bool p1, float (&o)[16]) {
      uint32_t v[16];
      const uint32_t a0 = t_row + (uint32_t)(ab * NI * NT + 16 * c);
      ptx::tmem_ld16(a0, v);
      ptx::tmem_wait_ld();
#pragma unroll
      for (int x = 0; x < 16; ++x) o[x] = __uint_as_float(v[x]);
      if (p1) {
        ptx::tmem_ld16(a0 + NT, v);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 16; ++x) o[x] += __uint_as_float(v[x]);
      }
    };
    // accumulator buffer ab read: free it for the next tile (the leader's barrier in a pair)
    auto release_acc = [&](int ab) {
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (PAIR && !leader) ptx::mbar_arrive_remote(in_cta(&tempty[ab], 0));
        else ptx::mbar_arrive(&tempty[ab]);
      }
    };
    // bf16(alpha * v * 2^-e) of token row t (< m)
    auto out_bits = [&](float v, int t) {
      const __nv_bfloat16 o = __float2bfloat16_rn(alpha * v * __ldg(p.rs + t));
      return *reinterpret_cast<const uint16_t *>(&o);
    };
    MixedIter mi(mixed, cluster);
    int tile, kb0, kb1;
    uint32_t gen = 0;                        // posts of split-tile sums (thread et == 0)
    for (; mi.next(tile, kb0, kb1); ++it) {
      const int ab = it & 1;
      const bool got = ptx::mbar_wait_bounded(&tfull[ab], (uint32_t)((it >> 1) & 1), limit, kTimeoutNs, abort_flag);
      if (!got) give_up();
      if (ptx::bar_any(2, 128, !got || *abort_flag)) break;   // the four warps leave together
      ptx::tc_fence_after();
      const int n = ((tile / p.ttiles) * CL + (int)rank) * 128 + row;
      const int t0 = (tile % p.ttiles) * NT;  // first token row of the tile
      const int mt = min(p.m - t0, NT);
      const bool p1 = NI > 1 && nsub_of(kb0) > SUB / 2;   // issuer 1 added half 1 of some k-block
      const bool split_tile = mixed.is_split(tile);
      const int64_t c_first = split_tile ? mixed.cta_of((int64_t)tile * p.nkb) : cluster;
      const int64_t c_last = split_tile ? mixed.cta_of((int64_t)tile * p.nkb + p.nkb - 1) : cluster;
      if (c_last == c_first) {
#pragma unroll 1
        for (int c = 0; c < NT / 16; ++c) {
          float v[16];
          load_acc(ab, c, p1, v);
          if (n < p.n) {
#pragma unroll
            for (int x = 0; x < 16; ++x)
              if (16 * c + x < mt) p.d[(size_t)(t0 + 16 * c + x) * p.n + n] = out_bits(v[x], t0 + 16 * c + x);
          }
        }
        release_acc(ab);
        continue;
      }
      // partial slot of contributor cc: its fragment index is 0 except for
      // c_first (every later contributor's run starts inside this tile)
      const int f_first = tile - (int)(mixed.start(c_first) / p.nkb);
      auto slot = [&](int64_t cc) {
        return p.partials + (((size_t)cc * p.maxfrag + (cc == c_first ? f_first : 0)) * CL + rank) * NT * 128;
      };
      float *mine = slot(cluster);
#pragma unroll 1
      for (int c = 0; c < NT / 16; ++c) {
        float v[16];
        load_acc(ab, c, p1, v);
#pragma unroll
        for (int x = 0; x < 16; ++x)
          if (16 * c + x < mt) mine[(16 * c + x) * 128 + row] = v[x];
      }
      release_acc(ab);
      epi_bar();                    // every partial write of the CTA precedes the release below
      if (et == 0)
        *last_flag = atom_add_acq_rel_gpu(&p.counters[tile * CL + (int)rank], 1) == (uint32_t)(c_last - c_first);
      epi_bar();
      if (!*last_flag) continue;
      if (et == 0) p.counters[tile * CL + (int)rank] = 0;
      bool chunked = false;
      if constexpr (NT == 128) {
        // ~512 loads a thread if this group summed alone (16 round trips):
        // post it in chunks, which converter warps done dequantizing take too,
        // once at least half of them are, or when at most one tile is left
        // to dequantize (they join as soon as it is done); otherwise sum
        // alone (an 8-token chunk costs as many round trips as the 16 token
        // rows of a pass below, and later tiles' accumulators wait)
        const int later = (mi.x < mi.end ? 1 : 0) + (mi.t_end - mi.t);   // fragments after this one
        if (et == 0) task->use = *reinterpret_cast<volatile int *>(&task->idle) >= 8 || later <= 1;
        epi_bar();
        chunked = task->use != 0;
      }
      if (chunked) {
        if (et == 0) {
          task->c_first = c_first;
          task->c_last = c_last;
          task->tile = tile;
          task->t0 = t0;
          task->mt = mt;
          task->f_first = f_first;
          atomicExch(&task->done, 0);
          ++gen;
          __threadfence_block();
          atomicExch(&task->word, (gen << 16) | ((uint32_t)((mt + 7) >> 3) * 4u << 8));
        }
        epi_bar();
        take_chunks();
        bool ok = true;
        if (et == 0) {
          const int nch = (int)((mt + 7) >> 3) * 4;
          uint64_t w0 = 0;
          for (uint32_t polls = 1; *reinterpret_cast<volatile int *>(&task->done) < nch; ++polls) {
            if (*abort_flag || (limit && polls >= limit)) { ok = false; break; }
            if (!limit && (polls & 63u) == 0) {
              const uint64_t now = ptx::globaltimer();
              if (w0 == 0) w0 = now;
              else if (now - w0 > kTimeoutNs) { ok = false; break; }
            }
            __nanosleep(64);
          }
          if (!ok) give_up();
          __threadfence_block();              // the chunks' stores before the next post
        }
        if (ptx::bar_any(2, 128, !ok || *abort_flag)) break;
      } else {
#pragma unroll 1
      for (int g0 = 0; g0 < mt; g0 += TG) {
        float acc[TG];
#pragma unroll
        for (int x = 0; x < TG; ++x) acc[x] = 0.0f;
        for (int64_t c0 = c_first; c0 <= c_last; c0 += MAXC) {   // K order; MAXC loads in flight
          float pv[MAXC][TG];
#pragma unroll
          for (int u = 0; u < MAXC; ++u) {
            const bool have = c0 + u <= c_last;
            const float *pc = slot(have ? c0 + u : c0) + (size_t)g0 * 128 + row;
#pragma unroll
            for (int x = 0; x < TG; ++x) pv[u][x] = (have && g0 + x < mt) ? __ldcg(pc + x * 128) : 0.0f;
          }
#pragma unroll
          for (int u = 0; u < MAXC; ++u)
            if (c0 + u <= c_last) {
#pragma unroll
              for (int x = 0; x < TG; ++x) acc[x] += pv[u][x];
            }
        }
        if (n < p.n) {
#pragma unroll
          for (int x = 0; x < TG; ++x)
            if (g0 + x < mt) p.d[(size_t)(t0 + g0 + x) * p.n + n] = out_bits(acc[x], t0 + g0 + x);
        }
      }
      }
    }
    if (NT == 128 && et == 0) {
      __threadfence_block();
      *reinterpret_cast<volatile int *>(&task->stop) = 1;   // the converter warps may leave
    }
  }

  __syncthreads();
  if (*abort_flag) {
    volatile int no_abort = 0;
    if (warp == kWarpProdW && issued_w) {
      for (int r = 0; r < WST; ++r)
        if (issued_w & (1u << r)) ptx::mbar_wait_bounded(&wfull[r], (issued_w_par >> r) & 1u, kDrainPolls, 0, &no_abort);
    }
    if (warp == kWarpProdX && issued_x) {
      for (int r = 0; r < XST; ++r)
        if (issued_x & (1u << r)) ptx::mbar_wait_bounded(&xfull[r], (issued_x_par >> r) & 1u, kDrainPolls, 0, &no_abort);
    }
    if ((warp == kWarpMma0 || warp == kWarpMma1) && mma_issued) {
      uint64_t *dr = &drain[warp == kWarpMma0 ? 0 : 1];
      if constexpr (PAIR) ptx::tc_commit_pair(ptx::smem_u32(dr));
      else ptx::tc_commit(dr);
      ptx::mbar_wait_bounded(dr, 0, kDrainPolls, 0, &no_abort);
    }
    if (PAIR && threadIdx.x == 0) {
      // some of a pair CTA's copies complete on the other CTA's barrier: a
      // short settle time covers those
      const uint64_t t0 = ptx::globaltimer();
      while (ptx::globaltimer() - t0 < kSettleNs) __nanosleep(1000);
    }
  }
  ptx::tc_fence_before();
  if constexpr (PAIR) ptx::cluster_sync();   // the partner's MMAs and copies no longer touch this CTA
  else __syncthreads();
  ptx::tc_fence_after();
  if (warp == kWarpMma0) {
    if constexpr (PAIR) ptx::tmem_dealloc_pair(tmem, C::TMEM_COLS);
    else ptx::tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// Token rows of x (times the AWQ pre-scale s when given, rounded to bf16 as
// the separate multiply does) -> f16 x16 = x * 2^e with e per row bringing
// the row's largest finite magnitude into [2^15, 2^16), and rs[row] = 2^-e.
// One CTA per row; a row of up to kPrepThreads * kPrepVecs * 8 elements
// (18432) is read once into registers (all loads in flight together), longer
// rows read their remainder twice.  256 threads a CTA, so that several rows
// are in flight on an SM (a 1024-thread CTA at this register count took the
// whole register file: one row at a time, ~1/4 of HBM at 1024 rows).
constexpr int kPrepThreads = 256, kPrepVecs = 9;

__global__ void __launch_bounds__(kPrepThreads) w4a16_act_f16_kernel(const uint16_t *__restrict__ x,
                                                                     const uint16_t *__restrict__ s, int64_t k,
                                                                     uint16_t *__restrict__ x16,
                                                                     float *__restrict__ rs) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[kPrepThreads / 32];
  const int64_t row = blockIdx.x;
  const uint4 *xr = reinterpret_cast<const uint4 *>(x + row * k);
  const uint4 *sr = reinterpret_cast<const uint4 *>(s);
  const int n8 = (int)(k >> 3);
  auto load = [&](int i) {
    uint4 v = xr[i];
    if (s) {
      const uint4 sv = __ldg(sr + i);
      v = make_uint4(bf16x2_mul(v.x, sv.x), bf16x2_mul(v.y, sv.y), bf16x2_mul(v.z, sv.z), bf16x2_mul(v.w, sv.w));
    }
    return v;
  };
  auto fmax_finite = [](float a, float v) { return fabsf(v) <= FLT_MAX ? fmaxf(a, fabsf(v)) : a; };
  auto vmax = [&](float a, const uint4 &v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int u = 0; u < 4; ++u) a = fmax_finite(fmax_finite(a, bf16_lo(w[u])), bf16_hi(w[u]));
    return a;
  };
  uint4 keep[kPrepVecs];
#pragma unroll
  for (int u = 0; u < kPrepVecs; ++u) {
    const int i = threadIdx.x + u * kPrepThreads;
    keep[u] = i < n8 ? load(i) : make_uint4(0, 0, 0, 0);
  }
  float amax = 0.0f;
#pragma unroll
  for (int u = 0; u < kPrepVecs; ++u) amax = vmax(amax, keep[u]);
  for (int i = threadIdx.x + kPrepVecs * kPrepThreads; i < n8; i += kPrepThreads) amax = vmax(amax, load(i));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = 0.0f;
#pragma unroll
  for (int i = 0; i < kPrepThreads / 32; ++i) amax = fmaxf(amax, red[i]);
  int e = 0;
  if (amax > 0.0f) {
    int ex;
    (void)frexpf(amax, &ex);             // amax in [2^(ex-1), 2^ex)
    e = min(max(16 - ex, -126), 126);
  }
  const float up = __uint_as_float((uint32_t)(127 + e) << 23);
  if (threadIdx.x == 0) rs[row] = __uint_as_float((uint32_t)(127 - e) << 23);
  uint4 *outr = reinterpret_cast<uint4 *>(x16 + row * k);
  auto convert = [&](const uint4 &v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const __half2 hv = __floats2half2_rn(bf16_lo(w[u]) * up, bf16_hi(w[u]) * up);
      o[u] = *reinterpret_cast<const uint32_t *>(&hv);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
  };
#pragma unroll
  for (int u = 0; u < kPrepVecs; ++u) {
    const int i = threadIdx.x + u * kPrepThreads;
    if (i < n8) outr[i] = convert(keep[u]);
  }
  for (int i = threadIdx.x + kPrepVecs * kPrepThreads; i < n8; i += kPrepThreads) outr[i] = convert(load(i));
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

int pick_nt(int64_t m) { return m <= 16 ? 16 : m <= 32 ? 32 : m <= 64 ? 64 : 128; }

// Work split and workspace layout of one call: [arrival counters |
// fp32 partials of shared tiles | f16 activations | row scales].
struct TPlan {
  int nt, cl, wtiles, ttiles, nkb, grid, maxfrag, whole, split_tiles;   // grid: CTA clusters (pairs or single CTAs)
  size_t x16_off, rs_off, ws_bytes;
};

TPlan make_tplan(int64_t m, int64_t n, int64_t k) {
  TPlan pl{};
  pl.nt = pick_nt(m);
  pl.cl = pl.nt == 128 ? 2 : 1;          // 128-token tiles: CTA pairs, 256 weight rows per tile
  const int bk = pl.nt <= 64 ? TCfg<16>::BK : TCfg<128, true>::BK;
  pl.wtiles = (int)((n + 128 * pl.cl - 1) / (128 * pl.cl));
  pl.ttiles = (int)((m + pl.nt - 1) / pl.nt);
  pl.nkb = (int)((k + bk - 1) / bk);     // the last k-block may be narrower (64-wide steps)
  const int tiles = pl.wtiles * pl.ttiles;
  const int units = num_sms() / pl.cl;   // clusters that fit, one CTA per SM
  const int64_t w = (int64_t)tiles * pl.nkb;
  pl.grid = (int)(w < units ? w : units);
  // every cluster gets `whole` whole tiles; the remaining tiles are cut into
  // one contiguous run of (tile, k-block) pairs per cluster, and every cluster
  // must own at least one k-block of them when there are any
  pl.whole = tiles / pl.grid;
  pl.split_tiles = tiles - pl.whole * pl.grid;
  if (pl.whole > 0 && pl.split_tiles > 0 && (int64_t)pl.split_tiles * pl.nkb < pl.grid) {
    --pl.whole;
    pl.split_tiles += pl.grid;
  }
  const int64_t su = (int64_t)pl.split_tiles * pl.nkb;
  const int64_t per = (su + pl.grid - 1) / pl.grid;
  pl.maxfrag = (int)((per + pl.nkb - 1) / pl.nkb + 1);
  const bool shared = su > 0 && ((su % pl.grid != 0) || ((su / pl.grid) % pl.nkb != 0));
  const size_t part_bytes = shared ? (size_t)pl.grid * pl.maxfrag * pl.cl * pl.nt * 128 * 4 : 0;
  pl.x16_off = kCounterArea + round256(part_bytes);
  pl.rs_off = pl.x16_off + round256((size_t)(m * k * 2));
  pl.ws_bytes = pl.rs_off + round256((size_t)m * 4);
  return pl;
}

template <int NT, bool PAIR>
cudaError_t launch_nt(const TPlan &pl, const uint16_t *x, const uint16_t *pre, const uint8_t *w, const uint8_t *wsf,
                      const float *alpha, uint16_t *d, int64_t m, int64_t n, int64_t k, uint8_t *ws,
                      uint32_t wait_limit, cudaStream_t st) {
  using C = TCfg<NT, PAIR>;
  static PerDeviceOnce smem_attr;   // the shared-memory limit is a setting of each device's context
  if (cudaError_t e = smem_attr.run([] {
        return cudaFuncSetAttribute(w4a16_tmem_kernel<NT, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)C::SMEM_BYTES);
      }))
    return e;
  uint16_t *x16 = reinterpret_cast<uint16_t *>(ws + pl.x16_off);
  float *rs = reinterpret_cast<float *>(ws + pl.rs_off);
  CUtensorMap tm_x, tm_w;
  // f16 activations [m, k]: box 128 bytes (64 elements) x XROWS rows, 128-byte swizzle;
  // weight codes [n, k/2]: box BK/2 bytes x 128 rows, swizzled as wide as the box
  if (!make_byte_map(&tm_x, x16, m, k * 2, 128, C::XROWS, 128) ||
      !make_byte_map(&tm_w, w, n, k / 2, C::CODE_ROW, 128, (int)C::CODE_ROW))
    return cudaErrorInvalidValue;
  TArgs a{};
  a.wsf = wsf;
  a.alpha = alpha;
  a.rs = rs;
  a.d = d;
  a.m = (int32_t)m;
  a.n = (int32_t)n;
  a.k = (int32_t)k;
  a.wtiles = pl.wtiles;
  a.ttiles = pl.ttiles;
  a.nkb = pl.nkb;
  a.grid = pl.grid;
  a.maxfrag = pl.maxfrag;
  a.whole = pl.whole;
  a.split_tiles = pl.split_tiles;
  a.counters = reinterpret_cast<int *>(ws);
  a.partials = reinterpret_cast<float *>(ws + kCounterArea);
  a.wait_limit = wait_limit;
  a.status = device_status_ptr();
  if (!a.status) return cudaErrorInvalidValue;
  if (cudaError_t e =
          launch_pdl(w4a16_act_f16_kernel, dim3((unsigned)m), dim3(kPrepThreads), 0, st, x, pre, k, x16, rs))
    return e;
  if constexpr (!PAIR)
    return launch_pdl(w4a16_tmem_kernel<NT, PAIR>, dim3(a.grid), dim3(kThreads), C::SMEM_BYTES, st, tm_x, tm_w, a);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = C::CL;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(a.grid * C::CL);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, w4a16_tmem_kernel<NT, PAIR>, tm_x, tm_w, a);
}

}  // namespace

bool w4a16_tmem_supported(int64_t m, int64_t n, int64_t k) {
  return m > 0 && w4a16_tc_supported(m, n, k) && (size_t)m * (size_t)k < ((size_t)1 << 31);
}

size_t w4a16_tmem_workspace_bytes(int64_t m, int64_t n, int64_t k) {
  if (!w4a16_tmem_supported(m, n, k)) return 0;
  return make_tplan(m, n, k).ws_bytes;
}

cudaError_t launch_w4a16_tmem(const uint16_t *x, const uint16_t *pre_scale, const uint8_t *w, const uint8_t *wsf,
                              const float *alpha, uint16_t *d, int64_t m, int64_t n, int64_t k, void *ws,
                              size_t ws_bytes, uint32_t wait_limit, cudaStream_t st) {
  if (!w4a16_tmem_supported(m, n, k)) return cudaErrorNotSupported;
  const TPlan pl = make_tplan(m, n, k);
  if (!ws || ws_bytes < pl.ws_bytes) return cudaErrorInvalidValue;
  uint8_t *wsb = static_cast<uint8_t *>(ws);
  switch (pl.nt) {
    case 16: return launch_nt<16, false>(pl, x, pre_scale, w, wsf, alpha, d, m, n, k, wsb, wait_limit, st);
    case 32: return launch_nt<32, false>(pl, x, pre_scale, w, wsf, alpha, d, m, n, k, wsb, wait_limit, st);
    case 64: return launch_nt<64, false>(pl, x, pre_scale, w, wsf, alpha, d, m, n, k, wsb, wait_limit, st);
    default: return launch_nt<128, true>(pl, x, pre_scale, w, wsf, alpha, d, m, n, k, wsb, wait_limit, st);
  }
}

}  // namespace nvfp4
