// tcgen05 tensor-core GEMMs: NVFP4 block-scaled MMA (E2M1 x E2M1, UE4M3 per
// 16 elements), accumulators in TMEM.
//
// Kernel shape (clusters of two CTAs, one CTA per SM, persistent over output
// tiles; the roles are listed at the kernel):
//   warp 0      TMA producer: A/B code tiles (2-D tensor maps, 128-byte
//               swizzle) and the matching 512-byte tiles of the swizzled
//               block scales (1-D bulk copies), one mbarrier per stage; the
//               weight half-tiles are multicast to both CTAs of the cluster;
//   warp 1      allocates TMEM; one elected thread issues the MMAs and
//               commits each stage back to both producers;
//   warps 10-13 write each stage's block scales into TMEM (tcgen05.st);
//   warps 2..9  epilogue: TMEM -> registers (tcgen05.ld), TMEM released at
//               once, then bf16 output or the fused SwiGLU + NVFP4 requantize
//               of the gate_up GEMM while the next tile's MMAs run.
// Tile 128 (M) x 256 (N) x 256 (K) per CTA; one MMA instruction covers K =
// 64, so a stage holds four.  Every mbarrier wait is bounded: a wait that
// gives up records NVFP4_ERR_DEVICE_TIMEOUT, every role leaves its loop,
// outstanding copies and MMAs are drained with a second bounded wait, TMEM is
// freed and the kernel returns.
#include <cudaTypedefs.h>

#include <mutex>

#include "common.cuh"
#include "internal.h"
#include "tc_ptx.cuh"

namespace nvfp4 {

// Status word of this device: a kernel that gives up a bounded wait records
// NVFP4_ERR_DEVICE_TIMEOUT here (first writer wins).
__device__ int g_device_status = 0;

cudaError_t read_and_clear_device_status(int *out) {
  const int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(out, g_device_status, sizeof(int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
}

int *device_status_ptr() {
  static int *cache[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  if (!cache[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_status) == cudaSuccess) cache[dev] = static_cast<int *>(p);
  }
  return cache[dev];
}

namespace {

constexpr int BM = 128, BN = 256, BK = 256;
constexpr int KSTEPS = BK / 64;                 // MMAs per stage
constexpr int STAGES = 4;
constexpr uint32_t A_BYTES = BM * BK / 2;       // 16 KB
constexpr uint32_t B_BYTES = BN * BK / 2;       // 32 KB (two 16 KB halves, one per CTA of the pair)
constexpr uint32_t B_HALF = B_BYTES / 2;
constexpr uint32_t SFA_BYTES = (BM / 128) * KSTEPS * 512;
constexpr uint32_t SFB_BYTES = (BN / 128) * KSTEPS * 512;
constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES + SFA_BYTES + SFB_BYTES;
constexpr uint32_t SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
constexpr int kThreads = 448;           // producer, MMA, 8 epilogue warps, 4 scale-writer warps
constexpr int kCluster = 2;             // CTAs sharing one weight tile
constexpr uint16_t kPairMask = 0x3;
constexpr uint32_t TMEM_COLS = 512;
// accumulator 256 columns; one scale slot of 48 columns (SFA 16 + SFB 32,
// 64-column pitch) per smem stage.  With a slot per stage the stage's data
// barrier orders everything: the producer refills stage s only after the
// MMAs of its previous use have completed (both CTAs' commits), so a writer
// that has seen the new data of stage s may overwrite slot s — no barrier of
// its own for freeing the slot, and one commit per stage for the MMA issuer.
constexpr int SF_SLOTS = STAGES;
constexpr uint32_t ACC_COL = 0, SF_COL = 256, SF_SLOT = 64, SFB_OFF = 4 * KSTEPS;
static_assert(SF_COL + SF_SLOTS * SF_SLOT <= 512, "TMEM columns");
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s
constexpr uint32_t kDrainPolls = 1u << 22;

// Instruction descriptor, kind::mxf4nvf4: A/B format E2M1 (1) in bits 7-9 and
// 10-12, K-major both, N >> 3 in bits 17-22, scale type UE4M3 (0) in bit 23,
// M >> 4 in bits 24-28, scale-factor ids 0, dense K = 64.
constexpr uint32_t idesc_nvfp4(int m, int n) {
  return (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

struct TcArgs {
  const uint8_t *sfa;     // swizzled scales of A (M rows)
  const uint8_t *sfb;     // swizzled scales of B (N rows)
  const float *alpha;
  const float *out_gs;
  uint16_t *d;            // bf16 [M, N]
  uint8_t *out_fp4;       // fused: [M, N/4]
  uint8_t *out_sf;        // fused: swizzled over M rows, N/32 columns
  int32_t m, n, k;
  int32_t num_m, num_n, num_mpairs;
  uint32_t wait_limit;
  int *status;            // device status word
  const float *rs;        // optional per-row activation dequant factor [M]
  int32_t group_mp;       // tile order: m-pairs per group (see tile_of)
};

struct Smem {
  uint8_t *base;
  __device__ uint8_t *a(int s) const { return base + s * STAGE_BYTES; }
  __device__ uint8_t *b(int s) const { return a(s) + A_BYTES; }
  __device__ uint8_t *sfa(int s) const { return b(s) + B_BYTES; }
  __device__ uint8_t *sfb(int s) const { return sfa(s) + SFA_BYTES; }
  __device__ uint64_t *full() const { return reinterpret_cast<uint64_t *>(base + STAGES * STAGE_BYTES); }
  __device__ uint64_t *empty() const { return full() + STAGES; }
  __device__ uint64_t *tfull() const { return empty() + STAGES; }
  __device__ uint64_t *tempty() const { return tfull() + 1; }
  __device__ uint64_t *drain() const { return tempty() + 1; }
  __device__ uint64_t *sf_full() const { return drain() + 1; }
  __device__ uint32_t *tslot() const { return reinterpret_cast<uint32_t *>(sf_full() + SF_SLOTS); }
  __device__ volatile int *abort_flag() const { return reinterpret_cast<volatile int *>(tslot() + 1); }
};

__device__ __forceinline__ void give_up(volatile int *abort_flag, int *status) {
  *abort_flag = 1;
  atomicCAS(status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

// Kernel shape (clusters of two CTAs, one CTA per SM, persistent): the two
// CTAs of a cluster compute the 128-row tiles 2p and 2p+1 of M against the
// same 256-row weight tile, k-block by k-block in lockstep.  Each CTA loads
// its own activation tile and scales, and one 128-row half of the weight tile
// plus that half's scales, delivered by TMA multicast to both CTAs -- so the
// weight stream is read from L2 once per pair.  A stage is refilled only when
// the MMAs of both CTAs are done with it (their commits arrive on both CTAs'
// empty barriers).  Roles per CTA:
//   warp 0      TMA producer;
//   warp 1      TMEM owner, single-thread MMA issuer;
//   warps 10-13 write each stage's block scales into one of two TMEM scale
//               slots (tcgen05.st, one warp per lane quarter) ahead of the MMAs;
//   warps 2..9  epilogue: TMEM -> registers, TMEM released at once, then bf16
//               output or the fused SwiGLU + NVFP4 requantize.
template <int MODE>  // TC_W4A4: bf16 out; TC_W4A4_SWIGLU: fused SwiGLU + NVFP4 requant
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const TcArgs p) {
  extern __shared__ uint8_t smem_raw[];
  Smem sm{reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023))};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *abort_flag = sm.abort_flag();
  const int rank = (int)ptx::cluster_ctarank();
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(&sm.full()[s], 1);
      ptx::mbar_init(&sm.empty()[s], kCluster);   // one commit from each CTA's MMA
    }
    ptx::mbar_init(sm.tfull(), 1);
    ptx::mbar_init(sm.tempty(), 256);
    ptx::mbar_init(sm.drain(), 1);
    for (int b = 0; b < SF_SLOTS; ++b) ptx::mbar_init(&sm.sf_full()[b], 4);   // one arrival per scale-writer warp
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tm_a);
    ptx::prefetch_tensormap(&tm_b);
  }
  if (warp == 1) {
    ptx::tmem_alloc(sm.tslot(), TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();          // both CTAs' barriers exist before any multicast lands
  ptx::tc_fence_after();
  const uint32_t tmem = *sm.tslot();

  const int cluster = blockIdx.x / kCluster, num_clusters = gridDim.x / kCluster;
  const int num_pairs = p.num_mpairs * p.num_n;
  const int ksteps_total = p.k >> 6;              // K / 64
  const int num_kb = (ksteps_total + KSTEPS - 1) / KSTEPS;
  const int cp4 = ksteps_total;                   // 512-byte scale tiles per 128-row block
  const int nrb_b = (p.n + 127) >> 7;             // 128-row blocks of B
  const uint32_t limit = p.wait_limit;
  // Work order: groups of group_mp m-pairs; within a group the m-pair runs
  // fastest, then the weight tile.  The clusters running at one time then
  // share a bounded set of activation rows (kept in L2 across the group's
  // sweep over the weights), and every weight tile is read once per group.
  auto tile_of = [&](int pair, int &mt, int &nt) {
    const int per_group = p.group_mp * p.num_n;
    const int g = pair / per_group;
    const int r = pair - g * per_group;
    const int gsz = min(p.group_mp, p.num_mpairs - g * p.group_mp);
    nt = r / gsz;
    mt = (g * p.group_mp + (r - nt * gsz)) * kCluster + rank;
  };

  uint32_t issued_mask = 0, issued_parity = 0;
  bool mma_issued = false;

  if (warp == 0) {
    if (ptx::elect_one()) {
      const uint64_t pol_a = ptx::l2_policy_evict_last();
      const uint64_t pol_b = ptx::l2_policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      // The first STAGES stages get their weight halves before the previous
      // kernel on the stream has finished; the activation tiles follow once
      // it has.
      int pend_s[STAGES], pend_kb[STAGES], pend_mt[STAGES];
      int npend = 0, c = 0;
      bool flushed = false;
      auto issue_a = [&](int st, int mt, int kb) {
        const int nk = min(KSTEPS, ksteps_total - kb * KSTEPS);
        ptx::tma_load_2d(sm.a(st), &tm_a, &sm.full()[st], kb * (BK / 2), mt * BM, pol_a);
        if (mt < p.num_m)
          ptx::bulk_load(sm.sfa(st), p.sfa + ((size_t)mt * cp4 + kb * KSTEPS) * 512, nk * 512u,
                         &sm.full()[st], pol_a);
      };
      auto flush = [&]() {
        pdl_wait();
        for (int i = 0; i < npend; ++i) issue_a(pend_s[i], pend_mt[i], pend_kb[i]);
        flushed = true;
      };
      for (int pair = cluster; pair < num_pairs && !*abort_flag; pair += num_clusters) {
        int mt, nt;
        tile_of(pair, mt, nt);
        const int nbv = min(2, nrb_b - nt * 2);
        for (int kb = 0; kb < num_kb; ++kb, ++c) {
          if (c == STAGES && !flushed) flush();
          if (!ptx::mbar_wait_bounded(&sm.empty()[s], ph ^ 1u, limit, kDefaultTimeoutNs, abort_flag)) {
            give_up(abort_flag, p.status);
            break;
          }
          const int nk = min(KSTEPS, ksteps_total - kb * KSTEPS);
          const uint32_t sfa_bytes = mt < p.num_m ? (uint32_t)nk * 512u : 0u;
          ptx::mbar_arrive_expect_tx(&sm.full()[s], A_BYTES + B_BYTES + sfa_bytes + (uint32_t)nk * 512u * nbv);
          // my half of the weight tile and of its scales, to both CTAs
          ptx::tma_load_2d_mc(sm.b(s) + rank * B_HALF, &tm_b, &sm.full()[s], kb * (BK / 2), nt * BN + rank * 128,
                              kPairMask, pol_b);
          if (rank < nbv)
            ptx::bulk_load_mc(sm.sfb(s) + rank * (KSTEPS * 512),
                              p.sfb + ((size_t)(nt * 2 + rank) * cp4 + kb * KSTEPS) * 512, nk * 512u,
                              &sm.full()[s], kPairMask, pol_b);
          if (c < STAGES) {
            pend_s[npend] = s;
            pend_kb[npend] = kb;
            pend_mt[npend] = mt;
            ++npend;
          } else {
            issue_a(s, mt, kb);
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
      constexpr uint32_t idesc = idesc_nvfp4(BM, BN);
      int s = 0, g = 0;                            // stage, global k-block count
      uint32_t ph = 0;
      int it = 0;
      for (int pair = cluster; pair < num_pairs && !*abort_flag; pair += num_clusters, ++it) {
        if (!ptx::mbar_wait_bounded(sm.tempty(), (uint32_t)(it & 1) ^ 1u, limit, kDefaultTimeoutNs,
                                    abort_flag)) {
          give_up(abort_flag, p.status);
          break;
        }
        ptx::tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          // The scale writers saw the stage's TMA data complete before they
          // filled its scale slot: one barrier covers both.
          if (!ptx::mbar_wait_bounded(&sm.sf_full()[s], ph, limit, kDefaultTimeoutNs, abort_flag)) {
            give_up(abort_flag, p.status);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const int nk = min(KSTEPS, ksteps_total - kb * KSTEPS);
          const uint32_t sf = tmem + SF_COL + s * SF_SLOT;
          const uint32_t a_s = ptx::smem_u32(sm.a(s)), b_s = ptx::smem_u32(sm.b(s));
          for (int j = 0; j < nk; ++j)
            ptx::mma_nvfp4(tmem + ACC_COL, ptx::smem_desc(a_s + 32 * j, 16, 1024, 2),
                           ptx::smem_desc(b_s + 32 * j, 16, 1024, 2), idesc, sf + 4 * j, sf + SFB_OFF + 8 * j,
                           (kb | j) != 0);
          mma_issued = true;
          ptx::tc_commit_mc(&sm.empty()[s], kPairMask);   // this stage and its scale slot are free
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        ptx::tc_commit(sm.tfull());
      }
    }
  } else if (warp >= 10) {
    // ------------------------------------------------------ scale writers
    // Warp w fills TMEM lane quarter w % 4 (a warp reaches only its own
    // quarter) of the stage's scale slot from registers with tcgen05.st: the
    // same 4 columns x 32 lanes per 512-byte scale tile that a warpx4 copy
    // of the tile would write, replicated in every quarter.  These stores
    // do not queue behind the MMAs in the tensor pipe as tcgen05.cp does.
    pdl_wait();
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    int s = 0, g = 0;
    uint32_t ph = 0;
    for (int pair = cluster; pair < num_pairs && !*abort_flag; pair += num_clusters) {
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb, ++g) {
        // the stage's data: its arrival also means the MMAs that read this
        // scale slot last have completed (the producer refilled the stage
        // only after they committed it)
        if (!ptx::mbar_wait_bounded(&sm.full()[s], ph, limit, kDefaultTimeoutNs, abort_flag)) {
          give_up(abort_flag, p.status);
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // lane l takes bytes 16l .. 16l+15 of every scale tile of the stage
        // (rows l, l+32, l+64, l+96; 4 scales each).  Tiles past the K tail
        // or the last weight block hold stale bytes the MMAs never use.
        const uint8_t *sfa = sm.sfa(s) + lane * 16, *sfb = sm.sfb(s) + lane * 16;
        uint32_t ra[16], rb0[16], rb1[16];
#pragma unroll
        for (int j = 0; j < KSTEPS; ++j) {
          const uint4 v = *reinterpret_cast<const uint4 *>(sfa + 512 * j);
          ra[4 * j] = v.x; ra[4 * j + 1] = v.y; ra[4 * j + 2] = v.z; ra[4 * j + 3] = v.w;
        }
#pragma unroll
        for (int j = 0; j < KSTEPS; ++j)
#pragma unroll
          for (int rb = 0; rb < 2; ++rb) {
            const uint4 v = *reinterpret_cast<const uint4 *>(sfb + rb * (KSTEPS * 512) + 512 * j);
            uint32_t *d = (j < 2 ? rb0 : rb1) + 8 * (j & 1) + 4 * rb;   // column 8j + 4rb of the SFB slot
            d[0] = v.x; d[1] = v.y; d[2] = v.z; d[3] = v.w;
          }
        const uint32_t sf = tmem + lane_off + SF_COL + s * SF_SLOT;
        ptx::tmem_st16(sf, ra);
        ptx::tmem_st16(sf + SFB_OFF, rb0);
        ptx::tmem_st16(sf + SFB_OFF + 16, rb1);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(&sm.sf_full()[s]);
        if (++s == STAGES) { s = 0; ph ^= 1u; }
      }
      if (!ok) break;
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // Warp w reads TMEM lane quarter w % 4 (the hardware lets a warp reach
    // only its own quarter) and column half (w - 2) / 4: 128 accumulator
    // columns of its 32 rows, held in registers; TMEM is released before any
    // math or store, so the next tile's MMAs run meanwhile.
    pdl_wait();
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int row = q * 32 + lane;
    const uint32_t t_base = tmem + ((uint32_t)(q * 32) << 16) + ACC_COL + 128 * half;
    const float alpha = __ldg(p.alpha);
    int it = 0;
    for (int pair = cluster; pair < num_pairs; pair += num_clusters, ++it) {
      if (!ptx::mbar_wait_bounded(sm.tfull(), (uint32_t)(it & 1), limit, kDefaultTimeoutNs, abort_flag)) {
        give_up(abort_flag, p.status);
        break;
      }
      ptx::tc_fence_after();
      uint32_t acc[128];
#pragma unroll
      for (int c = 0; c < 8; ++c) ptx::tmem_ld16(t_base + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&acc[16 * c]));
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      ptx::mbar_arrive(sm.tempty());            // accumulator free for the next tile

      int mt, nt;
      tile_of(pair, mt, nt);
      if (mt >= p.num_m) continue;              // odd tail: this CTA only fed its partner
      const int m = mt * BM + row;
      const float am = (p.rs && m < p.m) ? alpha * p.rs[m] : alpha;
      if constexpr (MODE == TC_W4A4) {
        const int n0 = nt * BN + 128 * half;
        if (m < p.m) {
          uint16_t *drow = p.d + (size_t)m * p.n;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const int n = n0 + 8 * c;
            if (n < p.n) {
              uint4 o;
              o.x = pack_bf16x2(am * __uint_as_float(acc[8 * c + 0]), am * __uint_as_float(acc[8 * c + 1]));
              o.y = pack_bf16x2(am * __uint_as_float(acc[8 * c + 2]), am * __uint_as_float(acc[8 * c + 3]));
              o.z = pack_bf16x2(am * __uint_as_float(acc[8 * c + 4]), am * __uint_as_float(acc[8 * c + 5]));
              o.w = pack_bf16x2(am * __uint_as_float(acc[8 * c + 6]), am * __uint_as_float(acc[8 * c + 7]));
              *reinterpret_cast<uint4 *>(drow + n) = o;
            }
          }
        }
      } else {
        // this half's columns: [up 64 | gate 64] for features nt*128 + 64*half + (0..63)
        const int inter = p.n >> 1;
        const int f0 = nt * 128 + 64 * half;
        if (f0 < inter) {
          const float gs = __ldg(p.out_gs);
          const int ocp4 = ((inter >> 4) + 3) >> 2;
          uint32_t sfw = 0;
          if (m < p.m) {
            uint32_t codes[8];
#pragma unroll
            for (int qb = 0; qb < 4; ++qb) {
              float hv[16];
#pragma unroll
              for (int i = 0; i < 16; ++i)
                hv[i] = silu_mul_fast(am * __uint_as_float(acc[64 + 16 * qb + i]),
                                      am * __uint_as_float(acc[16 * qb + i]));
              sfw |= quantize_block16(hv, gs, codes[2 * qb], codes[2 * qb + 1]) << (8 * qb);
            }
            uint4 *dst = reinterpret_cast<uint4 *>(p.out_fp4 + (size_t)m * (inter >> 1) + f0 / 2);
            dst[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
            dst[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
          }
          // scale columns f0/16 .. +3 of this row in one word; padding rows past M get 0
          *reinterpret_cast<uint32_t *>(p.out_sf + sf_swizzled_offset(m, f0 >> 4, ocp4)) = sfw;
        }
      }
    }
  }

  __syncthreads();
  if (*abort_flag) {
    // Drain: wait (bounded) for this CTA's copies still in flight and for
    // every MMA it issued, so nothing lands in shared memory or TMEM after
    // the CTA is gone.
    if (warp == 0 && issued_mask) {
      for (int s = 0; s < STAGES; ++s)
        if (issued_mask & (1u << s)) {
          volatile int no_abort = 0;
          ptx::mbar_wait_bounded(&sm.full()[s], (issued_parity >> s) & 1u, kDrainPolls, 0, &no_abort);
        }
    }
    if (warp == 1 && mma_issued) {
      volatile int no_abort = 0;
      ptx::tc_commit(sm.drain());
      ptx::mbar_wait_bounded(sm.drain(), 0, kDrainPolls, 0, &no_abort);
    }
  }
  ptx::tc_fence_before();
  ptx::cluster_sync();          // the partner no longer multicasts into this CTA
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, TMEM_COLS);
}

// ------------------------------------------------------------------ host side
PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void *f = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

}  // namespace

bool make_byte_map(CUtensorMap *tm, const void *ptr, int64_t rows, int64_t row_bytes, uint32_t box_bytes,
                   uint32_t box_rows, bool swizzle128) {
  auto encode = get_encode();
  if (!encode) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {box_bytes, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE,
                swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return 148;
  if (!cache[dev]) {
    int v = 0;
    cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    cache[dev] = v > 0 ? v : 148;
  }
  return cache[dev];
}

namespace {

template <int MODE>
cudaError_t launch_mode(const uint8_t *a, const uint8_t *a_sf, const uint8_t *b, const uint8_t *b_sf,
                        const float *alpha, const float *out_gs, uint16_t *d, uint8_t *out_fp4,
                          uint8_t *out_sf, int64_t m, int64_t n, int64_t k, uint32_t wait_limit,
                        cudaStream_t st, const float *rs) {
  static int max_clusters[64] = {0};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (!max_clusters[dev]) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)SMEM_BYTES);
    if (e != cudaSuccess) return e;
    // how many 2-CTA clusters of this kernel the device holds at once
    cfg.gridDim = dim3(kCluster * (num_sms() / kCluster));
    int nc = 0;
    e = cudaOccupancyMaxActiveClusters(&nc, tc_gemm_kernel<MODE>, &cfg);
    if (e != cudaSuccess || nc <= 0) nc = num_sms() / kCluster;
    max_clusters[dev] = nc;
  }
  CUtensorMap tm_a, tm_b;
  // codes [rows, k/2] bytes; box 128 bytes of K x (128 activation rows | 128
  // weight rows = half a weight tile), 128-byte swizzle
  if (!make_byte_map(&tm_a, a, m, k / 2, 128, BM, true) || !make_byte_map(&tm_b, b, n, k / 2, 128, BN / 2, true))
    return cudaErrorInvalidValue;
  TcArgs args{a_sf, b_sf, alpha, out_gs, d, out_fp4, out_sf, (int32_t)m, (int32_t)n, (int32_t)k,
              (int32_t)((m + BM - 1) / BM), (int32_t)((n + BN - 1) / BN), 0, wait_limit, device_status_ptr(), rs};
  if (!args.status) return cudaErrorInvalidValue;
  args.num_mpairs = (args.num_m + kCluster - 1) / kCluster;
  {
    // Activation rows of one group: at most ~32 MiB, so that, together with
    // the weight tiles in flight (and any copies the two dies' L2 halves
    // keep), they stay in the 129 MB L2 while the group sweeps the weights.
    const int64_t pair_bytes = (int64_t)kCluster * BM * (k / 2);
    const int64_t g = (int64_t(32) << 20) / pair_bytes;
    args.group_mp = (int32_t)(g < 1 ? 1 : g > args.num_mpairs ? args.num_mpairs : g);
  }
  const int pairs = args.num_mpairs * args.num_n;
  const int clusters = pairs < max_clusters[dev] ? pairs : max_clusters[dev];
  cfg.gridDim = dim3(kCluster * clusters);
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<MODE>, tm_a, tm_b, args);
}

}  // namespace

bool tc_supported(TcMode mode, bool swap_ab, int64_t m, int64_t n, int64_t k) {
  if (swap_ab || mode == TC_W4A16) return false;
  if (k % 64 != 0 || n % 32 != 0 || m <= 0) return false;
  if (mode == TC_W4A4_SWIGLU && n % 128 != 0) return false;
  if (m > (1 << 30) || n > (1 << 30) || k > (1 << 30)) return false;
  return get_encode() != nullptr;
}

cudaError_t launch_tc(TcMode mode, bool swap_ab, const void *a, const uint8_t *a_sf, const uint8_t *b,
                      const uint8_t *b_sf, const float *alpha, const float *out_gs, uint16_t *d,
                      uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n, int64_t k,
                      uint32_t wait_limit, cudaStream_t st, const float *a_row_scale) {
  if (!tc_supported(mode, swap_ab, m, n, k)) return cudaErrorNotSupported;
  const uint8_t *a8 = static_cast<const uint8_t *>(a);
  if (mode == TC_W4A4)
    return launch_mode<TC_W4A4>(a8, a_sf, b, b_sf, alpha, out_gs, d, out_fp4, out_sf, m, n, k, wait_limit, st,
                                a_row_scale);
  return launch_mode<TC_W4A4_SWIGLU>(a8, a_sf, b, b_sf, alpha, out_gs, d, out_fp4, out_sf, m, n, k,
                                     wait_limit, st, a_row_scale);
}

}  // namespace nvfp4
