// tcgen05 tensor-core GEMMs for prefill-sized M: NVFP4 block-scaled MMA
// (E2M1 x E2M1, UE4M3 per 16 elements), accumulators in TMEM.
//
// Output tile 128 (M) x 256 (N) per CTA, k-blocks of 256 (four K = 64 MMAs
// per pipeline stage), persistent over output tiles.  Two instances:
//   PAIR (the default): clusters of two CTAs on two SMs issue 2-SM MMAs
//     (cta_group::2, 256 x 256 x 64).  Each CTA loads its own 128 rows of A
//     and one 128-row half of the 256-row weight tile; the MMA reads both
//     CTAs' halves, so each SM stages 32 KB of operands per 256-wide k-block
//     instead of 48 KB, and five stages fit where one CTA per tile fits four.
//     The pair's even CTA (the leader) issues the MMAs and owns the
//     pipeline's full barriers; both CTAs' loads and both CTAs' scale
//     writers complete on the leader's barrier, and the leader's commits
//     free both CTAs' stages.
//   1-SM: one CTA per 128 x 256 tile loads the whole weight tile itself.
// Roles per CTA (480 threads):
//   warp 0      TMA producer of the operand tiles (2-D tensor maps, 128-byte
//               swizzle);
//   warp 14     scale producer: the matching 512-byte tiles of the swizzled
//               block scales (1-D bulk copies) into a scale ring that runs
//               ahead of the operand ring;
//   warp 1      TMEM owner (the pair allocates collectively); one elected
//               thread issues the MMAs (the leader's only, in a pair);
//   warps 10-13 write each stage's block scales into this CTA's TMEM
//               (tcgen05.st) as soon as the stage's previous MMAs commit;
//   warps 2..9  epilogue: TMEM -> registers (tcgen05.ld), TMEM released at
//               once, then bf16 output or the fused SwiGLU + NVFP4 requantize
//               of the gate_up GEMM while the next tile's MMAs run.
// Every mbarrier wait is bounded: a wait that gives up records
// NVFP4_ERR_DEVICE_TIMEOUT and tells the partner CTA, every role leaves its
// loop, outstanding copies and MMAs are drained with a second bounded wait,
// TMEM is freed and the kernel returns.
#include <cudaTypedefs.h>

#include <atomic>
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
constexpr uint32_t A_BYTES = BM * BK / 2;       // 16 KB: this CTA's 128 activation rows
constexpr uint32_t B_HALF = 128 * BK / 2;       // 16 KB: 128 weight rows
constexpr uint32_t SFA_BYTES = KSTEPS * 512;    // scale tiles of the activation rows
constexpr uint32_t SFB_BYTES = 2 * KSTEPS * 512;   // scale tiles of all 256 weight rows
constexpr int kThreads = 480;           // producer, MMA, 8 epilogue, 4 scale-writer warps, scale producer
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t ACC_COL = 0, SF_COL = 256, SFB_OFF = 4 * KSTEPS;
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;   // 2 s
constexpr uint64_t kDrainNs = 2000000ull;               // 2 ms per drain wait after a give-up
constexpr uint64_t kSettleNs = 50000ull;                // then 50 us for copies counted elsewhere

// Pipeline shape per instance: three rings indexed by the CTA's running
// k-block count g.
//   operand stages  (STAGES)   A and B tiles of k-block g in slot g % STAGES;
//   scale slots     (SF_SLOTS) the SFA + SFB tiles (6 KB) in shared memory,
//                              loaded up to SF_SLOTS k-blocks ahead;
//   TMEM scale slots (T_SLOTS) SFA 16 + SFB 32 columns after the 256
//                              accumulator columns.
// The scale writers fill TMEM slot g % T_SLOTS once the MMAs of k-block
// g - T_SLOTS have committed, from scales already waiting in shared memory,
// while k-block g's operands are still in flight -- so the scale path is off
// the refill loop (commit -> operand TMA -> MMA) that bounds the pipeline.
// The writers learn of that commit from the empty barrier of the operand
// stage that held k-block g - T_SLOTS, waited on by phase parity; the
// barrier's next phase belongs to k-block g - T_SLOTS + STAGES, whose MMAs
// cannot run before writer g is done, so the awaited phase is never
// overtaken.  With T_SLOTS == STAGES the TMEM slot of k-block g is its
// operand stage, and the writers arrive on that stage's full barrier next
// to the operand bytes: the MMA issuer waits on one barrier per k-block
// (each wait costs the single issuing thread a hundred-odd cycles even when
// the phase has already completed).  Both the producer's and the writers'
// arrivals for k-block g follow the commit of k-block g - STAGES, so no
// arrival lands in a neighbouring phase.
template <bool PAIR>
struct Cfg {
  static constexpr uint32_t B_BYTES = PAIR ? B_HALF : 2 * B_HALF;
  static constexpr uint32_t OPND_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t SF_BYTES = SFA_BYTES + SFB_BYTES;
  static constexpr int STAGES = PAIR ? 5 : 4;
  static constexpr int SF_SLOTS = PAIR ? 8 : 5;      // shared-memory scale slots
  static constexpr int T_SLOTS = STAGES;             // TMEM scale slots
  static constexpr uint32_t SF_SLOT = 48;
  static constexpr uint32_t SMEM_BYTES = STAGES * OPND_BYTES + SF_SLOTS * SF_BYTES + 1024 /*align*/ + 512 /*barriers*/;
  static constexpr int CLUSTER = PAIR ? 2 : 1;
  static_assert(SF_COL + T_SLOTS * SF_SLOT <= TMEM_COLS, "TMEM columns");
  static_assert(T_SLOTS == STAGES, "a k-block's scale slot is its operand stage (one full barrier for both)");
  static_assert(OPND_BYTES % 1024 == 0, "operand slots keep the 1024-byte swizzle alignment");
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

// Instruction descriptor, kind::mxf4nvf4: A/B format E2M1 (1) in bits 7-9 and
// 10-12, K-major both, N >> 3 in bits 17-22, scale type UE4M3 (0) in bit 23,
// M >> 4 in bits 24-28, scale-factor ids 0, dense K = 64.  For a pair MMA, M
// is the pair's 256 rows.
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
  int32_t num_m, num_n, num_mg;   // 128-row tiles of M and 256-row tiles of N; M tile groups (pairs or singles)
  uint32_t wait_limit;
  int *status;            // device status word
  const float *rs;        // optional per-row activation dequant factor [M]
  int32_t group_mp;       // tile order: M tile groups per L2 group (see tile_of)
};

template <bool PAIR>
struct Smem {
  using C = Cfg<PAIR>;
  uint8_t *base;
  __device__ uint8_t *a(int s) const { return base + s * C::OPND_BYTES; }
  __device__ uint8_t *b(int s) const { return a(s) + A_BYTES; }
  __device__ uint8_t *sfa(int s) const { return base + C::STAGES * C::OPND_BYTES + s * C::SF_BYTES; }
  __device__ uint8_t *sfb(int s) const { return sfa(s) + SFA_BYTES; }
  __device__ uint64_t *full() const {
    return reinterpret_cast<uint64_t *>(base + C::STAGES * C::OPND_BYTES + C::SF_SLOTS * C::SF_BYTES);
  }
  __device__ uint64_t *empty() const { return full() + C::STAGES; }
  __device__ uint64_t *sfull() const { return empty() + C::STAGES; }     // scales in shared memory
  __device__ uint64_t *sempty() const { return sfull() + C::SF_SLOTS; }  // scale slot copied to TMEM
  __device__ uint64_t *tfull() const { return sempty() + C::SF_SLOTS; }
  __device__ uint64_t *tempty() const { return tfull() + 1; }
  __device__ uint64_t *drain() const { return tempty() + 1; }
  __device__ uint32_t *tslot() const { return reinterpret_cast<uint32_t *>(drain() + 1); }
  __device__ volatile int *abort_flag() const { return reinterpret_cast<volatile int *>(tslot() + 1); }
};

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<const uint32_t *>(&v);
}

template <int MODE, bool PAIR>  // MODE TC_W4A4: bf16 out; TC_W4A4_SWIGLU: fused SwiGLU + NVFP4 requant
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                   const TcArgs p) {
  using C = Cfg<PAIR>;
  constexpr int STAGES = C::STAGES;
  constexpr int CL = C::CLUSTER;
  extern __shared__ uint8_t smem_raw[];
  const Smem<PAIR> sm{reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023))};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  volatile int *abort_flag = sm.abort_flag();
  // rank 0 of a pair is the leader: it issues the pair's MMAs and owns the
  // barriers both CTAs' loads and scale writes complete on
  const uint32_t rank = PAIR ? ptx::cluster_ctarank() : 0u;
  const bool leader = rank == 0;
  // shared::cluster address of one of this CTA's variables in CTA r
  auto in_cta = [&](const void *v, uint32_t r) { return ptx::map_to_cta(ptx::smem_u32(v), r); };
  auto give_up = [&]() {
    *abort_flag = 1;
    atomicCAS(p.status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
    if constexpr (PAIR) ptx::st_cluster_u32(in_cta(const_cast<const int *>(abort_flag), rank ^ 1u), 1u);
  };
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      // the operand producer's arrival (with the tile bytes) and one per
      // scale-writer warp of the pair
      ptx::mbar_init(&sm.full()[s], 1 + 4 * CL);
      ptx::mbar_init(&sm.empty()[s], 1);
    }
    for (int s = 0; s < C::SF_SLOTS; ++s) {
      ptx::mbar_init(&sm.sfull()[s], 1);
      ptx::mbar_init(&sm.sempty()[s], 4);         // one arrival per scale-writer warp of this CTA
    }
    ptx::mbar_init(sm.tfull(), 1);
    ptx::mbar_init(sm.tempty(), 8 * CL);          // one arrival per epilogue warp of the pair
    ptx::mbar_init(sm.drain(), 1);
    *abort_flag = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tm_a);
    ptx::prefetch_tensormap(&tm_b);
  }
  if (warp == 1) {
    if constexpr (PAIR) {
      ptx::tmem_alloc_pair(sm.tslot(), TMEM_COLS);
      ptx::tmem_relinquish_pair();
    } else {
      ptx::tmem_alloc(sm.tslot(), TMEM_COLS);
      ptx::tmem_relinquish();
    }
  }
  ptx::tc_fence_before();
  if constexpr (PAIR) ptx::cluster_sync();   // both CTAs' barriers exist before any remote arrival
  else __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *sm.tslot();

  const int cluster = blockIdx.x / CL, num_clusters = gridDim.x / CL;
  const int num_work = p.num_mg * p.num_n;
  const int ksteps_total = p.k >> 6;              // K / 64
  const int num_kb = (ksteps_total + KSTEPS - 1) / KSTEPS;
  const int cp4 = ksteps_total;                   // 512-byte scale tiles per 128-row block
  const int nrb_b = (p.n + 127) >> 7;             // 128-row blocks of B
  const uint32_t limit = p.wait_limit;
  // Work order: L2 groups of group_mp M tile groups; within an L2 group the
  // M tile group runs fastest, then the weight tile.  The clusters running at
  // one time then share a bounded set of activation rows (kept in L2 across
  // the group's sweep over the weights), and every weight tile is read once
  // per L2 group.
  auto tile_of = [&](int w, int &mt, int &nt) {
    const int per_group = p.group_mp * p.num_n;
    const int g = w / per_group;
    const int r = w - g * per_group;
    const int gsz = min(p.group_mp, p.num_mg - g * p.group_mp);
    nt = r / gsz;
    mt = (g * p.group_mp + (r - nt * gsz)) * CL + (int)rank;
  };

  uint32_t issued_mask = 0, issued_parity = 0;      // operand (warp 0) or scale (warp 14) copies in flight
  bool mma_issued = false;

  if (warp == 0) {
    if (ptx::elect_one()) {
      const uint64_t pol_a = ptx::l2_policy_evict_last();
      const uint64_t pol_b = ptx::l2_policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      // The first STAGES stages get their weight tiles before the previous
      // kernel on the stream has finished; the activation tiles follow once
      // it has.
      int pend_s[STAGES], pend_kb[STAGES], pend_mt[STAGES];
      int npend = 0, c = 0;
      bool flushed = false;
      // operand tile into this CTA's smem, counted on the leader's full barrier
      auto load_tile = [&](void *dst, const CUtensorMap *tm, int st, int x, int y, uint64_t pol) {
        if (PAIR && !leader)
          ptx::tma_load_2d_to_pair_bar(dst, tm, in_cta(&sm.full()[st], 0), x, y, pol);
        else
          ptx::tma_load_2d(dst, tm, &sm.full()[st], x, y, pol);
      };
      auto issue_a = [&](int st, int mt, int kb) { load_tile(sm.a(st), &tm_a, st, kb * (BK / 2), mt * BM, pol_a); };
      auto flush = [&]() {
        pdl_wait();
        for (int i = 0; i < npend; ++i) issue_a(pend_s[i], pend_mt[i], pend_kb[i]);
        flushed = true;
      };
      for (int w = cluster; w < num_work && !*abort_flag; w += num_clusters) {
        int mt, nt;
        tile_of(w, mt, nt);
        for (int kb = 0; kb < num_kb; ++kb, ++c) {
          if (c == STAGES && !flushed) flush();
          if (!ptx::mbar_wait_bounded(&sm.empty()[s], ph ^ 1u, limit, kDefaultTimeoutNs, abort_flag)) {
            give_up();
            break;
          }
          // the operand tiles land on the leader's barrier, which expects
          // both CTAs' A and B halves
          if (!PAIR) ptx::mbar_arrive_expect_tx(&sm.full()[s], A_BYTES + 2 * B_HALF);
          else if (leader) ptx::mbar_arrive_expect_tx(&sm.full()[s], 2 * (A_BYTES + B_HALF));
          if constexpr (PAIR) {
            load_tile(sm.b(s), &tm_b, s, kb * (BK / 2), nt * BN + (int)rank * 128, pol_b);
          } else {
            load_tile(sm.b(s), &tm_b, s, kb * (BK / 2), nt * BN, pol_b);
            load_tile(sm.b(s) + B_HALF, &tm_b, s, kb * (BK / 2), nt * BN + 128, pol_b);
          }
          if (c < STAGES) {
            pend_s[npend] = s;
            pend_kb[npend] = kb;
            pend_mt[npend] = mt;
            ++npend;
          } else {
            issue_a(s, mt, kb);
          }
          if (!PAIR || leader) {   // (the other CTA's tiles complete on the leader's barrier)
            issued_mask |= 1u << s;
            issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
          }
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
      if (!flushed) flush();
    }
  } else if (warp == 1) {
    pdl_wait();
    if (leader && ptx::elect_one()) {
      constexpr uint32_t idesc = idesc_nvfp4(BM * CL, BN);
      int g = 0;                                    // k-blocks of this CTA so far
      int it = 0;
      for (int w = cluster; w < num_work && !*abort_flag; w += num_clusters, ++it) {
        if (!ptx::mbar_wait_bounded(sm.tempty(), (uint32_t)(it & 1) ^ 1u, limit, kDefaultTimeoutNs, abort_flag)) {
          give_up();
          break;
        }
        ptx::tc_fence_after();
        bool ok = true;
        for (int kb = 0; kb < num_kb; ++kb, ++g) {
          const int s = g % STAGES;
          const uint32_t ph = (uint32_t)(g / STAGES) & 1u;
          // the stage's operand tiles (both CTAs' halves in a pair) and its
          // TMEM scale slot (usually written while the operands were in
          // flight)
          if (!ptx::mbar_wait_bounded(&sm.full()[s], ph, limit, kDefaultTimeoutNs, abort_flag)) {
            give_up();
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const int nk = min(KSTEPS, ksteps_total - kb * KSTEPS);
          const uint32_t sf = tmem + SF_COL + s * C::SF_SLOT;
          const uint32_t a_s = ptx::smem_u32(sm.a(s)), b_s = ptx::smem_u32(sm.b(s));
          for (int j = 0; j < nk; ++j) {
            const uint64_t ad = ptx::smem_desc(a_s + 32 * j, 16, 1024, 2);
            const uint64_t bd = ptx::smem_desc(b_s + 32 * j, 16, 1024, 2);
            if constexpr (PAIR)
              ptx::mma_nvfp4_pair(tmem + ACC_COL, ad, bd, idesc, sf + 4 * j, sf + SFB_OFF + 8 * j, (kb | j) != 0);
            else
              ptx::mma_nvfp4(tmem + ACC_COL, ad, bd, idesc, sf + 4 * j, sf + SFB_OFF + 8 * j, (kb | j) != 0);
          }
          mma_issued = true;
          // this stage and its scale slots are free again (in both CTAs)
          if constexpr (PAIR) {
            ptx::tc_commit_pair(ptx::smem_u32(&sm.empty()[s]));
            ptx::tc_commit_pair(in_cta(&sm.empty()[s], 1));
          } else {
            ptx::tc_commit(&sm.empty()[s]);
          }
        }
        if (!ok) break;
        if constexpr (PAIR) {
          ptx::tc_commit_pair(ptx::smem_u32(sm.tfull()));
          ptx::tc_commit_pair(in_cta(sm.tfull(), 1));
        } else {
          ptx::tc_commit(sm.tfull());
        }
      }
    }
  } else if (warp == 14) {
    // ---------------------------------------------------- scale producer
    // Loads each k-block's block scales (this CTA's activation rows and all
    // 256 weight rows of the tile) into the scale ring as soon as the
    // writers have copied the slot's previous contents to TMEM: it runs up
    // to a whole ring ahead of the operand producer.
    if (ptx::elect_one()) {
      pdl_wait();                                   // activation scales come from the previous kernel
      const uint64_t pol_a = ptx::l2_policy_evict_last();
      const uint64_t pol_b = ptx::l2_policy_evict_first();
      int s = 0;
      uint32_t ph = 0;
      for (int w = cluster; w < num_work && !*abort_flag; w += num_clusters) {
        int mt, nt;
        tile_of(w, mt, nt);
        const int nbv = min(2, nrb_b - nt * 2);
        for (int kb = 0; kb < num_kb; ++kb) {
          if (!ptx::mbar_wait_bounded(&sm.sempty()[s], ph ^ 1u, limit, kDefaultTimeoutNs, abort_flag)) {
            give_up();
            break;
          }
          const int nk = min(KSTEPS, ksteps_total - kb * KSTEPS);
          const uint32_t sfa_bytes = mt < p.num_m ? (uint32_t)nk * 512u : 0u;
          ptx::mbar_arrive_expect_tx(&sm.sfull()[s], sfa_bytes + (uint32_t)nk * 512u * nbv);
          if (sfa_bytes)
            ptx::bulk_load(sm.sfa(s), p.sfa + ((size_t)mt * cp4 + kb * KSTEPS) * 512, sfa_bytes, &sm.sfull()[s],
                           pol_a);
          // every CTA's MMA share reads the scales of all 256 weight rows
          for (int rb = 0; rb < nbv; ++rb)
            ptx::bulk_load(sm.sfb(s) + rb * (KSTEPS * 512), p.sfb + ((size_t)(nt * 2 + rb) * cp4 + kb * KSTEPS) * 512,
                           nk * 512u, &sm.sfull()[s], pol_b);
          issued_mask |= 1u << s;
          issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
          if (++s == C::SF_SLOTS) { s = 0; ph ^= 1u; }
        }
      }
    }
  } else if (warp >= 10) {
    // ------------------------------------------------------ scale writers
    // Warp w fills TMEM lane quarter w % 4 (a warp reaches only its own
    // quarter) of the stage's scale slot from registers with tcgen05.st: the
    // same 4 columns x 32 lanes per 512-byte scale tile that a warpx4 copy
    // of the tile would write, replicated in every quarter.  These stores
    // do not queue behind the MMAs in the tensor pipe as tcgen05.cp does.
    // In a pair each CTA fills its own TMEM: the scales of its own 128
    // activation rows and of all 256 weight rows.
    pdl_wait();
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    int g = 0;                                      // k-blocks of this CTA so far
    for (int w = cluster; w < num_work && !*abort_flag; w += num_clusters) {
      bool ok = true;
      for (int kb = 0; kb < num_kb; ++kb, ++g) {
        const int ss = g % C::SF_SLOTS, t = g % C::T_SLOTS;
        // the k-block's scales in shared memory, and a free TMEM scale slot:
        // the MMAs of k-block g - T_SLOTS (its stage's empty barrier) have
        // committed
        const int gp = g - C::T_SLOTS;
        if (!ptx::mbar_wait_bounded(&sm.sfull()[ss], (uint32_t)(g / C::SF_SLOTS) & 1u, limit, kDefaultTimeoutNs,
                                    abort_flag) ||
            (gp >= 0 && !ptx::mbar_wait_bounded(&sm.empty()[gp % STAGES], (uint32_t)(gp / STAGES) & 1u, limit,
                                                kDefaultTimeoutNs, abort_flag))) {
          give_up();
          ok = false;
          break;
        }
        ptx::tc_fence_after();
        // lane l takes bytes 16l .. 16l+15 of every scale tile of the stage
        // (rows l, l+32, l+64, l+96; 4 scales each).  Tiles past the K tail
        // or the last weight block hold stale bytes the MMAs never use.
        const uint8_t *sfa = sm.sfa(ss) + lane * 16, *sfb = sm.sfb(ss) + lane * 16;
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
        const uint32_t sf = tmem + lane_off + SF_COL + t * C::SF_SLOT;
        ptx::tmem_st16(sf, ra);
        ptx::tmem_st16(sf + SFB_OFF, rb0);
        ptx::tmem_st16(sf + SFB_OFF + 16, rb1);
        ptx::tmem_wait_st();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(&sm.sempty()[ss]);       // the smem scale slot may be refilled
          // the k-block's scale slot is ready: one arrival on its stage's
          // full barrier (the leader's in a pair)
          if constexpr (PAIR) ptx::mbar_arrive_remote(in_cta(&sm.full()[t], 0));
          else ptx::mbar_arrive(&sm.full()[t]);
        }
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
    const uint32_t tempty_leader = PAIR ? in_cta(sm.tempty(), 0) : 0u;
    const float alpha = __ldg(p.alpha);
    int it = 0;
    for (int w = cluster; w < num_work; w += num_clusters, ++it) {
      if (!ptx::mbar_wait_bounded(sm.tfull(), (uint32_t)(it & 1), limit, kDefaultTimeoutNs, abort_flag)) {
        give_up();
        break;
      }
      ptx::tc_fence_after();
      uint32_t acc[128];
#pragma unroll
      for (int c = 0; c < 8; ++c) ptx::tmem_ld16(t_base + 16 * c, *reinterpret_cast<uint32_t(*)[16]>(&acc[16 * c]));
      ptx::tmem_wait_ld();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) {                          // accumulator free for the next tile
        if constexpr (PAIR) ptx::mbar_arrive_remote(tempty_leader);
        else ptx::mbar_arrive(sm.tempty());
      }

      int mt, nt;
      tile_of(w, mt, nt);
      if (mt >= p.num_m) continue;              // odd tail: this CTA's rows are past M
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
    // the CTA is gone.  In a pair some of a CTA's copies complete on the
    // other CTA's barrier: a short settle time covers those.  An operand
    // stage whose scale writers gave up before arriving never completes its
    // phase; its wait runs out its bound, far longer than any copy's flight.
    if ((warp == 0 || warp == 14) && issued_mask) {
      uint64_t *bars = warp == 0 ? sm.full() : sm.sfull();
      for (int s = 0; s < (warp == 0 ? STAGES : C::SF_SLOTS); ++s)
        if (issued_mask & (1u << s)) {
          volatile int no_abort = 0;
          ptx::mbar_wait_bounded(&bars[s], (issued_parity >> s) & 1u, 0, kDrainNs, &no_abort);
        }
    }
    if (warp == 1 && mma_issued) {
      volatile int no_abort = 0;
      if constexpr (PAIR) ptx::tc_commit_pair(ptx::smem_u32(sm.drain()));
      else ptx::tc_commit(sm.drain());
      ptx::mbar_wait_bounded(sm.drain(), 0, 0, kDrainNs, &no_abort);
    }
    if (PAIR && threadIdx.x == 0) {
      const uint64_t t0 = ptx::globaltimer();
      while (ptx::globaltimer() - t0 < kSettleNs) __nanosleep(1000);
    }
  }
  ptx::tc_fence_before();
  if constexpr (PAIR) ptx::cluster_sync();   // the partner's MMAs and copies no longer touch this CTA
  else __syncthreads();
  ptx::tc_fence_after();
  if (warp == 1) {
    if constexpr (PAIR) ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
    else ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
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
                   uint32_t box_rows, int swizzle_bytes) {
  auto encode = get_encode();
  if (!encode) return false;
  cuuint64_t dims[2] = {(cuuint64_t)row_bytes, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)row_bytes};
  cuuint32_t box[2] = {box_bytes, box_rows};
  cuuint32_t estr[2] = {1u, 1u};
  return encode(tm, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(ptr), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE,
                swizzle_bytes == 128  ? CU_TENSOR_MAP_SWIZZLE_128B
                : swizzle_bytes == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                      : CU_TENSOR_MAP_SWIZZLE_NONE,
                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int num_sms() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
  int v = cache[dev].load(std::memory_order_relaxed);
  if (!v) {
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0) v = 148;
    cache[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

namespace {

template <int MODE, bool PAIR>
cudaError_t launch_mode(const uint8_t *a, const uint8_t *a_sf, const uint8_t *b, const uint8_t *b_sf,
                        const float *alpha, const float *out_gs, uint16_t *d, uint8_t *out_fp4,
                        uint8_t *out_sf, int64_t m, int64_t n, int64_t k, uint32_t wait_limit,
                        cudaStream_t st, const float *rs) {
  using C = Cfg<PAIR>;
  constexpr int CL = C::CLUSTER;
  // clusters of this kernel the device holds at once, per device
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CL;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = PAIR ? 2 : 1;
  int mc = max_clusters[dev].load(std::memory_order_relaxed);
  if (!mc) {
    cudaError_t e = cudaFuncSetAttribute(tc_gemm_kernel<MODE, PAIR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    mc = num_sms() / CL;                 // one CTA per SM
    if (PAIR) {
      cfg.gridDim = dim3(CL * mc);
      int nc = 0;
      e = cudaOccupancyMaxActiveClusters(&nc, tc_gemm_kernel<MODE, PAIR>, &cfg);
      if (e == cudaSuccess && nc > 0 && nc < mc) mc = nc;
    }
    max_clusters[dev].store(mc, std::memory_order_relaxed);
  }
  CUtensorMap tm_a, tm_b;
  // codes [rows, k/2] bytes; box 128 bytes of K x 128 rows (activation rows
  // or half a weight tile), 128-byte swizzle
  if (!make_byte_map(&tm_a, a, m, k / 2, 128, BM, 128) || !make_byte_map(&tm_b, b, n, k / 2, 128, 128, 128))
    return cudaErrorInvalidValue;
  TcArgs args{a_sf, b_sf, alpha, out_gs, d, out_fp4, out_sf, (int32_t)m, (int32_t)n, (int32_t)k,
              (int32_t)((m + BM - 1) / BM), (int32_t)((n + BN - 1) / BN), 0, wait_limit, device_status_ptr(), rs};
  if (!args.status) return cudaErrorInvalidValue;
  args.num_mg = (args.num_m + CL - 1) / CL;
  {
    // Activation rows of one L2 group: at most ~32 MiB, so that, together
    // with the weight tiles in flight (and any copies the two dies' L2
    // halves keep), they stay in the 129 MB L2 while the group sweeps the
    // weights.
    const int64_t mg_bytes = (int64_t)CL * BM * (k / 2);
    const int64_t g = (int64_t(32) << 20) / mg_bytes;
    args.group_mp = (int32_t)(g < 1 ? 1 : g > args.num_mg ? args.num_mg : g);
  }
  const int work = args.num_mg * args.num_n;
  const int clusters = work < mc ? work : mc;
  cfg.gridDim = dim3(CL * clusters);
  return cudaLaunchKernelEx(&cfg, tc_gemm_kernel<MODE, PAIR>, tm_a, tm_b, args);
}

}  // namespace

bool tc_supported(TcMode mode, int64_t m, int64_t n, int64_t k) {
  if (mode == TC_W4A16) return false;
  if (k % 64 != 0 || n % 32 != 0 || m <= 0) return false;
  if (mode == TC_W4A4_SWIGLU && n % 128 != 0) return false;
  if (m > (1 << 30) || n > (1 << 30) || k > (1 << 30)) return false;
  return get_encode() != nullptr;
}

cudaError_t launch_tc(TcMode mode, bool pair, const void *a, const uint8_t *a_sf, const uint8_t *b,
                      const uint8_t *b_sf, const float *alpha, const float *out_gs, uint16_t *d,
                      uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n, int64_t k,
                      uint32_t wait_limit, cudaStream_t st, const float *a_row_scale) {
  if (!tc_supported(mode, m, n, k)) return cudaErrorNotSupported;
  const uint8_t *a8 = static_cast<const uint8_t *>(a);
  if (mode == TC_W4A4)
    return pair ? launch_mode<TC_W4A4, true>(a8, a_sf, b, b_sf, alpha, out_gs, d, out_fp4, out_sf, m, n, k,
                                             wait_limit, st, a_row_scale)
                : launch_mode<TC_W4A4, false>(a8, a_sf, b, b_sf, alpha, out_gs, d, out_fp4, out_sf, m, n, k,
                                              wait_limit, st, a_row_scale);
  return pair ? launch_mode<TC_W4A4_SWIGLU, true>(a8, a_sf, b, b_sf, alpha, out_gs, d, out_fp4, out_sf, m, n, k,
                                                  wait_limit, st, a_row_scale)
              : launch_mode<TC_W4A4_SWIGLU, false>(a8, a_sf, b, b_sf, alpha, out_gs, d, out_fp4, out_sf, m, n,
                                                   k, wait_limit, st, a_row_scale);
}

}  // namespace nvfp4
