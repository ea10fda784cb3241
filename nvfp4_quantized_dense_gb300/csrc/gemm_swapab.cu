// Decode-sized NVFP4 GEMMs on the tensor cores with the weight as the MMA's
// 128-row operand ("swap AB"): D^T[n, t] = sum_k W[n, k] * X[t, k], with the
// tokens (M <= 64) as the MMA's N = 16, 32 or 64.  The weight stream is the
// roofline, so the kernel is a deep TMA pipeline (6-8 stages of 16 KB weight
// tiles per SM) feeding one MMA issuer.
//
// Work split, when there are at least twice as many SMs as weight tiles and
// C of them per tile fill at least 90 % of the SMs: clusters of C CTAs, one
// tile per cluster, the tile's
// k-blocks cut into C contiguous runs; the cluster's other CTAs publish their
// fp32 partial tiles in their own shared memory and its first CTA adds them
// in K order through distributed shared memory and runs the epilogue -- no
// workspace and no global round trip after the last MMA.
// Otherwise: the (128-row weight tile, 256-wide k-block) pairs are laid out
// tile-major and cut into one contiguous, equal run per CTA, so every SM
// streams the same number of weight bytes.  A CTA's run crosses tile
// boundaries; each piece of a tile it covers is a fragment.  A tile covered by
// one CTA is finished in place.  Otherwise each fragment writes its fp32
// partial tile to the caller's workspace and bumps the tile's arrival
// counter; the fragment that arrives last sums the partials in K order (so
// the result does not depend on which CTA finishes last), resets the counter
// to 0 and runs the epilogue.  The workspace must be zero-filled once before
// its first use; the kernel leaves its counters at zero after every complete
// call.
//
// Activation quantize folded in (decode gate_up): given bf16 x, the kernel
// writes x's NVFP4 codes and swizzled scales itself, exactly as
// nvfp4_quantize, into the buffers its activation loads read.  The CTAs
// first through the grid-dependency wait take chunks of x's 16-element
// blocks from a counter in the workspace (one block per epilogue thread),
// then chunks of the zero padding rows of the scale block; a producer issues
// its activation halves once every chunk of x's blocks has been counted.
// This takes the separate quantize launch, and the grid completion between
// it and the GEMM, off the decode chain.  The last CTA done with the
// counters resets them.
//
// Roles per CTA (192 threads, one CTA per SM): warp 0 TMA producer,
// warp 1 TMEM owner + MMA issuer (double-buffered accumulators), warps 2..5
// phase A (with the fold) and the epilogue (TMEM lane = weight row).
// Bounded waits as in gemm_tc.cu.
#include <algorithm>
#include <atomic>

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
constexpr int XCHUNK = 128;          // phase A: blocks of x per chunk (one per epilogue thread)
constexpr int PCHUNK = 1024;         // phase A: padding words of the scale block per chunk

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
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
};

struct SwapArgs {
  const uint8_t *sfw;   // weight scales, swizzled over N rows
  const uint8_t *sfx;   // activation scales, swizzled over M rows (one 128-row block)
  const float *alpha;
  const float *out_gs;
  uint16_t *d;          // bf16 [M, N]
  uint8_t *out_fp4;     // fused: [M, N/4]
  uint8_t *out_sf;      // fused: swizzled over M rows, N/32 columns
  float *partials;      // [grid][maxfrag][NT][128] fp32 (tiles shared by CTAs)
  int *counters;        // [tiles] arrival counters
  int32_t m, n, k;
  int32_t tiles, kb_total;   // weight tiles, k-blocks per tile
  int32_t grid, maxfrag;     // CTAs, fragment slots per CTA (split tiles)
  int32_t whole, split_tiles;   // mixed split: whole tiles per CTA, tiles shared by CTAs
  int32_t split_ok;          // 0: no workspace, every CTA owns whole tiles
  int32_t cl;                // > 1: clusters of cl CTAs, one tile each, reduced in shared memory
  uint32_t wait_limit;
  int *status;
  const float *rs;      // optional per-token activation dequant factor [M]
  // activation quantize folded in (xsrc != nullptr)
  const uint16_t *xsrc;  // bf16 x [M, K]
  const float *gs_x;     // x global scale
  uint8_t *xq;           // x codes [M, K/2] (what tm_x reads)
  uint8_t *xs;           // x scales, swizzled over M rows (what sfx reads)
  uint32_t *xsync;       // [0] chunk counter, [1] x chunks done, [2] CTAs done with both
  int32_t xchunks, pchunks;   // chunks of x's blocks (counted), of scale padding (not)
};

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// A CTA's fragments: the mixed split with a workspace, whole tiles without.
struct WorkIter {
  bool use_mixed;
  MixedIter mi;
  FragIter fi;
  __device__ __forceinline__ WorkIter(bool m, const MixedPartition &mp, int64_t cta, int64_t start, int64_t end,
                                      int64_t kbt)
      : use_mixed(m), mi(mp, cta), fi{start, end, kbt} {}
  __device__ __forceinline__ bool next(int &tile, int &kb0, int &kb1) {
    return use_mixed ? mi.next(tile, kb0, kb1) : fi.next(tile, kb0, kb1);
  }
};

// FOLD: the activation quantize folded in (a separate instance, so that the
// plain kernel carries none of its code)
template <int MODE, int NT, bool FOLD = false>
__global__ void __launch_bounds__(kThreads, 1)
    swapab_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
                  const SwapArgs p) {
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
  uint64_t *parts = drain + 1;           // cluster split: [0] partials published, [1] partials read
  uint32_t *tslot = reinterpret_cast<uint32_t *>(parts + 2);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(tslot + 1);
  volatile int *last_flag = abort_flag + 1;
  volatile int *x_phase_done = abort_flag + 2;
  volatile uint32_t *x_grab = reinterpret_cast<volatile uint32_t *>(abort_flag + 3);   // two slots
  auto st_w = [&](int s) { return base + s * C::STAGE_BYTES; };
  auto st_x = [&](int s) { return st_w(s) + W_BYTES; };
  auto st_sfw = [&](int s) { return st_x(s) + C::X_BYTES; };
  auto st_sfx = [&](int s) { return st_sfw(s) + SFW_BYTES; };

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_trigger();
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
    ptx::mbar_init(&parts[0], 128 * (p.cl > 1 ? p.cl - 1 : 1));   // every epilogue thread of the others
    ptx::mbar_init(&parts[1], 128);                               // every epilogue thread of the first CTA
    *abort_flag = 0;
    *x_phase_done = 0;
    ptx::fence_barrier_init();
    ptx::prefetch_tensormap(&tm_w);
    ptx::prefetch_tensormap(&tm_x);
  }
  if (warp == 1) {
    ptx::tmem_alloc(tslot, C::TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  if (p.cl > 1) ptx::cluster_sync();   // every CTA's barriers exist before any remote arrival
  else __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;

  // With a workspace: the mixed split (the tiles shared by CTAs first, then
  // whole tiles of its own), so that no CTA ends its run with a reduction.
  // Without: whole tiles per CTA.
  const MixedPartition mixed{p.kb_total, p.grid, p.whole, p.split_tiles};
  const Partition part{(int64_t)p.tiles * p.kb_total, p.grid, p.kb_total, true, p.tiles};
  int64_t my_start = part.start(blockIdx.x), my_end = part.start(blockIdx.x + 1);
  if (p.cl > 1) {   // cluster split: tile blockIdx / cl, this CTA's run of its k-blocks
    const int64_t tile = blockIdx.x / p.cl, j = blockIdx.x % p.cl;
    my_start = tile * p.kb_total + p.kb_total * j / p.cl;
    my_end = tile * p.kb_total + p.kb_total * (j + 1) / p.cl;
  }
  auto work = [&]() { return WorkIter(p.split_ok != 0, mixed, blockIdx.x, my_start, my_end, p.kb_total); };
  const int ksteps_total = p.k >> 6;
  const int cp4 = ksteps_total;          // 512-byte scale tiles per 128-row block
  const uint32_t limit = p.wait_limit;
  uint32_t issued_mask = 0, issued_parity = 0;
  bool mma_issued = false;

  if (warp == 0) {
    if (ptx::elect_one()) {
      const uint64_t pol_w = ptx::l2_policy_evict_first();
      const uint64_t pol_x = ptx::l2_policy_evict_last();
      int s = 0;
      uint32_t ph = 0;
      WorkIter fi = work();
      int tile, kb0, kb1;
      // The first STAGES stages get their weight tiles before the previous
      // kernel on the stream has finished; their activation tiles (that
      // kernel's output) follow once it has.
      int pend_s[STAGES], pend_kb[STAGES];
      int npend = 0, c = 0;
      bool flushed = false;
      auto issue_x = [&](int st, int kb) {
        const int nk = min(KSTEPS, ksteps_total - kb * KSTEPS);
        ptx::tma_load_2d(st_x(st), &tm_x, &full[st], kb * (BK / 2), 0, pol_x);
        ptx::bulk_load(st_sfx(st), p.sfx + (size_t)kb * KSTEPS * 512, nk * 512u, &full[st], pol_x);
      };
      auto flush = [&]() {
        pdl_wait();
        // with the fold: x's blocks are quantized by the first CTAs through
        // the wait (after a give-up the halves still go out, reading
        // whatever the buffers hold, so that every stage completes)
        if constexpr (FOLD) {
          if (!ptx::counter_wait_bounded(&p.xsync[1], (uint32_t)p.xchunks, limit, kTimeoutNs, abort_flag)) {
            *abort_flag = 1;
            atomicCAS(p.status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
          }
        }
        for (int i = 0; i < npend; ++i) issue_x(pend_s[i], pend_kb[i]);
        flushed = true;
      };
      while (!*abort_flag && fi.next(tile, kb0, kb1)) {
        for (int kb = kb0; kb < kb1; ++kb, ++c) {
          if (c == STAGES && !flushed) flush();
          if (!ptx::mbar_wait_bounded(&empty[s], ph ^ 1u, limit, kTimeoutNs, abort_flag)) {
            *abort_flag = 1;
            atomicCAS(p.status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
            break;
          }
          const int nk = min(KSTEPS, ksteps_total - kb * KSTEPS);
          ptx::mbar_arrive_expect_tx(&full[s], W_BYTES + C::X_BYTES + 2u * (uint32_t)nk * 512u);
          ptx::tma_load_2d(st_w(s), &tm_w, &full[s], kb * (BK / 2), tile * 128, pol_w);
          ptx::bulk_load(st_sfw(s), p.sfw + ((size_t)tile * cp4 + kb * KSTEPS) * 512, nk * 512u, &full[s],
                         pol_w);
          if (c < STAGES) {
            pend_s[npend] = s;
            pend_kb[npend] = kb;
            ++npend;
          } else {
            issue_x(s, kb);
          }
          issued_mask |= 1u << s;
          issued_parity = (issued_parity & ~(1u << s)) | (ph << s);
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
      }
      if (!flushed) flush();
      if constexpr (FOLD) {
        // This CTA reads and takes no phase-A counter any more once its own
        // epilogue warps are past phase A; the last CTA to get here resets
        // the counters for the next call.
        uint64_t t0 = 0;
        bool ok = true;
        for (uint32_t polls = 1; !*x_phase_done && !*abort_flag; ++polls) {
          if (limit ? polls >= limit : false) ok = false;
          if (!limit && (polls & 63u) == 0) {
            const uint64_t now = ptx::globaltimer();
            if (t0 == 0) t0 = now;
            else if (now - t0 > kTimeoutNs) ok = false;
          }
          if (!ok) {
            *abort_flag = 1;
            atomicCAS(p.status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
            break;
          }
          __nanosleep(64);
        }
        if (ok && !*abort_flag &&
            atom_add_acq_rel_gpu(reinterpret_cast<int *>(&p.xsync[2]), 1) == (uint32_t)p.grid - 1) {
          p.xsync[0] = 0;
          p.xsync[1] = 0;
          asm volatile("fence.acq_rel.gpu;" ::: "memory");
          p.xsync[2] = 0;
        }
      }
    }
  } else if (warp == 1) {
    pdl_wait();
    if (ptx::elect_one()) {
      // kind::mxf4nvf4, E2M1 x E2M1, UE4M3 scales, M = 128 (weights), N = NT (tokens)
      constexpr uint32_t idesc = (1u << 7) | (1u << 10) | ((uint32_t)(NT >> 3) << 17) | (8u << 24);
      int s = 0;
      uint32_t ph = 0;
      int it = 0;
      WorkIter fi = work();
      int tile, kb0, kb1;
      for (; !*abort_flag && fi.next(tile, kb0, kb1); ++it) {
        const int ab = it & 1;
        if (!ptx::mbar_wait_bounded(&tempty[ab], (uint32_t)((it >> 1) & 1) ^ 1u, limit, kTimeoutNs, abort_flag)) {
          *abort_flag = 1;
          atomicCAS(p.status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
          break;
        }
        ptx::tc_fence_after();
        bool ok = true;
        for (int kb = kb0; kb < kb1; ++kb) {
          if (!ptx::mbar_wait_bounded(&full[s], ph, limit, kTimeoutNs, abort_flag)) {
            *abort_flag = 1;
            atomicCAS(p.status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
            ok = false;
            break;
          }
          ptx::tc_fence_after();
          const int nk = min(KSTEPS, ksteps_total - kb * KSTEPS);
          const uint32_t sfw_s = ptx::smem_u32(st_sfw(s)), sfx_s = ptx::smem_u32(st_sfx(s));
          for (int j = 0; j < nk; ++j) {
            ptx::tmem_cp_32x128b_x4(tmem + C::SFW_COL + 4 * j, ptx::smem_desc(sfw_s + 512 * j, 0, 128, 0));
            ptx::tmem_cp_32x128b_x4(tmem + C::SFX_COL + 4 * j, ptx::smem_desc(sfx_s + 512 * j, 0, 128, 0));
          }
          const uint32_t w_s = ptx::smem_u32(st_w(s)), x_s = ptx::smem_u32(st_x(s));
          for (int j = 0; j < nk; ++j)
            ptx::mma_nvfp4(tmem + ab * NT, ptx::smem_desc(w_s + 32 * j, 16, 1024, 2),
                           ptx::smem_desc(x_s + 32 * j, 16, 1024, 2), idesc, tmem + C::SFW_COL + 4 * j,
                           tmem + C::SFX_COL + 4 * j, (kb != kb0) || (j != 0));
          mma_issued = true;
          ptx::tc_commit(&empty[s]);
          if (++s == STAGES) { s = 0; ph ^= 1u; }
        }
        if (!ok) break;
        ptx::tc_commit(&tfull[ab]);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();
    const int q = warp & 3;
    const int r = q * 32 + lane;                 // weight row within the tile
    const int et = threadIdx.x - 64;             // 0..127 across the epilogue warps
    if constexpr (FOLD) {
      // phase A: chunks of x's blocks (counted), then chunks of the padding
      // rows m..127 of the scale block (zero), until none is left
      const int cols = p.k >> 4, xcp4 = cols >> 2;
      const float gsx = __ldg(p.gs_x);
      const int64_t nblk = (int64_t)p.m * cols, npad = (int64_t)(128 - p.m) * xcp4;
      for (int par = 0;; par ^= 1) {
        if (et == 0) x_grab[par] = atomicAdd(&p.xsync[0], 1u);
        epi_bar();
        const uint32_t ci = x_grab[par];
        if (ci >= (uint32_t)(p.xchunks + p.pchunks)) break;
        if (ci < (uint32_t)p.xchunks) {
          const int64_t b = (int64_t)ci * XCHUNK + et;
          if (b < nblk) {
            const int row = (int)(b / cols), j = (int)(b - (int64_t)row * cols);
            const uint4 *src = reinterpret_cast<const uint4 *>(p.xsrc + (size_t)row * p.k + 16 * j);
            const uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
            const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
            float xv[16];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              xv[2 * i] = bf16_lo(w[i]);
              xv[2 * i + 1] = bf16_hi(w[i]);
            }
            uint32_t lo, hi;
            const uint32_t sf = quantize_block16(xv, gsx, lo, hi);
            *reinterpret_cast<uint2 *>(p.xq + (size_t)row * (p.k >> 1) + 8 * j) = make_uint2(lo, hi);
            p.xs[sf_swizzled_offset(row, j, xcp4)] = (uint8_t)sf;
          }
          ptx::fence_proxy_async_global();     // these stores -> the activation TMA reads
          epi_bar();
          if (et == 0) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(&p.xsync[1]) : "memory");
        } else {
          for (int i = et; i < PCHUNK; i += 128) {
            const int64_t w = (int64_t)(ci - p.xchunks) * PCHUNK + i;
            if (w < npad) {
              const int row = p.m + (int)(w / xcp4), j4 = (int)(w % xcp4);
              *reinterpret_cast<uint32_t *>(p.xs + sf_swizzled_offset(row, 4 * j4, xcp4)) = 0u;
            }
          }
        }
      }
      if (et == 0) *x_phase_done = 1;
    }
    const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16);
    const float alpha = __ldg(p.alpha);
    const int mt = min(p.m, NT);
    int it = 0;
    WorkIter fi = work();
    int tile, kb0, kb1;
    for (; fi.next(tile, kb0, kb1); ++it) {
      const int ab = it & 1;
      const bool got =
          ptx::mbar_wait_bounded(&tfull[ab], (uint32_t)((it >> 1) & 1), limit, kTimeoutNs, abort_flag);
      if (!got) {
        *abort_flag = 1;
        atomicCAS(p.status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
      }
      if (ptx::bar_any(1, 128, !got || *abort_flag)) break;   // the four warps leave together
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
      ptx::mbar_arrive(&tempty[ab]);              // accumulator buffer free again

      // CTAs sharing this tile: the owners of its first and last k-block
      const bool split_tile = p.split_ok != 0 && mixed.is_split(tile);
      const int64_t c_first = split_tile ? mixed.cta_of((int64_t)tile * p.kb_total) : blockIdx.x;
      const int64_t c_last = split_tile ? mixed.cta_of((int64_t)tile * p.kb_total + p.kb_total - 1) : blockIdx.x;
      if (c_last > c_first) {
        // partial slot of contributor c: its fragment index is 0 except for
        // c_first (every later contributor's run starts inside this tile)
        const int f_first = tile - (int)(mixed.start(c_first) / p.kb_total);
        auto slot = [&](int64_t c) {
          return p.partials + ((size_t)c * p.maxfrag + (c == c_first ? f_first : 0)) * NT * 128;
        };
        float *mine = slot(blockIdx.x);
#pragma unroll
        for (int t = 0; t < NT; ++t)
          if (t < mt) mine[t * 128 + r] = v[t];
        epi_bar();                    // every partial write of the CTA precedes the release below
        if (et == 0)
          *last_flag = atom_add_acq_rel_gpu(&p.counters[tile], 1) == (uint32_t)(c_last - c_first);
        epi_bar();
        if (!*last_flag) continue;
        sum_partials_in_k_order<NT>(v, c_first, c_last, mt, r, slot);
        if (et == 0) p.counters[tile] = 0;
      }

      if (p.cl > 1) {
        // the cluster's other CTAs publish their partials (row r, pitch
        // PITCH, in their own staging buffer); the first CTA adds them in
        // rank order -- K order -- and runs the epilogue
        const uint32_t crank = blockIdx.x % p.cl;
        bool ok = true;
        if (crank != 0) {
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t < mt) s_out[r * C::PITCH + t] = v[t];
          ptx::mbar_arrive_remote_release_cluster(ptx::map_to_cta(ptx::smem_u32(&parts[0]), 0));
          ok = ptx::mbar_wait_bounded(&parts[1], 0, limit, kTimeoutNs, abort_flag);    // read by the first CTA
        } else {
          ok = ptx::mbar_wait_bounded_acq_cluster(&parts[0], 0, limit, kTimeoutNs, abort_flag);
          if (ok) {
            for (int c = 1; c < p.cl; ++c) {
              const uint32_t src = ptx::map_to_cta(ptx::smem_u32(s_out + r * C::PITCH), (uint32_t)c);
#pragma unroll
              for (int t = 0; t < NT; ++t)
                if (t < mt) v[t] += ptx::ld_cluster_f32(src + 4u * t);
            }
            for (int c = 1; c < p.cl; ++c) ptx::mbar_arrive_remote(ptx::map_to_cta(ptx::smem_u32(&parts[1]), (uint32_t)c));
          }
        }
        if (!ok) {
          *abort_flag = 1;
          atomicCAS(p.status, 0, (int)NVFP4_ERR_DEVICE_TIMEOUT);
        }
        if (ptx::bar_any(1, 128, !ok)) break;
        if (crank != 0) continue;
      }

      const int n = tile * 128 + r;
      if constexpr (MODE == TC_W4A4) {
        if (n < p.n) {
#pragma unroll
          for (int t = 0; t < NT; ++t)
            if (t < mt) {
              const float at = p.rs ? alpha * p.rs[t] : alpha;
              const __nv_bfloat16 o = __float2bfloat16_rn(at * v[t]);
              p.d[(size_t)t * p.n + n] = *reinterpret_cast<const uint16_t *>(&o);
            }
        }
      } else {
        // rows 0..63 of the tile are up, 64..127 gate, for features 64*tile + (0..63)
#pragma unroll
        for (int t = 0; t < NT; ++t) s_out[r * C::PITCH + t] = (p.rs && t < mt ? alpha * p.rs[t] : alpha) * v[t];
        epi_bar();
        // SwiGLU one element per thread; h replaces the up value in s_out
        for (int idx = et; idx < mt * 64; idx += 128) {
          const int t = idx >> 6, i = idx & 63;
          s_out[i * C::PITCH + t] = silu_mul_fast(s_out[(64 + i) * C::PITCH + t], s_out[i * C::PITCH + t]);
        }
        epi_bar();
        const int inter = p.n >> 1;
        const int ocp4 = ((inter >> 4) + 3) >> 2;
        const float gs = __ldg(p.out_gs);
        for (int idx = et; idx < mt * 4; idx += 128) {
          const int t = idx >> 2, qb = idx & 3;
          float h[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) h[i] = s_out[(16 * qb + i) * C::PITCH + t];
          uint32_t lo, hi;
          const uint32_t sf = quantize_block16(h, gs, lo, hi);
          const int f = 64 * tile + 16 * qb;
          *reinterpret_cast<uint2 *>(p.out_fp4 + (size_t)t * (inter >> 1) + f / 2) = make_uint2(lo, hi);
          p.out_sf[sf_swizzled_offset(t, f >> 4, ocp4)] = (uint8_t)sf;
        }
        // padding rows of the 128-row scale block: zero this tile's 4 columns
        const int mpad = (p.m + 127) & ~127;
        for (int t = p.m + et; t < mpad; t += 128)
          *reinterpret_cast<uint32_t *>(p.out_sf + sf_swizzled_offset(t, tile * 4, ocp4)) = 0u;
        epi_bar();
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
  if (p.cl > 1) ptx::cluster_sync();   // no CTA leaves while the first CTA may still read its partials
  ptx::tc_fence_after();
  if (warp == 1) ptx::tmem_dealloc(tmem, C::TMEM_COLS);
}

struct Plan {
  int nt, tiles, kb_total, grid, maxfrag, whole, split_tiles;
  int cl;                 // > 1: cluster split (one tile per cluster of cl CTAs)
  size_t ws_bytes;        // workspace the mixed split needs (0: no tile shared)
  bool split;             // mixed split (false: whole tiles per CTA, no workspace)
};

// Clusters of cl CTAs of the NT instance the device holds at once (both
// modes use the same resources); without a device, as many as the SMs allow.
int max_clusters(int nt, int cl) {
  static std::atomic<int> cache[64][3][9];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms() / cl;
  const int ni = nt == 16 ? 0 : nt == 32 ? 1 : 2;
  int v = cache[dev][ni][cl].load(std::memory_order_relaxed);
  if (v) return v;
  auto query = [&](auto kernel, uint32_t smem) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return 0;
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(cl * (num_sms() / cl));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    return cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess ? n : 0;
  };
  v = ni == 0 ? query(swapab_kernel<TC_W4A4, 16>, Cfg<16>::SMEM_BYTES)
      : ni == 1 ? query(swapab_kernel<TC_W4A4, 32>, Cfg<32>::SMEM_BYTES)
                : query(swapab_kernel<TC_W4A4, 64>, Cfg<64>::SMEM_BYTES);
  if (v <= 0) v = 1;
  cache[dev][ni][cl].store(v, std::memory_order_relaxed);
  return v;
}


Plan make_plan(int64_t m, int64_t n, int64_t k) {
  Plan pl{};
  pl.nt = m <= 16 ? 16 : m <= 32 ? 32 : 64;
  pl.tiles = (int)((n + 127) / 128);
  pl.kb_total = (int)((k + BK - 1) / BK);
  const int sms = num_sms();
  // Cluster split when the tiles are at most half the SMs: cl CTAs per tile
  // (at most 8, the portable cluster size, and at most one per k-block),
  // provided the clusters keep at least 90 % of the SMs busy and all fit at
  // once.  The weight stream is spread over every SM either way: with fewer
  // CTAs streaming (40 tiles x 3 = 120 of 152 SMs for the H5120 down_proj)
  // the cluster split measured slower than the global one, whose reduction
  // costs two global round trips after the last MMA.
  for (int cl = std::min(std::min(8, sms / std::max(pl.tiles, 1)), pl.kb_total);
       cl >= 2 && (int64_t)pl.tiles * cl * 10 >= (int64_t)sms * 9; --cl) {
    if (max_clusters(pl.nt, cl) >= pl.tiles) {
      pl.cl = cl;
      pl.grid = pl.tiles * cl;
      pl.maxfrag = 1;
      pl.ws_bytes = 0;
      pl.split = false;
      return pl;
    }
  }
  pl.cl = 1;
  const int64_t w = (int64_t)pl.tiles * pl.kb_total;
  pl.grid = (int)(w < sms ? w : sms);
  // every CTA gets `whole` whole tiles; the remaining tiles are cut into one
  // contiguous run of (tile, k-block) pairs per CTA
  pl.whole = pl.tiles / pl.grid;
  pl.split_tiles = pl.tiles - pl.whole * pl.grid;
  // a shared tile counts every CTA between its first and last owner as a
  // contributor: each CTA must own at least one shared k-block
  if (pl.whole > 0 && pl.split_tiles > 0 && (int64_t)pl.split_tiles * pl.kb_total < pl.grid) {
    --pl.whole;
    pl.split_tiles += pl.grid;
  }
  const int64_t ws = (int64_t)pl.split_tiles * pl.kb_total;
  const int64_t per = (ws + pl.grid - 1) / pl.grid;          // split k-blocks per CTA, rounded up
  pl.maxfrag = (int)((per + pl.kb_total - 1) / pl.kb_total + 1);
  const bool shared_tiles = (ws % pl.grid != 0) || ((ws / pl.grid) % pl.kb_total != 0);
  // counters: one per shared tile (tiles [0, split_tiles), fewer than twice the grid)
  pl.ws_bytes = shared_tiles ? kCounterArea + (size_t)pl.grid * pl.maxfrag * pl.nt * 128 * 4 : 0;
  pl.split = true;
  return pl;
}

// The activation quantize folded into the launch (bf16 x in, the quantized
// activation buffers written by the kernel itself).
struct Fold {
  const uint16_t *x;
  const float *gs_x;
};

template <int MODE, int NT>
cudaError_t launch_nt(const Plan &pl, const uint8_t *x, const uint8_t *x_sf, const uint8_t *w,
                      const uint8_t *w_sf, const float *alpha, const float *out_gs, uint16_t *d,
                      uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n, int64_t k, void *ws,
                      uint32_t wait_limit, cudaStream_t st, const float *rs, const Fold *fold) {
  using C = Cfg<NT>;
  // the shared-memory limit is a setting of each device's context
  static PerDeviceOnce smem_attr;
  if (cudaError_t e = smem_attr.run([] {
        if constexpr (MODE == TC_W4A4_SWIGLU)
          if (cudaError_t e2 = cudaFuncSetAttribute(swapab_kernel<MODE, NT, true>,
                                                    cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES))
            return e2;
        return cudaFuncSetAttribute(swapab_kernel<MODE, NT>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM_BYTES);
      }))
    return e;
  auto kernel = swapab_kernel<MODE, NT>;
  if constexpr (MODE == TC_W4A4_SWIGLU)
    if (fold) kernel = swapab_kernel<MODE, NT, true>;
  CUtensorMap tm_w, tm_x;
  if (!make_byte_map(&tm_w, w, n, k / 2, 128, 128, 128) || !make_byte_map(&tm_x, x, m, k / 2, 128, NT, 128))
    return cudaErrorInvalidValue;
  SwapArgs a{};
  a.sfw = w_sf;
  a.sfx = x_sf;
  a.alpha = alpha;
  a.out_gs = out_gs;
  a.d = d;
  a.out_fp4 = out_fp4;
  a.out_sf = out_sf;
  const bool split = pl.split;
  if (split && ws != nullptr) {   // (no workspace is used when no tile is shared)
    a.counters = static_cast<int *>(ws);
    a.partials = reinterpret_cast<float *>(static_cast<uint8_t *>(ws) + kCounterArea);
  }
  a.m = (int32_t)m;
  a.n = (int32_t)n;
  a.k = (int32_t)k;
  a.tiles = pl.tiles;
  a.kb_total = pl.kb_total;
  a.maxfrag = pl.maxfrag;
  a.whole = pl.whole;
  a.split_tiles = pl.split_tiles;
  a.split_ok = split ? 1 : 0;
  a.cl = pl.cl;
  // without a workspace each CTA owns whole tiles (at most one CTA per tile)
  a.grid = pl.cl > 1 ? pl.grid : split ? pl.grid : (pl.tiles < num_sms() ? pl.tiles : num_sms());
  a.wait_limit = wait_limit;
  a.status = device_status_ptr();
  a.rs = rs;
  if (fold) {
    // the three phase-A words sit in the last 256 bytes of the counter area,
    // past every tile counter
    a.xsrc = fold->x;
    a.gs_x = fold->gs_x;
    a.xq = const_cast<uint8_t *>(x);
    a.xs = const_cast<uint8_t *>(x_sf);
    a.xsync = reinterpret_cast<uint32_t *>(static_cast<uint8_t *>(ws) + kCounterArea - 256);
    a.xchunks = (int32_t)((m * (k / 16) + XCHUNK - 1) / XCHUNK);
    a.pchunks = (int32_t)(((128 - m) * (k / 64) + PCHUNK - 1) / PCHUNK);
  }
  if (!a.status) return cudaErrorInvalidValue;
  if (pl.cl <= 1)
    return launch_pdl(kernel, dim3(a.grid), dim3(kThreads), C::SMEM_BYTES, st, tm_w, tm_x, a);
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = pl.cl;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.gridDim = dim3(a.grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = C::SMEM_BYTES;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, tm_w, tm_x, a);
}

template <int MODE>
cudaError_t launch_mode(const Plan &pl, const uint8_t *x, const uint8_t *x_sf, const uint8_t *w,
                        const uint8_t *w_sf, const float *alpha, const float *out_gs, uint16_t *d,
                        uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n, int64_t k, void *ws,
                        uint32_t wait_limit, cudaStream_t st, const float *rs, const Fold *fold = nullptr) {
  switch (pl.nt) {
    case 16:
      return launch_nt<MODE, 16>(pl, x, x_sf, w, w_sf, alpha, out_gs, d, out_fp4, out_sf, m, n, k, ws,
                                 wait_limit, st, rs, fold);
    case 32:
      return launch_nt<MODE, 32>(pl, x, x_sf, w, w_sf, alpha, out_gs, d, out_fp4, out_sf, m, n, k, ws,
                                 wait_limit, st, rs, fold);
    default:
      return launch_nt<MODE, 64>(pl, x, x_sf, w, w_sf, alpha, out_gs, d, out_fp4, out_sf, m, n, k, ws,
                                 wait_limit, st, rs, fold);
  }
}

}  // namespace

bool swapab_supported(TcMode mode, int64_t m, int64_t n, int64_t k) {
  if (mode == TC_W4A16) return false;
  if (m <= 0 || m > 64 || k % 64 != 0 || n % 32 != 0) return false;
  if (mode == TC_W4A4_SWIGLU && n % 128 != 0) return false;
  return n < (1 << 30) && k < (1 << 30);
}

size_t swapab_workspace_bytes(TcMode mode, int64_t m, int64_t n, int64_t k) {
  if (!swapab_supported(mode, m, n, k)) return 0;
  return make_plan(m, n, k).ws_bytes;
}

size_t swapab_fold_workspace_bytes(int64_t m, int64_t n, int64_t k) {
  if (!swapab_supported(TC_W4A4_SWIGLU, m, n, k)) return 0;
  return std::max(make_plan(m, n, k).ws_bytes, kCounterArea);
}

cudaError_t launch_swapab_quantize_fold(const uint16_t *x, const float *gs_x, uint8_t *x_fp4, uint8_t *x_sf,
                                        const uint8_t *w_int, const uint8_t *w_int_sf, const float *alpha,
                                        const float *out_gs, uint8_t *out_fp4, uint8_t *out_sf, int64_t m,
                                        int64_t n, int64_t k, void *workspace, size_t ws_bytes,
                                        uint32_t wait_limit, cudaStream_t st) {
  if (!swapab_supported(TC_W4A4_SWIGLU, m, n, k) || workspace == nullptr ||
      ws_bytes < swapab_fold_workspace_bytes(m, n, k))
    return cudaErrorNotSupported;
  const Plan pl = make_plan(m, n, k);
  const Fold fold{x, gs_x};
  return launch_mode<TC_W4A4_SWIGLU>(pl, x_fp4, x_sf, w_int, w_int_sf, alpha, out_gs, nullptr, out_fp4, out_sf,
                                     m, n, k, workspace, wait_limit, st, nullptr, &fold);
}

cudaError_t launch_swapab(TcMode mode, const void *a, const uint8_t *a_sf, const uint8_t *b,
                          const uint8_t *b_sf, const float *alpha, const float *out_gs, uint16_t *d,
                          uint8_t *out_fp4, uint8_t *out_sf, int64_t m, int64_t n, int64_t k,
                          void *workspace, size_t ws_bytes, uint32_t wait_limit, cudaStream_t st,
                          const float *a_row_scale) {
  if (!swapab_supported(mode, m, n, k)) return cudaErrorNotSupported;
  Plan pl = make_plan(m, n, k);
  if (pl.ws_bytes > 0 && (workspace == nullptr || ws_bytes < pl.ws_bytes)) {
    // not enough scratch to share tiles between CTAs: whole tiles per CTA
    pl.split = false;
    pl.ws_bytes = 0;
    workspace = nullptr;
  }
  const uint8_t *x = static_cast<const uint8_t *>(a);
  if (mode == TC_W4A4)
    return launch_mode<TC_W4A4>(pl, x, a_sf, b, b_sf, alpha, out_gs, d, out_fp4, out_sf, m, n, k, workspace,
                                wait_limit, st, a_row_scale);
  return launch_mode<TC_W4A4_SWIGLU>(pl, x, a_sf, b, b_sf, alpha, out_gs, d, out_fp4, out_sf, m, n, k,
                                     workspace, wait_limit, st, a_row_scale);
}

}  // namespace nvfp4
