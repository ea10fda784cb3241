// Split-K work partition shared by the weight-streaming (swap-AB) kernels:
// the (128-row weight tile, k-block) pairs laid out tile-major and cut into
// one contiguous, equal run per CTA.
#pragma once
#include <cstdint>

namespace nvfp4 {

// Contiguous partition of W = tiles * kb_total k-blocks over `grid` CTAs:
// CTA j owns [start(j), start(j+1)), start(j) = floor(j * W / grid).  Without
// a workspace the cut points are rounded to whole tiles instead.
struct Partition {
  int64_t w, grid, kbt;
  bool whole_tiles;
  int64_t tiles;
  __device__ __forceinline__ int64_t start(int64_t j) const {
    if (whole_tiles) return (j * tiles / grid) * kbt;
    return j * w / grid;
  }
  // CTA owning global k-block x (inverse of start)
  __device__ __forceinline__ int64_t cta_of(int64_t x) const {
    if (whole_tiles) {
      const int64_t t = x / kbt;
      return ((t + 1) * grid - 1) / tiles;
    }
    return ((x + 1) * grid - 1) / w;
  }
};

// Iterates the fragments of one CTA: tile, [kb0, kb1) within the tile.
struct FragIter {
  int64_t x, end, kbt;
  __device__ __forceinline__ bool next(int &tile, int &kb0, int &kb1) {
    if (x >= end) return false;
    tile = (int)(x / kbt);
    kb0 = (int)(x - (int64_t)tile * kbt);
    const int64_t room = end - x;
    kb1 = (int)min((int64_t)kbt, kb0 + room);
    x += kb1 - kb0;
    return true;
  }
};

// Mixed split for one weight-streaming GEMM with at least as many tiles as
// CTAs: every CTA gets `whole` whole tiles (done last; no reduction with
// other CTAs), and the remaining split_tiles tiles are cut into a contiguous
// run of (tile, k-block) pairs per CTA (done first, so the tiles they share
// are complete while the whole tiles stream).  With fewer tiles than CTAs,
// whole = 0 and every tile is split.  Split tiles are [0, split_tiles); CTA
// j's whole tiles are split_tiles + j*whole + [0, whole).
struct MixedPartition {
  int64_t kbt, grid, whole, split_tiles;
  __device__ __forceinline__ int64_t split_units() const { return split_tiles * kbt; }
  __device__ __forceinline__ int64_t start(int64_t j) const { return j * split_units() / grid; }
  // CTA owning split unit x (inverse of start); only for x < split_units()
  __device__ __forceinline__ int64_t cta_of(int64_t x) const { return ((x + 1) * grid - 1) / split_units(); }
  __device__ __forceinline__ bool is_split(int tile) const { return tile < split_tiles; }
};

// The fragments of CTA j under a MixedPartition: its split run, then its
// whole tiles.
struct MixedIter {
  int64_t x, end, kbt;
  int t, t_end;
  __device__ __forceinline__ MixedIter(const MixedPartition &mp, int64_t j)
      : x(mp.start(j)), end(mp.start(j + 1)), kbt(mp.kbt), t((int)(mp.split_tiles + j * mp.whole)),
        t_end((int)(mp.split_tiles + (j + 1) * mp.whole)) {}
  __device__ __forceinline__ bool next(int &tile, int &kb0, int &kb1) {
    if (x < end) {
      tile = (int)(x / kbt);
      kb0 = (int)(x - (int64_t)tile * kbt);
      kb1 = (int)min((int64_t)kbt, kb0 + (end - x));
      x += kb1 - kb0;
      return true;
    }
    if (t < t_end) {
      tile = t++;
      kb0 = 0;
      kb1 = (int)kbt;
      return true;
    }
    return false;
  }
};

// Arrival on a split-K tile counter: release of this CTA's partial tile
// (written by the epilogue threads before a CTA barrier) and acquire of the
// other contributors' partials, in one atomic.
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(int *p, int v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// v[t] = sum of the fp32 partial tiles of contributors c_first..c_last, in
// that order (so the result does not depend on which contributor finished
// last), for accumulator row r and tokens t < mt.  The loads of up to MAXC
// contributors are issued together, so the sum costs about one L2 round
// trip per MAXC contributors instead of one per contributor.
template <int NT, class SlotFn>
__device__ __forceinline__ void sum_partials_in_k_order(float (&v)[NT], int64_t c_first, int64_t c_last, int mt,
                                                        int r, SlotFn slot) {
  constexpr int MAXC = NT <= 16 ? 8 : NT <= 32 ? 4 : 2;
#pragma unroll
  for (int t = 0; t < NT; ++t) v[t] = 0.0f;
  for (int64_t c0 = c_first; c0 <= c_last; c0 += MAXC) {
    float pv[MAXC][NT];
#pragma unroll
    for (int i = 0; i < MAXC; ++i) {
      const bool have = c0 + i <= c_last;
      const float *pc = slot(have ? c0 + i : c0);
#pragma unroll
      for (int t = 0; t < NT; ++t) pv[i][t] = (have && t < mt) ? __ldcg(pc + t * 128 + r) : 0.0f;
    }
#pragma unroll
    for (int i = 0; i < MAXC; ++i)
      if (c0 + i <= c_last) {
#pragma unroll
        for (int t = 0; t < NT; ++t) v[t] += pv[i][t];
      }
  }
}

}  // namespace nvfp4
