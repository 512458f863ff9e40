// specv_segments.cuh -- inverse-CDF search over segments of a row, shared by
// the row kernels.
//
// A slice of a row (a run of 16-byte groups) is cut into segments of
// consecutive groups.  segment_masses sums the sampler weights of every
// segment (one warp per segment) and forms the running sums in index order;
// find_segment routes a target t to the segment whose running-sum interval
// holds it; segment_walk lets one warp walk that segment in index order to
// the entry at which the running sum first exceeds t.  Only the chosen segment
// is read a second time.  A tile of a segment is LG 16-byte loads per lane
// (32 * LG groups), coalesced across the warp.
//
// The shared-memory struct SH provides `bs` (BlockScratch<NT>) and the arrays
// `segm` and `segi` (one float per segment).
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "specv_block.cuh"
#include "specv_device.cuh"

namespace specv {

// Load group g (VW consecutive elements) of a row as one 16-byte vector.  In
// the aligned case every row starts on a 16-byte boundary and V is a multiple
// of VW, so a group is one 16-byte load (streaming: no L1 allocation; cached:
// through L1, for the segment walk).  Otherwise the vector is assembled from
// scalar loads and entries past V read as -inf (they add nothing to a max or
// a sum).  Elements are widened to fp32 where they are used (Elem<T>::get),
// which keeps bf16 groups at 4 registers.
template <typename T, bool ALIGNED, bool CACHED = false>
__device__ __forceinline__ uint4 load_group(const T *row, int64_t g, int V) {
  constexpr int VW = Elem<T>::kPerVec;
  if constexpr (ALIGNED) {
    if constexpr (CACHED)
      return __ldg(reinterpret_cast<const uint4 *>(row + g * VW));
    else
      return ld_stream16(row + g * VW);
  } else {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      const int64_t idx = g * VW + e;
      Elem<T>::put_bits(v, e, idx < V ? Elem<T>::load_bits(row + idx) : Elem<T>::kNegInfBits);
    }
    return v;
  }
}

// A 16-byte vector of -inf entries.
template <typename T>
__device__ __forceinline__ uint4 neg_inf_group() {
  const uint32_t w = sizeof(T) == 4 ? Elem<T>::kNegInfBits
                                    : (Elem<T>::kNegInfBits << 16) | Elem<T>::kNegInfBits;
  return make_uint4(w, w, w, w);
}

// Sampler weight of each of the nseg segments of [g_lo, g_hi) into sh.segm,
// then the inclusive running sums in index order into sh.segi; returns the
// slice's mass (equal to the last running sum).  Warp w takes segments
// w, w + NT/32, ...; an empty segment weighs 0.
template <typename T, int MODE, bool ALIGNED, int LG, int NT, typename SH>
__device__ float segment_masses(SH &sh, const T *rowA, const T *rowB, int V, int g_lo, int g_hi,
                                int seg_groups, int nseg, int kind, const SampleParams &sp) {
  constexpr int VW = Elem<T>::kPerVec;
  constexpr int kNW = NT / 32;
  constexpr int kTile = 32 * LG;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int s = warp; s < nseg; s += kNW) {
    const int sg_lo = g_lo + s * seg_groups;
    const int sg_hi = min(g_hi, sg_lo + seg_groups);
    float acc = 0.0f;
    for (int g0 = sg_lo; g0 < sg_hi; g0 += kTile) {
      uint4 za[LG], zb[LG];
#pragma unroll
      for (int u = 0; u < LG; ++u) {
        const int g = g0 + u * 32 + lane;
        if (g < sg_hi) {
          za[u] = load_group<T, ALIGNED>(rowA, g, V);
          if (kind != kWBonus) zb[u] = load_group<T, ALIGNED>(rowB, g, V);
        }
      }
#pragma unroll
      for (int u = 0; u < LG; ++u) {
        const int g = g0 + u * 32 + lane;
        if (g < sg_hi) {
#pragma unroll
          for (int e = 0; e < VW; ++e)
            if (ALIGNED || (int64_t)g * VW + e < V)
              acc = __fadd_rn(acc, sample_weight(MODE, kind, sp, Elem<T>::get(za[u], e),
                                                 kind != kWBonus ? Elem<T>::get(zb[u], e) : 0.0f));
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1)
      acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
    if (lane == 0) sh.segm[s] = acc;
  }
  __syncthreads();
  float base = 0.0f;
  for (int s0 = 0; s0 < nseg; s0 += NT) {
    const int s = s0 + (int)threadIdx.x;
    float excl, incl, total;
    block_scan<NT>(sh.bs, s < nseg ? sh.segm[s] : 0.0f, excl, incl, total);
    if (s < nseg) sh.segi[s] = __fadd_rn(base, incl);
    base = __fadd_rn(base, total);
  }
  __syncthreads();
  return base;
}

// The segment whose running-sum interval [segi[s-1], segi[s]) holds t (the
// intervals are disjoint: the running sums never decrease).  If none does (t
// at or past the slice's mass: u >= 1 or round-off), the last segment of
// positive mass, with t set to +inf so that its walk takes its last entry of
// positive weight.  *lo gets the running sum before the segment.
template <int NT, typename SH>
__device__ int find_segment(SH &sh, int nseg, float &t, float *lo) {
  if (threadIdx.x == 0) sh.bs.found = -1;
  __syncthreads();
  int lastpos = -1;
  for (int s = threadIdx.x; s < nseg; s += NT) {
    const float l = s ? sh.segi[s - 1] : 0.0f;
    if (l <= t && t < sh.segi[s]) sh.bs.found = s;
    if (sh.segm[s] > 0.0f) lastpos = s;
  }
  __syncthreads();
  int s = sh.bs.found;
  __syncthreads();
  if (s < 0) {
    s = block_max_index<NT>(sh.bs, lastpos);
    t = INFINITY;
  }
  *lo = s > 0 ? sh.segi[s - 1] : 0.0f;
  return s;
}

// One warp walks the groups [sg_lo, sg_hi) of the row(s) in index order,
// starting from running sum c, and returns the first entry at which the
// running sum of sampler weights exceeds t; if round-off leaves no crossing,
// the last entry of positive weight (-1 if none).  Index order within a tile
// is (load u, lane, element): the 32 lanes of one load are scanned together.
template <typename T, int MODE, bool ALIGNED, int LG>
__device__ int segment_walk(const T *rowA, const T *rowB, int V, int sg_lo, int sg_hi, int kind,
                            const SampleParams &sp, float c, float t) {
  constexpr int VW = Elem<T>::kPerVec;
  constexpr int kTile = 32 * LG;
  const int lane = threadIdx.x & 31;
  int lastpos = -1;
  for (int g0 = sg_lo; g0 < sg_hi; g0 += kTile) {
    uint4 za[LG], zb[LG];
#pragma unroll
    for (int u = 0; u < LG; ++u) {
      const int g = g0 + u * 32 + lane;
      za[u] = g < sg_hi ? load_group<T, ALIGNED, true>(rowA, g, V) : neg_inf_group<T>();
      zb[u] = (g < sg_hi && kind != kWBonus) ? load_group<T, ALIGNED, true>(rowB, g, V) : za[u];
    }
#pragma unroll
    for (int u = 0; u < LG; ++u) {
      const int g = g0 + u * 32 + lane;
      float w[VW];
      float s = 0.0f;
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        const int idx = g * VW + e;
        w[e] = (g < sg_hi && (ALIGNED || idx < V))
                   ? sample_weight(MODE, kind, sp, Elem<T>::get(za[u], e), Elem<T>::get(zb[u], e))
                   : 0.0f;
        s = __fadd_rn(s, w[e]);
        if (w[e] > 0.0f) lastpos = idx;
      }
      float incl = s;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl = __fadd_rn(incl, y);
      }
      const float hi = __fadd_rn(c, incl);
      const float prev = __shfl_up_sync(0xffffffffu, hi, 1);
      const float lo = lane == 0 ? c : prev;
      const unsigned cross = __ballot_sync(0xffffffffu, hi > t);
      if (cross != 0u) {  // warp-uniform
        const int L = __ffs(cross) - 1;
        int pick = -1, lastl = -1;
        float cc = lo;
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          cc = __fadd_rn(cc, w[e]);
          if (w[e] > 0.0f) lastl = g * VW + e;
          if (pick < 0 && cc > t) pick = g * VW + e;
        }
        pick = pick >= 0 ? pick : lastl;
        return __shfl_sync(0xffffffffu, pick, L);
      }
      c = __shfl_sync(0xffffffffu, hi, 31);
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1)
    lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, off));
  return lastpos;
}

}  // namespace specv
