// specv_sampler.cuh -- the inverse-CDF sampler over a row slice, shared by
// the cluster row kernels: sampler weights summed per warp chunk, and an
// index-order search routed to one warp by those sums.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "specv_block.cuh"
#include "specv_device.cuh"

namespace specv {

// The slice is staged in shared memory (bA, bB: its groups of the target and
// draft rows).  Sampler weights of the slice, by warp chunks: warp w owns the contiguous
// groups [w*Cw, (w+1)*Cw) and its lanes stride through them.  Each warp's
// mass goes to wmass[w] (fixed-order butterfly); the CTA mass is their sum in
// warp order, so the search below routes by exactly these numbers.
template <typename T, int MODE, int NT, typename SH>
__device__ float chunk_masses(SH &sh, const uint4 *bA, const uint4 *bB, int ng, int kind,
                              const SampleParams &sp) {
  constexpr int VW = Elem<T>::kPerVec;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int Cw = (ng + (NT / 32) - 1) / (NT / 32);
  const int lo = warp * Cw, hi = min(ng, lo + Cw);
  float acc = 0.0f;
  for (int g = lo + lane; g < hi; g += 32) {
    const uint4 za = bA[g];
    const uint4 zb = kind != kWBonus ? bB[g] : za;
#pragma unroll
    for (int e = 0; e < VW; ++e)
      acc = __fadd_rn(acc, sample_weight(MODE, kind, sp, Elem<T>::get(za, e), Elem<T>::get(zb, e)));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, off));
  if (lane == 0) sh.wmass[warp] = acc;
  __syncthreads();
  float m = 0.0f;
#pragma unroll
  for (int w = 0; w < (NT / 32); ++w) m = __fadd_rn(m, sh.wmass[w]);
  return m;
}

// Index-order search of the slice for the first entry whose running weight
// sum exceeds t, using the warp masses of chunk_masses: the warp whose range
// holds t walks it in tiles of 32 groups with warp scans (no CTA barriers
// inside).  Returns the slice-local element index; if round-off leaves no
// crossing, the last entry with positive weight of the routed warp's range
// (-1 if none).  Call after chunk_masses, with the same kind and parameters.
template <typename T, int MODE, int NT, typename SH>
__device__ int chunk_search(SH &sh, const uint4 *bA, const uint4 *bB, int ng, int kind,
                            const SampleParams &sp, float t) {
  constexpr int VW = Elem<T>::kPerVec;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int Cw = (ng + (NT / 32) - 1) / (NT / 32);
  // route: the first warp whose cumulative mass exceeds t, else the last with mass
  int wstar = -1, wlast = -1;
  float base = 0.0f, wbase = 0.0f, tw = t;
  for (int w = 0; w < (NT / 32); ++w) {
    const float nb = __fadd_rn(base, sh.wmass[w]);
    if (sh.wmass[w] > 0.0f) wlast = w;
    if (wstar < 0 && nb > t) {
      wstar = w;
      wbase = base;
    }
    base = nb;
  }
  if (wstar < 0) {
    wstar = wlast;
    tw = INFINITY;
  }
  if (threadIdx.x == 0) sh.found = -1;
  __syncthreads();
  if (warp == wstar) {
    const int lo = warp * Cw, hi = min(ng, lo + Cw);
    float run = wbase;
    int lastpos = -1, res = -1;
    for (int g0 = lo; g0 < hi && res < 0; g0 += 32) {
      const int g = g0 + lane;
      float w[VW];
      float gs = 0.0f;
      if (g < hi) {
        const uint4 za = bA[g];
        const uint4 zb = kind != kWBonus ? bB[g] : za;
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          w[e] = sample_weight(MODE, kind, sp, Elem<T>::get(za, e), Elem<T>::get(zb, e));
          gs = __fadd_rn(gs, w[e]);
          if (w[e] > 0.0f) lastpos = g * VW + e;
        }
      } else {
#pragma unroll
        for (int e = 0; e < VW; ++e) w[e] = 0.0f;
      }
      float incl = gs;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const float y = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl = __fadd_rn(incl, y);
      }
      float excl = __shfl_up_sync(0xffffffffu, incl, 1);
      if (lane == 0) excl = 0.0f;
      const float lo_v = __fadd_rn(run, excl), hi_v = __fadd_rn(run, incl);
      const bool own = g < hi && lo_v <= tw && tw < hi_v;  // at most one lane
      int pick = -1;
      if (own) {
        float c = lo_v;
        int lastg = -1;
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          c = __fadd_rn(c, w[e]);
          if (w[e] > 0.0f) lastg = g * VW + e;
          if (pick < 0 && c > tw) pick = g * VW + e;
        }
        if (pick < 0) pick = lastg;
      }
      const unsigned owner = __ballot_sync(0xffffffffu, own);
      const int picked = __shfl_sync(0xffffffffu, pick, owner ? __ffs(owner) - 1 : 0);
      if (owner) res = picked;
      run = __fadd_rn(run, __shfl_sync(0xffffffffu, incl, 31));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, off));
    if (lane == 0) sh.found = res >= 0 ? res : lastpos;
  }
  __syncthreads();
  return sh.found;
}

}  // namespace specv
