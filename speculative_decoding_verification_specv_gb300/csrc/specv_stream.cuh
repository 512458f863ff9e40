// specv_stream.cuh -- the streaming row-statistics loop shared by the cluster
// row kernels (verify, tree verify, acceptance probabilities).
//
// A CTA of NT threads streams groups [g_lo, g_hi) of an A row (the p~ source:
// the target row, or the mixed row z_t + lambda (z_q - z_t) in logit mode when
// a draft row is present) and, if `pair`, of the B row (the draft row), with
// U 16-byte loads per thread and row in flight.  Each thread keeps running
// (max, sum-exp) statistics with a per-batch max: one exp per element,
// 2^(z log2e - m log2e) as one fused multiply-add and the SFU's 2^x, with
// m log2e rounded once per batch (which scales the batch's terms by a common
// factor within half an ulp of m log2e of 1: a relative error below 1e-6 of
// the sum for |m| < 64, the order of the fp32 accumulation itself), and a
// rescale only when the max grows.  The A and B rows go through the same
// instruction sequence, so identical rows give bitwise identical statistics.
#pragma once

#include <climits>
#include <cstdint>
#include <cuda_runtime.h>

#include "specv_device.cuh"
#include "specv_segments.cuh"

namespace specv {

// Elementwise maximum of two pairs of bf16 values (exact: the result is one of
// the inputs).
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// Maximum of the elements of groups z[0..U) with ok[u] set (-inf if none).
// bf16 rows reduce packed pairs first (one max per two elements), then widen
// the two halves of the surviving pair; fp32 rows take one max per element.
template <typename T, int U>
__device__ __forceinline__ float batch_max(const uint4 (&z)[U], const bool (&ok)[U]) {
  if constexpr (sizeof(T) == 2) {
    uint32_t m = 0xff80ff80u;  // (-inf, -inf)
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (ok[u]) m = bf16x2_max(bf16x2_max(m, z[u].x), bf16x2_max(z[u].y, bf16x2_max(z[u].z, z[u].w)));
    return fmaxf(__uint_as_float(m & 0xffff0000u), __uint_as_float(m << 16));
  } else {
    float m = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (ok[u]) m = fmaxf(fmaxf(__uint_as_float(z[u].x), __uint_as_float(z[u].y)),
                           fmaxf(fmaxf(__uint_as_float(z[u].z), __uint_as_float(z[u].w)), m));
    return m;
  }
}

// Folds one batch of U groups per row (groups with ok[u] unset are skipped)
// into the running statistics (mA, sA) of the A row and, if `pair`, (mB, sB)
// of the B row.
template <typename T, int MODE, int U>
__device__ __forceinline__ void fold_batch(const uint4 (&za)[U], const uint4 (&zb)[U],
                                           const bool (&ok)[U], bool pair, float lam, float &mA,
                                           float &sA, float &mB, float &sB) {
  constexpr int VW = Elem<T>::kPerVec;
  if constexpr (MODE == kLogitMix) {
    // lambda = 0 or 1: the mixed row is the target or the draft row itself
    // (mix_logit's exact cases), folded as a plain row (an invalid lambda
    // only makes its sequence invalid, whatever is folded)
    if (pair && !(lam > 0.0f && lam < 1.0f)) {
      const uint4(&src)[U] = lam == 0.0f ? za : zb;
      fold_batch<T, kProbMix, U>(src, zb, ok, pair, lam, mA, sA, mB, sB);
      return;
    }
  }
  // A-row value of element e of group u: the target logit, or in logit mode
  // the mixed logit (entries past V stay -inf)
  auto a_val = [&](int u, int e) -> float {
    const float zt = Elem<T>::get(za[u], e);
    if (MODE == kLogitMix && pair) return mix_logit_interior(zt, Elem<T>::get(zb[u], e), lam);
    return zt;
  };
  // logit mode: the mixed logits are formed in both passes (maximum, then
  // exponentials) rather than kept: keeping a batch of fp32 ones spilled
  // registers (batched workload, logit mode: 274.0 us kept vs 260.9 us formed
  // twice)
  float bmA;
  if (MODE == kLogitMix && pair) {
    bmA = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u)
#pragma unroll
      for (int e = 0; e < VW; ++e) bmA = fmaxf(bmA, ok[u] ? a_val(u, e) : -INFINITY);
  } else {
    bmA = batch_max<T, U>(za, ok);
  }
  const float bmB = pair ? batch_max<T, U>(zb, ok) : -INFINITY;
  if (bmA > mA) {
    sA = __fmul_rn(sA, exp_shifted(mA, bmA));
    mA = bmA;
  }
  if (pair && bmB > mB) {
    sB = __fmul_rn(sB, exp_shifted(mB, bmB));
    mB = bmB;
  }
  const float nA = neg_scaled_max(mA), nB = neg_scaled_max(mB);
#pragma unroll
  for (int u = 0; u < U; ++u)
    if (ok[u]) {
#pragma unroll
      for (int e = 0; e < VW; ++e) {
        sA = __fadd_rn(sA, ex2(__fmaf_rn(a_val(u, e), kLog2e, nA)));
        if (pair) sB = __fadd_rn(sB, ex2(__fmaf_rn(Elem<T>::get(zb[u], e), kLog2e, nB)));
      }
    }
}

// Early exit while streaming: every kExitEvery batches each warp reads the
// sequence's early-exit word (every lane the same address: one transaction)
// and, when it shows a rejection before position `pos`, stops reading; a value
// is acted on kExitEvery batches after it was loaded, so the load's latency is
// never waited for.  Measured at the batched workload (B = 256, K = 8,
// V = 128256 fp32), every 1 / 2 / 4 batches: probability 255.7 / 256.8 /
// 258.0 us, greedy 80.4 / 82.7 / 86.8 us (a position that started before its
// sequence's rejection was published stops sooner).
constexpr int kExitEvery = 1;

// Returns true if the thread stopped early (its statistics are then partial:
// the position lies after the sequence's first rejection and is never used).
// With mirA / mirB set (aligned rows only), every group streamed is also
// stored there, at the same index: a device copy of the rows for a second
// read when the rows themselves sit across a slow link.
template <typename T, int MODE, bool ALIGNED, int NT, int U>
__device__ __forceinline__ bool slice_stats(const T *rowA, const T *rowB, bool pair, float lam,
                                            int V, int g_lo, int g_hi, float &mA, float &sA,
                                            float &mB, float &sB,
                                            const unsigned *exit_word = nullptr, int pos = 0,
                                            int K = 0, T *mirA = nullptr, T *mirB = nullptr) {
  unsigned seen = 0u;
  int it = 0;
  for (int g0 = g_lo + (int)threadIdx.x; g0 < g_hi; g0 += NT * U, ++it) {
    if (exit_word != nullptr && it % kExitEvery == 0) {
      if (seen != 0u && K + 1 - (int)seen < pos) return true;
      seen = __ldcg(exit_word);
    }
    uint4 za[U], zb[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int g = g0 + u * NT;
      ok[u] = g < g_hi;
      if (ok[u]) {
        za[u] = load_group<T, ALIGNED>(rowA, g, V);
        if (pair) zb[u] = load_group<T, ALIGNED>(rowB, g, V);
      }
    }
    if (ALIGNED && mirA != nullptr) {
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (ok[u]) {
          const int g = g0 + u * NT;
          constexpr int VW = Elem<T>::kPerVec;
          __stcs(reinterpret_cast<uint4 *>(mirA + (int64_t)g * VW), za[u]);
          if (pair) __stcs(reinterpret_cast<uint4 *>(mirB + (int64_t)g * VW), zb[u]);
        }
    }
    fold_batch<T, MODE, U>(za, zb, ok, pair, lam, mA, sA, mB, sB);
  }
  return false;
}

// Asynchronous 16-byte copy from global into shared memory, cached in L2
// only; copies are committed and waited on in groups.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem) {
  const unsigned dst = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// slice_stats over groups [g_lo, g_hi) of 16-byte aligned rows with the loads
// decoupled from the arithmetic: each thread keeps its next D groups of each
// row in flight as asynchronous copies into its own slots of a ring in
// shared memory (ring: [D + 1][2][NT] 16-byte slots; a slot is refilled only
// after the fold of the group it held, so no copy lands on a value still
// being read), instead of a batch of register loads that drains before the
// next is issued.  No thread reads another thread's slots: no barrier.
template <typename T, int MODE, int NT, int D>
__device__ __forceinline__ void slice_stats_staged(const T *rowA, const T *rowB, bool pair,
                                                   float lam, int g_lo, int g_hi, uint4 *ring,
                                                   float &mA, float &sA, float &mB, float &sB) {
  constexpr int VW = Elem<T>::kPerVec;
  const int tid = (int)threadIdx.x;
  int gi = g_lo + tid;  // the next group to copy
  auto issue = [&](int slot) {
    if (gi < g_hi) {
      cp_async16(&ring[(slot * 2) * NT + tid], rowA + (int64_t)gi * VW);
      if (pair) cp_async16(&ring[(slot * 2 + 1) * NT + tid], rowB + (int64_t)gi * VW);
      gi += NT;
    }
    cp_async_commit();  // an empty group past the last copy keeps the count uniform
  };
#pragma unroll
  for (int d = 0; d < D; ++d) issue(d);
  int slot = 0, fill = D;
  const bool ok[1] = {true};
  for (int g = g_lo + tid; g < g_hi; g += NT) {
    cp_async_wait<D - 1>();  // the oldest copy group (this group's) has landed
    uint4 za[1], zb[1];
    za[0] = ring[(slot * 2) * NT + tid];
    if (pair) zb[0] = ring[(slot * 2 + 1) * NT + tid];
    issue(fill);  // the slot folded in the previous step
    fold_batch<T, MODE, 1>(za, zb, ok, pair, lam, mA, sA, mB, sB);
    slot = slot == D ? 0 : slot + 1;
    fill = fill == D ? 0 : fill + 1;
  }
  cp_async_wait<0>();
}

// Asynchronous 4-byte copy from global into shared memory (no register
// holds the value while it is in flight); cp_async_wait_all waits for every
// copy this thread issued.
__device__ __forceinline__ void cp_async4(void *smem, const void *gmem) {
  const unsigned dst = (unsigned)__cvta_generic_to_shared(smem);
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// Greedy: folds one 16-byte group (elements idx0, idx0 + 1, ...) into this
// thread's candidate (best, bidx).  A thread visits its groups in increasing
// index order, so the first maximum in index order is kept by taking a group
// only when its maximum is strictly larger (or when it is the thread's first
// group), and then its first entry equal to that maximum; the per-element
// work is the score and one maximum.  Entries past V are -inf.
template <typename T>
__device__ __forceinline__ void greedy_fold_group(const uint4 &za, const uint4 &zb, bool pair,
                                                  float lam, int idx0, float &best, int &bidx) {
  constexpr int VW = Elem<T>::kPerVec;
  float w[VW];
#pragma unroll
  for (int e = 0; e < VW; ++e) {
    const float zt = Elem<T>::get(za, e);
    w[e] = pair ? greedy_score(zt, Elem<T>::get(zb, e), lam) : zt;
  }
  float gm = w[0];
#pragma unroll
  for (int e = 1; e < VW; ++e) gm = fmaxf(gm, w[e]);
  if (gm > best || (bidx == INT_MAX && gm == gm)) {
    int first = VW - 1;
#pragma unroll
    for (int e = VW - 1; e >= 0; --e)
      if (w[e] == gm) first = e;
    best = gm;
    bidx = idx0 + first;
  }
}

}  // namespace specv
