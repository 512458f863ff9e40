// specv_block.cuh -- CTA-level building blocks of the row kernels: fixed-order
// block reductions and scans, TMA bulk copies and bounded mbarrier waits.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "specv_device.cuh"

namespace specv {

// Shared scratch of the block helpers for a CTA of NT threads.
template <int NT>
struct BlockScratch {
  static constexpr int kNW = NT / 32;
  float red[kNW][4];
  float incl[NT];
  int lastpos[kNW];
  int found;
};

// Sum of one float per thread in a fixed order (warp butterflies, then the
// warps in index order); every thread returns the same total.
template <int NT>
__device__ __forceinline__ float block_sum(BlockScratch<NT> &bs, float x) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) x = __fadd_rn(x, __shfl_xor_sync(0xffffffffu, x, off));
  if (lane == 0) bs.red[warp][0] = x;
  __syncthreads();
  float t = 0.0f;
#pragma unroll
  for (int w = 0; w < BlockScratch<NT>::kNW; ++w) t = __fadd_rn(t, bs.red[w][0]);
  __syncthreads();
  return t;
}

// Merge of per-thread (m, s) statistics of the A and B rows in a fixed order;
// every thread returns the CTA's statistics.
template <int NT>
__device__ __forceinline__ void block_merge_stats(BlockScratch<NT> &bs, float &mA, float &sA,
                                                  float &mB, float &sB) {
  warp_merge_stats(mA, sA);
  warp_merge_stats(mB, sB);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) {
    bs.red[warp][0] = mA;
    bs.red[warp][1] = sA;
    bs.red[warp][2] = mB;
    bs.red[warp][3] = sB;
  }
  __syncthreads();
  float m0, s0, m1, s1;
  merge_stats2_n(
      BlockScratch<NT>::kNW,
      [&](int w) { return make_float4(bs.red[w][0], bs.red[w][1], bs.red[w][2], bs.red[w][3]); },
      m0, s0, m1, s1);
  __syncthreads();
  mA = m0;
  sA = s0;
  mB = m1;
  sB = s1;
}

// Inclusive block scan of one float per thread; returns the exclusive value
// (exactly the previous thread's inclusive value) and the block total.
template <int NT>
__device__ __forceinline__ void block_scan(BlockScratch<NT> &bs, float x, float &excl, float &incl,
                                           float &total) {
  constexpr int kNW = BlockScratch<NT>::kNW;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float v = x;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    float y = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v = __fadd_rn(v, y);
  }
  if (lane == 31) bs.red[warp][0] = v;
  __syncthreads();
  if (warp == 0) {
    float ws = lane < kNW ? bs.red[lane][0] : 0.0f;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      float y = __shfl_up_sync(0xffffffffu, ws, off);
      if (lane >= off) ws = __fadd_rn(ws, y);
    }
    if (lane < kNW) bs.red[lane][2] = ws;  // inclusive warp offsets
  }
  __syncthreads();
  const float woff = warp == 0 ? 0.0f : bs.red[warp - 1][2];
  incl = warp == 0 ? v : __fadd_rn(woff, v);
  bs.incl[threadIdx.x] = incl;
  __syncthreads();
  excl = threadIdx.x == 0 ? 0.0f : bs.incl[threadIdx.x - 1];
  total = bs.incl[NT - 1];
}

// Largest per-thread index over the CTA (-1 if none); every thread gets it.
template <int NT>
__device__ __forceinline__ int block_max_index(BlockScratch<NT> &bs, int idx) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) idx = max(idx, __shfl_xor_sync(0xffffffffu, idx, off));
  if (lane == 0) bs.lastpos[warp] = idx;
  __syncthreads();
  int r = -1;
#pragma unroll
  for (int k = 0; k < BlockScratch<NT>::kNW; ++k) r = max(r, bs.lastpos[k]);
  __syncthreads();
  return r;
}

// ------------------------------------------------------------------ TMA / mbarrier
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

// Makes mbarrier initialisation visible to the cluster and to the async
// (TMA) proxy that completes the transactions on it.
__device__ __forceinline__ void mbar_fence_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completing on `bar`.
// Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void tma_load_1d(void *dst, const void *src, uint32_t bytes,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait for phase `parity` of `bar` for at most kWaitLimitNs of wall time (an
// iteration cap backs the clock up); false on timeout.  A copy of a few KiB
// lands in microseconds, so the limit is only reached if the copy is lost.
constexpr uint64_t kWaitLimitNs = 200ull * 1000 * 1000;
constexpr uint32_t kSpinLimit = 1u << 22;
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t it = 0; it < kSpinLimit; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > kWaitLimitNs) break;
  }
  return false;
}

}  // namespace specv
