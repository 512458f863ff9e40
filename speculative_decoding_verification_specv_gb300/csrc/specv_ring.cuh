// specv_ring.cuh -- a ring of shared-memory stages filled by 1-D bulk copies
// (TMA), through which a CTA streams its slice of one row or of a row pair.
//
// The idea: a CTA that loads its slice into registers issues a batch of
// loads, waits for all of them, folds them, and only then issues the next
// batch; here the copies of the next kRingStages - 1 chunks are always in
// flight while the threads fold the current one.  Measured on GB300 it does
// not beat register loads (a stage is refilled only after the slowest of the
// CTA's warps is done with it, and the folds take two groups per thread per
// chunk instead of four), so the planner uses it only when asked
// (SPECV_ROWS_RING=1).
//
// Protocol (no producer warp, no CTA barrier per chunk):
//   - chunk j (kRingChunkGroups 16-byte groups of each row, the last one
//     shorter) goes to stage j % kRingStages; its copies complete on the
//     stage's mbarrier `full`, whose phase j / kRingStages every thread waits
//     for (bounded by %globaltimer);
//   - after folding a chunk, lane 0 of each warp adds 1 to the stage's
//     counter `done` (acquire-release, CTA scope); the warp that brings it to
//     a multiple of the warp count is the last reader of the stage, and it
//     issues the copies of chunk j + kRingStages into that stage.
// A copy that does not land within the wait limit makes every thread stop;
// the CTA then waits (bounded) for the copies it still has in flight and
// reports failure.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

#include "specv_block.cuh"

namespace specv {

constexpr int kRingStages = 3;
constexpr int kRingChunkGroups = 512;                          // 8 KiB of a row per stage
constexpr int kRingStageBytes = 2 * kRingChunkGroups * 16;     // A chunk, then B chunk
constexpr int kRingSmemBytes = kRingStages * kRingStageBytes;  // dynamic shared memory (48 KiB)

struct RingState {
  uint64_t full[kRingStages];  // copies of the stage's current chunk have landed
  unsigned done[kRingStages];  // warps done with the stage (modulo the warp count)
  int issued[kRingStages];     // chunks issued into the stage so far
  int fail;                    // a copy did not land in time
};

__device__ __forceinline__ unsigned atom_add_acq_rel_cta(unsigned *p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;"
               : "=r"(old)
               : "r"(smem_u32(p)), "r"(v)
               : "memory");
  return old;
}

// Issues the copies of chunk j (one thread).  The rows start on 16-byte
// boundaries, so every copy does, and every size is a multiple of 16.
template <typename T>
__device__ __forceinline__ void ring_issue(RingState &rs, unsigned char *buf, const T *rowA,
                                           const T *rowB, bool pair, int g_lo, int g_hi, int j) {
  const int s = j % kRingStages;
  const int c_lo = g_lo + j * kRingChunkGroups;
  const int cnt = min(kRingChunkGroups, g_hi - c_lo);
  const uint32_t bytes = (uint32_t)cnt * 16u;
  uint4 *dst = reinterpret_cast<uint4 *>(buf + s * kRingStageBytes);
  rs.issued[s] += 1;  // before the arrive: readers of the stage's phase see it
  mbar_arrive_expect_tx(&rs.full[s], pair ? 2u * bytes : bytes);
  tma_load_1d(dst, reinterpret_cast<const uint4 *>(rowA) + c_lo, bytes, &rs.full[s]);
  if (pair)
    tma_load_1d(dst + kRingChunkGroups, reinterpret_cast<const uint4 *>(rowB) + c_lo, bytes,
                &rs.full[s]);
}

// Streams groups [g_lo, g_hi) of rowA (and of rowB if `pair`) through the
// ring.  Every thread of the CTA calls it; for every chunk each thread calls
// fold(cA, cB, cnt, c_lo) with the stage's A and B chunks in shared memory
// (cnt groups, the first of which is group c_lo of the row).  Returns false
// on every thread if a copy did not land in time (the CTA's copies have then
// been waited for, bounded).  Ends with a CTA barrier.
template <int NT, typename T, typename Fold>
__device__ bool ring_stream(RingState &rs, unsigned char *buf, const T *rowA, const T *rowB,
                            bool pair, int g_lo, int g_hi, Fold &&fold) {
  constexpr int kNW = NT / 32;
  const int nchunks = g_hi > g_lo ? (g_hi - g_lo + kRingChunkGroups - 1) / kRingChunkGroups : 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kRingStages; ++s) {
      mbar_init(&rs.full[s], 1);
      rs.done[s] = 0;
      rs.issued[s] = 0;
    }
    rs.fail = 0;
    mbar_fence_init();
    for (int j = 0; j < nchunks && j < kRingStages; ++j)
      ring_issue(rs, buf, rowA, rowB, pair, g_lo, g_hi, j);
  }
  __syncthreads();
  for (int j = 0; j < nchunks; ++j) {
    const int s = j % kRingStages;
    if (!mbar_wait(&rs.full[s], (uint32_t)((j / kRingStages) & 1))) {
      rs.fail = 1;
      break;
    }
    const uint4 *cA = reinterpret_cast<const uint4 *>(buf + s * kRingStageBytes);
    const int c_lo = g_lo + j * kRingChunkGroups;
    fold(cA, cA + kRingChunkGroups, min(kRingChunkGroups, g_hi - c_lo), c_lo);
    __syncwarp();
    if ((threadIdx.x & 31) == 0) {
      const unsigned old = atom_add_acq_rel_cta(&rs.done[s], 1u);
      if ((old + 1u) % kNW == 0u && j + kRingStages < nchunks) {
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        ring_issue(rs, buf, rowA, rowB, pair, g_lo, g_hi, j + kRingStages);
      }
    }
  }
  __syncthreads();
  const bool failed = rs.fail != 0;
  if (failed && threadIdx.x == 0) {
    // wait for the last copy issued into every stage before the CTA may exit
    for (int s = 0; s < kRingStages; ++s)
      if (rs.issued[s] > 0) (void)mbar_wait(&rs.full[s], (uint32_t)((rs.issued[s] - 1) & 1));
  }
  __syncthreads();
  return !failed;
}

}  // namespace specv
