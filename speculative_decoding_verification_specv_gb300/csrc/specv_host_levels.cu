// specv_host_levels.cu -- the decision pass of the host-buffer call that
// copies only the rows the verify step reaches (specv_verify_host_early_exit).
//
// The pages' loop stops at the first rejection (RAPID explainer, "3) 候选验证
// 机制（伪代码）": break after the resample), so the rows of positions after it
// never influence the outputs.  The host-buffer call therefore copies the
// batch position by position: level i brings row pair (b, i) of every
// sequence still alive to the device, and this kernel decides position i of
// those sequences; a sequence whose position i rejects clearly is marked dead,
// and none of its later rows are copied.  The verify step then runs on the
// staged batch as usual.
//
// One cluster of S CTAs per sequence of a group (the host call interleaves
// groups of sequences so that one group's copies overlap another group's
// decision pass and read-back): the streaming statistics of
// the row pair's slices (or the greedy argmax), the partials pushed into rank
// 0's shared memory, and rank 0's decision.  A decision here must never stop
// a copy that the verify step needs, so the test is conservative:
//   - sampling: dead only when u >= min(1, ratio) (1 + kSlack) + kSlack, well
//     outside the rounding difference between this kernel's statistics and
//     the verify kernel's (both fp32, different summation orders);
//   - greedy: dead when the argmax differs from x_i (an argmax with the
//     smallest-index tie rule does not depend on the reduction order);
//   - invalid inputs (token outside [0, V), lambda outside [0, 1]) stay alive.
#include <climits>

#include <cooperative_groups.h>

#include "specv_block.cuh"
#include "specv_device.cuh"
#include "specv_internal.h"
#include "specv_segments.cuh"
#include "specv_stream.cuh"

namespace cg = cooperative_groups;

namespace specv {

namespace {

constexpr int kNT = kRowThreads;
constexpr int kNW = kNT / 32;
constexpr int kUnroll = 4;
constexpr float kSlack = 1e-4f;

struct __align__(16) LevelShared {
  BlockScratch<kNT> bs;
  float4 part[kMaxCluster];  // every rank's partial, pushed into rank 0's copy
};

template <typename T, int MODE, bool ALIGNED>
__global__ void __launch_bounds__(kNT, 4) level_kernel(LevelArgs a) {
  constexpr int VW = Elem<T>::kPerVec;
  __shared__ LevelShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int S = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t j = (int64_t)blockIdx.x / S;  // the sequence's index in its group
  const int64_t b = a.group + (int64_t)a.n_groups * j;
  // every rank of the cluster reads the same flag, so the whole cluster returns together
  if (a.alive[j] == 0) return;
  const int K = a.K, V = a.V, i = a.level;
  const T *rowA = static_cast<const T *>(a.target) + (b * (K + 1) + i) * (int64_t)V;
  const T *rowB = static_cast<const T *>(a.draft) + (b * K + i) * (int64_t)V;
  const int g_lo = rank * a.groups_per_slice;
  const int g_hi = min(a.num_groups, g_lo + a.groups_per_slice);
  const float lam = a.lam[b];

  // the decision's inputs, loaded while the slices stream
  int x = -1;
  float u = 0.0f, zt_x = 0.0f, zq_x = 0.0f;
  if (rank == 0 && threadIdx.x == 0) {
    x = a.tokens[b * K + i];
    u = a.u_accept[b * K + i];
    if (x >= 0 && x < V) {
      zt_x = Elem<T>::load(rowA + x);
      zq_x = Elem<T>::load(rowB + x);
    }
  }

  float4 mine;
  if constexpr (MODE == kGreedy) {
    float best = -INFINITY;
    int bidx = INT_MAX;
    for (int g0 = g_lo + (int)threadIdx.x; g0 < g_hi; g0 += kNT * kUnroll) {
      uint4 za[kUnroll], zb[kUnroll];
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const int g = g0 + k * kNT;
        if (g < g_hi) {
          za[k] = load_group<T, ALIGNED>(rowA, g, V);
          zb[k] = load_group<T, ALIGNED>(rowB, g, V);
        }
      }
#pragma unroll
      for (int k = 0; k < kUnroll; ++k) {
        const int g = g0 + k * kNT;
        if (g < g_hi) greedy_fold_group<T>(za[k], zb[k], true, lam, g * VW, best, bidx);
      }
    }
    warp_argmax(best, bidx);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) {
      sh.bs.red[warp][0] = best;
      sh.bs.red[warp][1] = __int_as_float(bidx);
    }
    __syncthreads();
    float m = -INFINITY;
    int ix = INT_MAX;
    for (int w = 0; w < kNW; ++w) argmax_merge(m, ix, sh.bs.red[w][0], __float_as_int(sh.bs.red[w][1]));
    mine = make_float4(m, __int_as_float(ix), 0.0f, 0.0f);
  } else {
    float mA = -INFINITY, sA = 0.0f, mB = -INFINITY, sB = 0.0f;
    slice_stats<T, MODE, ALIGNED, kNT, kUnroll>(rowA, rowB, true, lam, V, g_lo, g_hi, mA, sA, mB,
                                                sB);
    block_merge_stats<kNT>(sh.bs, mA, sA, mB, sB);
    mine = make_float4(mA, sA, mB, sB);
  }
  if (threadIdx.x == 0) cluster.map_shared_rank(sh.part, 0)[rank] = mine;
  cluster.sync();  // every partial is in rank 0's shared memory
  if (rank != 0 || threadIdx.x != 0) return;
  if (!(x >= 0 && x < V) || !lambda_valid(lam)) return;  // invalid input: keep copying
  bool dead;
  if constexpr (MODE == kGreedy) {
    float m = -INFINITY;
    int ix = INT_MAX;
    for (int r = 0; r < S; ++r) argmax_merge(m, ix, sh.part[r].x, __float_as_int(sh.part[r].y));
    dead = ix != x;
  } else {
    float m0, s0, m1, s1;
    merge_stats2_n(S, [&](int r) { return sh.part[r]; }, m0, s0, m1, s1);
    const PosStats st{m0, s0, m1, s1};
    float qx = 0.0f;
    const float ratio = accept_ratio(MODE, st, zt_x, zq_x, lam, nullptr, &qx);
    dead = u >= __fmaf_rn(fminf(1.0f, ratio), 1.0f + kSlack, kSlack);
  }
  if (dead) a.alive[j] = 0;
}

template <typename T, int MODE, bool ALIGNED>
cudaError_t launch_one(const LevelArgs &a, int S, int64_t grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kNT, 1, 1);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, level_kernel<T, MODE, ALIGNED>, a);
}

template <typename T, int MODE>
cudaError_t launch_aligned(const LevelArgs &a, bool aligned, int S, int64_t grid,
                           cudaStream_t stream) {
  return aligned ? launch_one<T, MODE, true>(a, S, grid, stream)
                 : launch_one<T, MODE, false>(a, S, grid, stream);
}

template <typename T, int MODE>
cudaError_t prepare_mode() {
  cudaError_t e = cudaFuncSetAttribute(level_kernel<T, MODE, true>,
                                       cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  const cudaError_t e2 = cudaFuncSetAttribute(level_kernel<T, MODE, false>,
                                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  return e != cudaSuccess ? e : e2;
}

}  // namespace

cudaError_t level_prepare() {
  cudaError_t e = cudaSuccess, r;
#define SPECV_PREP(T, M) \
  if ((r = prepare_mode<T, M>()) != cudaSuccess) e = r;
  SPECV_PREP(float, kProbMix)
  SPECV_PREP(float, kLogitMix)
  SPECV_PREP(float, kGreedy)
  SPECV_PREP(uint16_t, kProbMix)
  SPECV_PREP(uint16_t, kLogitMix)
  SPECV_PREP(uint16_t, kGreedy)
#undef SPECV_PREP
  return e;
}

cudaError_t level_launch(const LevelArgs &a, int dtype_bf16, int mode, bool aligned, int S,
                         cudaStream_t stream) {
  const int64_t grid = a.count * (int64_t)S;
  if (dtype_bf16) {
    if (mode == kGreedy) return launch_aligned<uint16_t, kGreedy>(a, aligned, S, grid, stream);
    return mode == kProbMix ? launch_aligned<uint16_t, kProbMix>(a, aligned, S, grid, stream)
                            : launch_aligned<uint16_t, kLogitMix>(a, aligned, S, grid, stream);
  }
  if (mode == kGreedy) return launch_aligned<float, kGreedy>(a, aligned, S, grid, stream);
  return mode == kProbMix ? launch_aligned<float, kProbMix>(a, aligned, S, grid, stream)
                          : launch_aligned<float, kLogitMix>(a, aligned, S, grid, stream);
}

}  // namespace specv
