// specv_alpha.cu -- exact acceptance probabilities of the drafted positions.
//
// For drafted position i of sequence b, a draft token x ~ q is accepted with
// probability min(1, p~(x)/q(x)), so the position's acceptance probability is
//   alpha_i = sum_x q(x) min(1, p~(x)/q(x)) = sum_v min(p~_v, q_v),
// the overlap of the two distributions (1 minus their total-variation
// distance).  The speculative-decoding explainer's speed-up analysis builds its
// expected-token count on this per-position rate; a host policy uses it to
// choose the draft length K (specv_choose_k).
//
// One thread-block cluster of S CTAs per drafted position; CTA `rank` owns the
// rank-th slice of the target and draft row.  Pass 1 streams the slice and
// keeps (max, sum-exp) of the p~ source row (target row, or the mixed row in
// logit mode) and of the draft row -- the same online statistics as the verify
// kernels; every rank then reads all S partials over DSMEM and merges them in
// rank order, so every rank holds the same row statistics.  Pass 2 reads the
// slice again and sums min(p~_v, q_v); the S slice sums are added in rank
// order.  Slices are small enough (the planner's cluster size) that the second
// pass mostly finds the slice still in L2.
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
constexpr int kUnroll = 4;

struct __align__(16) AlphaShared {
  BlockScratch<kNT> bs;
  float part[4];   // this rank's (mA, sA, mB, sB)
  float sum;       // this rank's sum of min(p~, q)
};

// p~_v and q_v of one entry from the row statistics.
template <int MODE>
__device__ __forceinline__ float overlap_term(float zt, float zq, float lam, const SampleParams &sp) {
  const float a = MODE == kLogitMix ? mix_logit(zt, zq, lam) : zt;
  const float pa = prob_from_offset(a, sp.nA);
  const float pq = prob_from_offset(zq, sp.nB);
  const float pt = MODE == kProbMix ? __fmaf_rn(lam, pq, __fmul_rn(__fsub_rn(1.0f, lam), pa)) : pa;
  return fminf(pt, pq);
}

template <typename T, int MODE, bool ALIGNED>
__global__ void __launch_bounds__(kNT, 4) alpha_kernel(AlphaArgs a) {
  constexpr int VW = Elem<T>::kPerVec;
  __shared__ AlphaShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int S = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t q = (int64_t)blockIdx.x / S;  // drafted position b*K + i
  const int K = a.K, V = a.V;
  const int64_t b = q / K;
  const int i = (int)(q - b * K);
  const T *rowA = static_cast<const T *>(a.target) + (b * (K + 1) + i) * (int64_t)V;
  const T *rowB = static_cast<const T *>(a.draft) + q * (int64_t)V;
  const int g_lo = rank * a.groups_per_slice;
  const int g_hi = min(a.num_groups, g_lo + a.groups_per_slice);
  const float lam = a.lam[b];

  // ------------------------------------------------ pass 1: row statistics
  float mA = -INFINITY, sA = 0.0f, mB = -INFINITY, sB = 0.0f;
  slice_stats<T, MODE, ALIGNED, kNT, kUnroll>(rowA, rowB, true, lam, V, g_lo, g_hi, mA, sA, mB, sB);
  block_merge_stats<kNT>(sh.bs, mA, sA, mB, sB);
  if (threadIdx.x == 0) {
    sh.part[0] = mA;
    sh.part[1] = sA;
    sh.part[2] = mB;
    sh.part[3] = sB;
  }
  cluster.sync();  // every rank's partials are visible
  float m0, s0, m1, s1;
  merge_stats2_n(  // every thread merges the same partials in rank order
      S,
      [&](int r) {
        const float *pr = cluster.map_shared_rank(sh.part, r);
        return make_float4(pr[0], pr[1], pr[2], pr[3]);
      },
      m0, s0, m1, s1);
  const SampleParams sp = make_sample_params(m0, s0, m1, s1, lam);

  // ------------------------------------------------ pass 2: sum of min(p~, q)
  float acc = 0.0f;
  for (int g0 = g_lo + (int)threadIdx.x; g0 < g_hi; g0 += kNT * kUnroll) {
    uint4 za[kUnroll], zb[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int g = g0 + u * kNT;
      if (g < g_hi) {
        za[u] = load_group<T, ALIGNED>(rowA, g, V);
        zb[u] = load_group<T, ALIGNED>(rowB, g, V);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int g = g0 + u * kNT;
      if (g < g_hi) {
#pragma unroll
        for (int e = 0; e < VW; ++e)
          if (ALIGNED || (int64_t)g * VW + e < V)
            acc = __fadd_rn(acc, overlap_term<MODE>(Elem<T>::get(za[u], e), Elem<T>::get(zb[u], e),
                                                    lam, sp));
      }
    }
  }
  const float slice_sum = block_sum<kNT>(sh.bs, acc);
  if (threadIdx.x == 0) sh.sum = slice_sum;
  cluster.sync();  // slice sums visible; every rank is done reading the partials
  if (rank == 0 && threadIdx.x == 0) {
    float total = 0.0f;
    for (int r = 0; r < S; ++r) total = __fadd_rn(total, *cluster.map_shared_rank(&sh.sum, r));
    a.out_alpha[q] = lambda_valid(lam) ? total : NAN;
  }
  cluster.sync();  // rank 0 is done reading the other ranks' sums before they exit
}

template <typename T, int MODE, bool ALIGNED>
cudaError_t launch_one(const AlphaArgs &a, int S, int64_t grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kNT, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, alpha_kernel<T, MODE, ALIGNED>, a);
}

template <typename T, int MODE, bool ALIGNED>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(alpha_kernel<T, MODE, ALIGNED>,
                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

}  // namespace

cudaError_t alpha_prepare() {
  cudaError_t e = cudaSuccess, r;
#define SPECV_PREP(T, M, A) \
  if ((r = prepare_one<T, M, A>()) != cudaSuccess) e = r;
  SPECV_PREP(float, kProbMix, true)
  SPECV_PREP(float, kProbMix, false)
  SPECV_PREP(float, kLogitMix, true)
  SPECV_PREP(float, kLogitMix, false)
  SPECV_PREP(uint16_t, kProbMix, true)
  SPECV_PREP(uint16_t, kProbMix, false)
  SPECV_PREP(uint16_t, kLogitMix, true)
  SPECV_PREP(uint16_t, kLogitMix, false)
#undef SPECV_PREP
  return e;
}

cudaError_t alpha_launch(const AlphaArgs &a, int dtype_bf16, int mode, bool aligned, int S,
                         int64_t grid, cudaStream_t stream) {
  if (dtype_bf16) {
    if (mode == kProbMix)
      return aligned ? launch_one<uint16_t, kProbMix, true>(a, S, grid, stream)
                     : launch_one<uint16_t, kProbMix, false>(a, S, grid, stream);
    return aligned ? launch_one<uint16_t, kLogitMix, true>(a, S, grid, stream)
                   : launch_one<uint16_t, kLogitMix, false>(a, S, grid, stream);
  }
  if (mode == kProbMix)
    return aligned ? launch_one<float, kProbMix, true>(a, S, grid, stream)
                   : launch_one<float, kProbMix, false>(a, S, grid, stream);
  return aligned ? launch_one<float, kLogitMix, true>(a, S, grid, stream)
                 : launch_one<float, kLogitMix, false>(a, S, grid, stream);
}

}  // namespace specv
