// specv_resident.cu -- the resident cluster row kernel: TMA-staged vocabulary
// slices that stay in shared memory, and sampling decided per position.
//
// Work decomposition as in the streaming row kernel: one thread-block cluster
// of S CTAs per position (b, i), i in [0, K]; CTA `rank` owns the rank-th
// slice of the position's row(s) (target row i and draft row i for i < K, the
// target row K alone for i = K).
//
//  1. Staging: thread 0 issues 1-D TMA bulk copies (cp.async.bulk, one
//     mbarrier per 16 KiB chunk) of the whole slice into shared memory, so
//     the CTA's entire slice is in flight at once.
//  2. Statistics: threads fold each chunk into running (max, sum-exp) as it
//     lands; the CTA partials are exchanged all-to-all over DSMEM, and every
//     CTA merges them in rank order (bitwise the same in every CTA).
//  3. Local decision: the acceptance test of position i depends only on row
//     i, so every cluster decides its own position (accept x_i iff
//     u_i < min(1, p~(x_i)/q(x_i))).  A rejecting position -- a candidate
//     for the first rejection -- and the bonus position draw their token at
//     once, by inverse CDF over the slice still in shared memory: slice
//     masses are exchanged over DSMEM and the CTA holding u * (total mass)
//     finds the token with block scans.  No row is read from HBM twice.
//  4. Publication: one record (accepted / rejected + token / bonus + token /
//     invalid) per position goes to scratch; an atomic counter per sequence
//     elects the last cluster, which takes the first rejection n over the
//     records and writes the outputs.
// Every wait is bounded; the only barriers are hardware CTA/cluster barriers
// and the mbarriers of this CTA's own copies.
#include <cooperative_groups.h>

#include "specv_block.cuh"
#include "specv_device.cuh"
#include "specv_internal.h"
#include "specv_sampler.cuh"

namespace cg = cooperative_groups;

namespace specv {

namespace {

constexpr int kNT = kRowThreads;
constexpr int kChunkGroups = kResidentChunkGroups;  // 16-byte groups per chunk (16 KiB)
constexpr int kMaxChunks = kResidentMaxChunks;

// status of a position record
enum : int { kRecAccepted = 1, kRecRejected = 0, kRecBonus = 2, kRecInvalid = -1, kRecError = -2 };

constexpr int kNW = kNT / 32;

struct __align__(16) ResShared {
  BlockScratch<kNT> bs;
  float wmass[kNW];          // sampler weight mass of each warp's chunk
  int found;
  float4 part[kMaxCluster];  // CTA partial statistics, indexed by source rank
  int perr[kMaxCluster];     // CTA copy-timeout flags, indexed by source rank
  float masses[2][kMaxCluster];
  uint64_t bar[kMaxChunks];
  int status;
  int kind;
  int last;
};

// Online (max, sum-exp) over this thread's groups of one chunk of the slice.
template <typename T, int MODE>
__device__ __forceinline__ void chunk_stats(const uint4 *cA, const uint4 *cB, int cnt, bool pair,
                                            float lam, float &mA, float &sA, float &mB, float &sB) {
  constexpr int VW = Elem<T>::kPerVec;
  constexpr int U = 4;
  for (int g0 = threadIdx.x; g0 < cnt; g0 += kNT * U) {
    uint4 za[U], zb[U];
    bool ok[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int g = g0 + u * kNT;
      ok[u] = g < cnt;
      if (ok[u]) {
        za[u] = cA[g];
        if (pair) zb[u] = cB[g];
      }
    }
    auto a_val = [&](int u, int e) -> float {
      const float zt = Elem<T>::get(za[u], e);
      if (MODE == kLogitMix && pair) return mix_logit(zt, Elem<T>::get(zb[u], e), lam);
      return zt;
    };
    float bmA = -INFINITY, bmB = -INFINITY;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (ok[u]) {
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          bmA = fmaxf(bmA, a_val(u, e));
          if (pair) bmB = fmaxf(bmB, Elem<T>::get(zb[u], e));
        }
      }
    if (bmA > mA) {
      sA = __fmul_rn(sA, exp_shifted(mA, bmA));
      mA = bmA;
    }
    if (pair && bmB > mB) {
      sB = __fmul_rn(sB, exp_shifted(mB, bmB));
      mB = bmB;
    }
    // while a running maximum is -inf every entry so far is masked: shift by 0
    // (2^(-inf) = 0) instead of by -inf (NaN)
    const float shA = mA == -INFINITY ? 0.0f : mA, shB = mB == -INFINITY ? 0.0f : mB;
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (ok[u]) {
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          sA = __fadd_rn(sA, exp_shifted(a_val(u, e), shA));
          if (pair) sB = __fadd_rn(sB, exp_shifted(Elem<T>::get(zb[u], e), shB));
        }
      }
  }
}

// The last cluster of sequence b: first rejection over the position records,
// then the outputs.  Run by one warp.  The records of the first 32 positions
// and their drafted tokens are loaded together, so that the token at n and
// the accepted prefix need no second round trip.
__device__ void finalize_sequence(const ResArgs &a, int64_t b) {
  const int K = a.K;
  const int lane = threadIdx.x & 31;
  int2 r0 = make_int2(kRecAccepted, -1);
  int x0 = -1;
  if (lane <= K) r0 = __ldcg(&a.rec[b * (K + 1) + lane]);
  if (lane < K) x0 = a.tokens[b * K + lane];
  int n = K, bad = 0;
  for (int j0 = 0; j0 <= K; j0 += 32) {
    const int j = j0 + lane;
    int st = kRecAccepted;
    if (j <= K) st = j0 == 0 ? r0.x : __ldcg(&a.rec[b * (K + 1) + j]).x;
    const unsigned rej = __ballot_sync(0xffffffffu, j < K && st == kRecRejected);
    if (rej != 0u && n == K) n = j0 + __ffs(rej) - 1;
    const bool any_err = __any_sync(0xffffffffu, st == kRecError);  // every lane votes
    const bool any_inv = __any_sync(0xffffffffu, st == kRecInvalid);
    if (any_err) bad = kRecError;
    else if (bad == 0 && any_inv) bad = kRecInvalid;
  }
  if (bad != 0) {
    for (int j = lane; j <= K; j += 32) a.out_tokens[b * (K + 1) + j] = -1;
    if (lane == 0) a.out_n[b] = bad;
    return;
  }
  const int tok_lo = __shfl_sync(0xffffffffu, r0.y, n & 31);
  const int tok_n = n < 32 ? tok_lo : __ldcg(&a.rec[b * (K + 1) + n]).y;
  for (int j = lane; j <= K; j += 32)
    a.out_tokens[b * (K + 1) + j] =
        j < n ? (j < 32 ? x0 : a.tokens[b * K + j]) : (j == n ? tok_n : -1);
  if (lane == 0) a.out_n[b] = n;
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kNT) resident_kernel(ResArgs a) {
  constexpr int VW = Elem<T>::kPerVec;
  extern __shared__ __align__(128) unsigned char dsm[];
  __shared__ ResShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int S = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t p = (int64_t)blockIdx.x / S;
  const int K = a.K;
  const int64_t b = p / (K + 1);
  const int i = (int)(p - b * (K + 1));
  const bool pair = i < K;
  const T *rowA = static_cast<const T *>(a.target) + (b * (K + 1) + i) * (int64_t)a.V;
  const T *rowB = static_cast<const T *>(a.draft) + (b * K + (pair ? i : 0)) * (int64_t)a.V;
  const int g_lo = rank * a.groups_per_slice;
  const int ng = max(0, min(a.num_groups, g_lo + a.groups_per_slice) - g_lo);
  // the slice in global memory, and its copy in shared memory
  const uint4 *gA = reinterpret_cast<const uint4 *>(rowA + (int64_t)g_lo * VW);
  const uint4 *gB = reinterpret_cast<const uint4 *>(rowB + (int64_t)g_lo * VW);
  uint4 *stA = reinterpret_cast<uint4 *>(dsm);
  uint4 *stB = stA + a.groups_per_slice;
  const uint4 *bA = stA;
  const uint4 *bB = stB;
  const int nch = (ng + kChunkGroups - 1) / kChunkGroups;
  const float lam = a.lam[b];

  // decision inputs, loaded now so their latency overlaps the statistics pass
  int x = 0;
  float u_acc = 0.0f, zt_x = 0.0f, zq_x = 0.0f;
  bool tok_ok = true;
  if (threadIdx.x == 0 && pair) {
    x = a.tokens[b * K + i];
    u_acc = a.u_accept[b * K + i];
    tok_ok = x >= 0 && x < a.V;
    if (tok_ok) {
      zt_x = Elem<T>::load(rowA + x);
      zq_x = Elem<T>::load(rowB + x);
    }
  }

  // ---------------------------------------------------------------- staging
  if (threadIdx.x == 0) {
    for (int c = 0; c < nch; ++c) mbar_init(&sh.bar[c], 1);
    mbar_fence_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int c = 0; c < nch; ++c) {
      const int g0 = c * kChunkGroups;
      const int cnt = min(kChunkGroups, ng - g0);
      const uint32_t bytes = (uint32_t)cnt * 16u;
      mbar_arrive_expect_tx(&sh.bar[c], pair ? 2u * bytes : bytes);
      tma_load_1d(stA + g0, gA + g0, bytes, &sh.bar[c]);
      if (pair) tma_load_1d(stB + g0, gB + g0, bytes, &sh.bar[c]);
    }
  }

  // ------------------------------------------------------------- statistics
  float mA = -INFINITY, sA = 0.0f, mB = -INFINITY, sB = 0.0f;
  int err = 0;
  for (int c = 0; c < nch; ++c) {
    if (!mbar_wait(&sh.bar[c], 0)) err = 1;
    const int g0 = c * kChunkGroups;
    chunk_stats<T, MODE>(bA + g0, bB + g0, min(kChunkGroups, ng - g0), pair, lam, mA, sA, mB, sB);
  }
  err = __syncthreads_or(err);
  block_merge_stats<kNT>(sh.bs, mA, sA, mB, sB);
  if (threadIdx.x == 0) {
    const float4 mine = make_float4(mA, sA, mB, sB);
    for (int r = 0; r < S; ++r) {
      cluster.map_shared_rank(sh.part, r)[rank] = mine;
      cluster.map_shared_rank(sh.perr, r)[rank] = err;
    }
  }
  cluster.sync();  // every CTA holds every partial
  float m0, s0, m1, s1;
  merge_stats2_n(S, [&](int r) { return sh.part[r]; }, m0, s0, m1, s1);
  int cerr = 0;
  for (int r = 0; r < S; ++r) cerr |= sh.perr[r];

  // --------------------------------------------------------- local decision
  if (threadIdx.x == 0) {
    int status, kind = -1;
    if (cerr) {
      status = kRecError;
    } else if (!lambda_valid(lam)) {
      status = kRecInvalid;
    } else if (!pair) {
      status = kRecBonus;
      kind = kWBonus;
    } else if (!tok_ok) {
      status = kRecInvalid;
    } else {
      float px = 0.0f, qx = 0.0f;
      const PosStats st{m0, s0, m1, s1};
      const float ratio =
          accept_ratio(MODE, st, zt_x, zq_x, lam, (rank == 0 && a.dbg_ptilde) ? &px : nullptr, &qx);
      const bool acc = accept_test(u_acc, ratio);
      if (rank == 0 && a.dbg_ptilde) {
        a.dbg_ptilde[b * K + i] = px;
        a.dbg_q[b * K + i] = qx;
      }
      status = acc ? kRecAccepted : kRecRejected;
      if (!acc) kind = !(lam < 1.0f) ? kWMixture : kWResidual;
    }
    if (rank == 0 && a.dbg_lse) {
      a.dbg_lse[p * 2 + 0] = m0 + lg2(s0) * kLn2;
      a.dbg_lse[p * 2 + 1] = pair ? m1 + lg2(s1) * kLn2 : 0.0f;
    }
    sh.status = status;
    sh.kind = kind;
    sh.last = 0;
  }
  __syncthreads();
  const int status = sh.status;
  int kind = sh.kind;

  // ------------------------------------- sampling (rejecting / bonus positions)
  int publisher = 0;  // rank that publishes the record
  int token = -1;
  if (kind >= 0) {
    const SampleParams sp = make_sample_params(m0, s0, m1, s1, lam);
    float R = 0.0f;
    int attempt = 0;
    for (;; ++attempt) {
      const float mass = chunk_masses<T, MODE, kNT>(sh, bA, bB, ng, kind, sp);
      if (threadIdx.x == 0)
        for (int r = 0; r < S; ++r) cluster.map_shared_rank(sh.masses[attempt], r)[rank] = mass;
      cluster.sync();  // all slice masses exchanged
      R = 0.0f;
      for (int r = 0; r < S; ++r) R = __fadd_rn(R, sh.masses[attempt][r]);
      if (R > 0.0f || kind != kWResidual || attempt == 1) break;
      kind = kWMixture;  // zero residual mass (round-off only): draw from p~ instead
    }
    if (R > 0.0f) {
      const float t = __fmul_rn(a.u_resample[b], R);
      int rstar = -1;
      float tloc = INFINITY, c = 0.0f;
      for (int r = 0; r < S; ++r) {
        const float cn = __fadd_rn(c, sh.masses[attempt][r]);
        if (cn > t) {
          rstar = r;
          tloc = __fsub_rn(t, c);
          break;
        }
        c = cn;
      }
      if (rstar < 0) {  // u*R not below the total (u >= 1 or round-off): last slice with mass
        for (int r = S - 1; r >= 0; --r)
          if (sh.masses[attempt][r] > 0.0f) {
            rstar = r;
            break;
          }
        tloc = INFINITY;
      }
      publisher = rstar;
      if (rank == rstar) {
        const int local = chunk_search<T, MODE, kNT>(sh, bA, bB, ng, kind, sp, tloc);
        token = local >= 0 ? g_lo * VW + local : -1;
      }
    }
  }
  if (rank != publisher) return;

  // -------------------------------------------------------------- publish
  if (threadIdx.x == 0) {
    a.rec[p] = make_int2(status, token);
    // one acquire-release atomic: the record before the count, and for the
    // last arrival every other position's record after it
    unsigned prev;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
                 : "=r"(prev) : "l"(&a.count[b]) : "memory");
    if (prev == (unsigned)K) {
      a.count[b] = 0;  // every position has arrived: leave the counter zero for the next call
      sh.last = 1;
    }
  }
  __syncthreads();
  if (sh.last && threadIdx.x < 32) finalize_sequence(a, b);
}

template <typename T, int MODE>
cudaError_t launch_one(const ResArgs &a, int S, int64_t grid, int smem, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kNT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, resident_kernel<T, MODE>, a);
}

template <typename T, int MODE>
cudaError_t prepare_one(int max_smem) {
  cudaError_t e = cudaFuncSetAttribute(resident_kernel<T, MODE>,
                                       cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(resident_kernel<T, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              max_smem);
}

}  // namespace

cudaError_t resident_prepare(int max_smem) {
  cudaError_t e = cudaSuccess, r;
#define SPECV_PREP(T, M) \
  if ((r = prepare_one<T, M>(max_smem)) != cudaSuccess) e = r;
  SPECV_PREP(float, kProbMix)
  SPECV_PREP(float, kLogitMix)
  SPECV_PREP(uint16_t, kProbMix)
  SPECV_PREP(uint16_t, kLogitMix)
#undef SPECV_PREP
  return e;
}

cudaError_t resident_launch(const ResArgs &a, int dtype_bf16, int mode, int S, int64_t grid,
                            int smem, cudaStream_t stream) {
  if (dtype_bf16)
    return mode == kProbMix ? launch_one<uint16_t, kProbMix>(a, S, grid, smem, stream)
                            : launch_one<uint16_t, kLogitMix>(a, S, grid, smem, stream);
  return mode == kProbMix ? launch_one<float, kProbMix>(a, S, grid, smem, stream)
                          : launch_one<float, kLogitMix>(a, S, grid, smem, stream);
}

}  // namespace specv
