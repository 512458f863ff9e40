// specv_tree.cu -- tree verification: the verify/accept step for a tree of
// drafted tokens per sequence.
//
// Reading (the speculative-decoding explainer's "Tree Speculation" section:
// several candidate branches per position, verified at once, so that another
// branch can be accepted when one is rejected; no multi-branch rule is given).
// Node 0 is the root; node j >= 1 has parent[j] < j and token x_j.  The
// children of node u were drawn independently from the draft distribution q_u
// (draft row draft_row[u]).  The walk starts at the root with p = p~_u (the
// mixture of the target row of u and q_u, or the target softmax when u has no
// draft row) and tests u's children in index order: x_c is accepted iff
// u_accept[c] < min(1, p(x_c)/q_u(x_c)); a rejection replaces p by
// normalize(max(0, p - q_u)); an acceptance moves the walk to c.  When every
// child is rejected the token is drawn from p by inverse CDF; at a node without
// children, from p~_u (the bonus).  A chain of single children is the chain
// verify step.
//
// After k rejections at u, p is max(0, p~_u - c_k q_u) / N(c_k) with
// N(c) = sum_v max(0, p~_u(v) - c q_u(v)), c_0 = 0, c_{k+1} = c_k + N(c_k) (equal
// in exact arithmetic to applying the normalised residual k times), so the
// test of the next child is u < min(1, max(0, r - c_k) / N(c_k)) with
// r = p~_u(x)/q_u(x) from the row statistics, and each rejection costs one
// cluster-wide pass over u's row pair for N(c_{k+1}).
//
// Decomposition: one thread-block cluster of S CTAs per node (the streaming
// row kernel's phase 1 computes every node's row statistics); the last cluster
// of a sequence to publish walks the tree.  Rank 0's first warp makes every
// decision and hands each pass, and the final draw, to all ranks through
// DSMEM, so the ranks never disagree on the number of cluster barriers.
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
constexpr int kUnroll = 4;

// What rank 0 asks of every rank: a pass over node u's rows with a weight
// kind (`final` = 0: the mass after a rejection; 1: the final draw), or the
// end of an invalid sequence (`final` = 2).
struct WalkCmd {
  int final;
  int kind;
  int u;
  int n;        // accepted drafts so far (index of the token the final draw writes)
  int reuse;    // final draw from the masses of the previous pass (no new pass)
  SampleParams sp;
};

struct __align__(16) TreeShared {
  BlockScratch<kNT> bs;
  float part[4];
  int last;
  WalkCmd cmd;
  float masses[2][kMaxCluster];
  float segm[kMaxSegs];
  float segi[kMaxSegs];
};

// The smallest j in (after, N] with parent[j] == u, or -1 (one warp, every
// lane gets it).
__device__ __forceinline__ int warp_first_child(const int32_t *par, int N, int u, int after) {
  const int lane = threadIdx.x & 31;
  for (int j0 = after + 1; j0 <= N; j0 += 32) {
    const int j = j0 + lane;
    const unsigned m = __ballot_sync(0xffffffffu, j <= N && __ldg(&par[j]) == u);
    if (m != 0u) return j0 + __ffs(m) - 1;
  }
  return -1;
}

// Structure and input checks of one sequence (one warp, every lane gets it).
__device__ __forceinline__ bool warp_tree_valid(const TreeArgs &a, int64_t base, float lam) {
  const int lane = threadIdx.x & 31;
  bool ok = lambda_valid(lam) && __ldg(&a.parent[base]) == -1;
  const int d0 = __ldg(&a.draft_row[base]);
  ok = ok && d0 >= -1 && d0 < a.M;
  for (int j = lane + 1; j <= a.N; j += 32) {
    const int p = __ldg(&a.parent[base + j]);
    const int d = __ldg(&a.draft_row[base + j]);
    const int x = __ldg(&a.tokens[base + j]);
    bool o = p >= 0 && p < j && d >= -1 && d < a.M && x >= 0 && x < a.V;
    if (o) o = __ldg(&a.draft_row[base + p]) >= 0;  // a node with children has a draft row
    ok = ok && o;
  }
  return __all_sync(0xffffffffu, ok);
}

// Sum of the sampler weights over node u's whole row (all S slices): segment
// masses and running sums stay in sh.segm/segi for routing, the slice masses
// in sh.masses[slot]; every thread of every rank gets the same total.
template <typename T, int MODE, bool ALIGNED>
__device__ float cluster_mass(TreeShared &sh, cg::cluster_group &cluster, int S, int rank,
                              const T *rowA, const T *rowB, int V, int g_lo, int g_hi,
                              int seg_groups, int nseg, int kind, const SampleParams &sp, int slot) {
  const float mass = segment_masses<T, MODE, ALIGNED, kSegLaneGroups, kNT>(
      sh, rowA, rowB, V, g_lo, g_hi, seg_groups, nseg, kind, sp);
  if (threadIdx.x == 0)
    for (int r = 0; r < S; ++r) cluster.map_shared_rank(sh.masses[slot], r)[rank] = mass;
  cluster.sync();  // all slice masses exchanged
  float R = 0.0f;
  for (int r = 0; r < S; ++r) R = __fadd_rn(R, sh.masses[slot][r]);
  return R;
}

template <typename T, int MODE, bool ALIGNED>
__global__ void __launch_bounds__(kNT, 4) tree_kernel(TreeArgs a) {
  __shared__ TreeShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int S = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t p = (int64_t)blockIdx.x / S;  // node index b*(N+1) + u
  const int N = a.N, V = a.V, M = a.M;
  const int64_t b = p / (N + 1);
  const int64_t base = b * (N + 1);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T *tgt = static_cast<const T *>(a.target);
  const T *dft = static_cast<const T *>(a.draft);
  const int g_lo = rank * a.groups_per_slice;
  const int g_hi = min(a.num_groups, g_lo + a.groups_per_slice);
  const float lam = a.lam[b];

  // ---------------------------------------------------------------- phase 1
  {
    const int d = __ldg(&a.draft_row[p]);
    const bool pair = d >= 0 && d < M;  // an out-of-range row is reported in phase 2
    const T *rowA = tgt + p * (int64_t)V;
    const T *rowB = dft + (b * M + (pair ? d : 0)) * (int64_t)V;
    float mA = -INFINITY, sA = 0.0f, mB = -INFINITY, sB = 0.0f;
    slice_stats<T, MODE, ALIGNED, kNT, kUnroll>(rowA, rowB, pair, lam, V, g_lo, g_hi, mA, sA, mB,
                                                sB);
    block_merge_stats<kNT>(sh.bs, mA, sA, mB, sB);
    if (threadIdx.x == 0) {
      sh.part[0] = mA;
      sh.part[1] = sA;
      sh.part[2] = mB;
      sh.part[3] = sB;
    }
  }
  cluster.sync();  // partials of every rank are visible
  if (rank == 0 && threadIdx.x == 0) {
    float m0, s0, m1, s1;
    merge_stats2_n(
        S,
        [&](int r) {
          const float *pr = cluster.map_shared_rank(sh.part, r);
          return make_float4(pr[0], pr[1], pr[2], pr[3]);
        },
        m0, s0, m1, s1);
    a.ws_stats[p] = make_float4(m0, s0, m1, s1);
    __threadfence();
    const unsigned prev = atomicAdd(&a.ws_count[b], 1u);
    const int last = prev == (unsigned)N;
    if (last) {
      __threadfence();
      a.ws_count[b] = 0;  // every node has arrived: leave the counter zero for the next call
    }
    for (int r = 0; r < S; ++r) *cluster.map_shared_rank(&sh.last, r) = last;
  }
  cluster.sync();  // sh.last is set in every rank; rank 0 is done reading partials
  if (!sh.last) return;

  // ---------------------------------------------------------------- phase 2
  // Walk state, kept identically by every lane of rank 0's first warp.
  int u = 0, n = 0, c = -1, after = 0, rejected = 0, pending_zero = 0;
  bool search = true;
  float cthr = 0.0f, Nc = 1.0f;
  const int seg_groups = a.seg_tiles * kSegGroups;
  const int nseg = a.segs_per_slice;
  int slot = 0, last_slot = 0;
  float R = 0.0f;
  bool first_cmd = true;
  for (;;) {
    if (rank == 0 && warp == 0) {
      __threadfence();
      WalkCmd cmd;
      cmd.final = 1;
      cmd.reuse = 0;
      if (first_cmd && !warp_tree_valid(a, base, lam)) {
        cmd.final = 2;
      } else {
        for (;;) {
          const float4 st4 = __ldcg(&a.ws_stats[base + u]);
          const int du = __ldg(&a.draft_row[base + u]);
          cmd.sp = make_sample_params(st4.x, st4.y, st4.z, st4.w, lam);
          cmd.u = u;
          if (pending_zero) {  // a residual of zero mass (round-off only): p~ of u
            cmd.kind = kWMixture;
            break;
          }
          if (search) {
            c = warp_first_child(a.parent + base, N, u, after);
            search = false;
          }
          if (c < 0) {  // no child left: the residual after rejections, or the bonus
            cmd.kind = rejected ? kWResidualC : (du >= 0 ? kWMixture : kWBonus);
            cmd.reuse = rejected;
            cmd.sp.c = cthr;
            break;
          }
          const int x = __ldg(&a.tokens[base + c]);
          const PosStats st{st4.x, st4.y, st4.z, st4.w};
          const float zt_x = Elem<T>::load(tgt + (base + u) * (int64_t)V + x);
          const float zq_x = Elem<T>::load(dft + (b * M + du) * (int64_t)V + x);
          float qx = 0.0f;
          const float r = accept_ratio(MODE == kLogitMix ? kLogitMix : kProbMix, st, zt_x, zq_x,
                                       lam, nullptr, &qx);
          const float ratio = rejected ? __fdiv_rn(fmaxf(0.0f, __fsub_rn(r, cthr)), Nc) : r;
          if (accept_test(__ldg(&a.u_accept[base + c]), ratio)) {
            if (lane == 0) {
              a.out_tokens[base + n] = x;
              a.out_path[base + n] = c;
            }
            ++n;
            u = c;
            after = c;
            search = true;
            rejected = 0;
            cthr = 0.0f;
            Nc = 1.0f;
            continue;
          }
          // rejected: the next threshold; the pass computes its mass N(cthr)
          rejected = 1;
          cthr = __fadd_rn(cthr, Nc);
          cmd.final = 0;
          cmd.kind = kWResidualC;
          cmd.sp.c = cthr;
          after = c;
          search = true;
          break;
        }
      }
      cmd.n = n;
      if (lane == 0)
        for (int r = 0; r < S; ++r) *cluster.map_shared_rank(&sh.cmd, r) = cmd;
      first_cmd = false;
    }
    cluster.sync();  // the command is visible in every rank
    const WalkCmd cmd = sh.cmd;
    if (cmd.final == 2) {  // invalid sequence
      if (rank == 0 && warp == 0) {
        for (int j = lane; j <= N; j += 32) {
          a.out_tokens[base + j] = -1;
          a.out_path[base + j] = -1;
        }
        if (lane == 0) a.out_n[b] = -1;
      }
      return;
    }
    const int du = __ldg(&a.draft_row[base + cmd.u]);
    const T *rowA = tgt + (base + cmd.u) * (int64_t)V;
    const T *rowB = dft + (b * M + (du >= 0 ? du : 0)) * (int64_t)V;
    if (!cmd.final || !cmd.reuse) {
      R = cluster_mass<T, MODE, ALIGNED>(sh, cluster, S, rank, rowA, rowB, V, g_lo, g_hi,
                                         seg_groups, nseg, cmd.kind, cmd.sp, slot);
      last_slot = slot;
      slot ^= 1;
    }
    if (!cmd.final) {  // the mass after a rejection
      Nc = R;
      if (!(R > 0.0f)) pending_zero = 1;
      continue;
    }

    // ---------------------------------------------- the final draw
    if (rank == 0 && warp == 0) {
      for (int j = lane; j <= N; j += 32) {
        if (j > cmd.n) a.out_tokens[base + j] = -1;
        if (j >= cmd.n) a.out_path[base + j] = -1;
      }
      if (lane == 0) a.out_n[b] = cmd.n;
    }
    if (!(R > 0.0f)) {
      if (rank == 0 && threadIdx.x == 0) a.out_tokens[base + cmd.n] = -1;
      return;
    }
    const float t = __fmul_rn(a.u_resample[b], R);
    int rstar = -1;
    float tloc = INFINITY, cum = 0.0f;
    for (int r = 0; r < S; ++r) {
      const float cn = __fadd_rn(cum, sh.masses[last_slot][r]);
      if (cn > t) {
        rstar = r;
        tloc = __fsub_rn(t, cum);
        break;
      }
      cum = cn;
    }
    if (rstar < 0) {  // u*R not below the total (round-off): last slice with mass
      for (int r = S - 1; r >= 0; --r)
        if (sh.masses[last_slot][r] > 0.0f) {
          rstar = r;
          break;
        }
      tloc = INFINITY;
    }
    if (rank != rstar) return;
    float lo = 0.0f;
    const int s = find_segment<kNT>(sh, nseg, tloc, &lo);
    if (warp != 0) return;
    int tok = -1;
    if (s >= 0) {
      const int sg_lo = g_lo + s * seg_groups;
      const int sg_hi = min(g_hi, sg_lo + seg_groups);
      tok = segment_walk<T, MODE, ALIGNED, kSegLaneGroups>(rowA, rowB, V, sg_lo, sg_hi, cmd.kind,
                                                           cmd.sp, lo, tloc);
    }
    if (lane == 0) a.out_tokens[base + cmd.n] = tok;
    return;
  }
}

template <typename T, int MODE, bool ALIGNED>
cudaError_t launch_one(const TreeArgs &a, int S, int64_t grid, cudaStream_t stream) {
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
  return cudaLaunchKernelEx(&cfg, tree_kernel<T, MODE, ALIGNED>, a);
}

template <typename T, int MODE, bool ALIGNED>
cudaError_t prepare_one() {
  return cudaFuncSetAttribute(tree_kernel<T, MODE, ALIGNED>,
                              cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

}  // namespace

cudaError_t tree_prepare() {
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

cudaError_t tree_launch(const TreeArgs &a, int dtype_bf16, int mode, bool aligned, int S,
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
