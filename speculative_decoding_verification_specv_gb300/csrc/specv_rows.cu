// specv_rows.cu -- the cluster row kernel: the verify/accept step for
// vocabularies too long for one CTA to hold a sequence.
//
// Work decomposition.  A "position" is (b, i), i in [0, K]: for i < K the pair
// (target row i, draft row i), for i = K the target row K alone (the bonus
// row).  Each position is one thread-block cluster of S CTAs; CTA `rank`
// streams the rank-th slice of the vocabulary of its position's row(s).
//
// Phase 1 (every cluster): one pass over HBM.  Each thread keeps running
// (max, sum-exp) statistics of its 16-byte groups (online softmax with a
// per-batch max, so each element costs one exp); warp butterflies and a
// fixed-order cross-warp merge give the CTA's partials; rank 0 merges the S
// partials over DSMEM in rank order and publishes the position's statistics
// to the scratch workspace.  The target and the draft row of a pair go
// through the same instruction sequence, so identical rows give bitwise
// identical statistics (and an acceptance ratio of exactly 1).  The bonus
// row is read by warps in segments (runs of consecutive groups), and the
// (max, sum-exp) of every segment is kept in the workspace as well.
//
// Phase 2 (the last cluster of sequence b to publish, found with one atomic
// counter per sequence): rank 0's first warp evaluates the acceptance test
// of every drafted position (the pages' loop: accept x_i iff
// u_i < min(1, p~(x_i)/q(x_i))), takes the first rejection n, and writes the
// accepted prefix.  The token at index n is then drawn by inverse CDF: over
// normalize(max(0, p~ - q)) of row n if n < K, over the target softmax of row
// K if every draft passed.  The search runs over segments.  For a rejected
// pair every warp sums the sampler weights of its segments of the slice, a
// block scan gives the running segment sums in index order, the S slice
// masses are exchanged over DSMEM, and the CTA whose slice holds
// u * (total mass) picks the segment holding it; one warp walks that segment
// in index order.  For the bonus row the segment masses follow from the
// phase-1 segment statistics, so only the chosen segment is read again.
// (Where round-off makes a walk end below its target, the last entry of
// positive weight in the segment is taken.)
//
// No thread ever waits on another cluster: the counter only decides which
// cluster does phase 2, and the only barriers are hardware cluster barriers.
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

constexpr int kNT = kRowThreads;  // threads per CTA
constexpr int kNW = kNT / 32;     // warps per CTA
constexpr int kUnroll = 4;        // 16-byte groups per thread per batch

struct Broadcast {
  int n;        // first rejected position (K if none), -1 if the sequence is invalid
  int kind;     // sampler weight kind (kWResidual / kWBonus / kWMixture)
  SampleParams sp;
  float u;      // u_resample[b]
};

struct __align__(16) RowsShared {
  BlockScratch<kNT> bs;
  float4 part[kMaxCluster];  // every rank's partial, pushed into rank 0's copy
  int last;
  Broadcast bc;
  float masses[2][kMaxCluster];
  float seg_lo;           // running sum before the chosen segment
  float segm[kMaxSegs];   // sampler weight of each segment of the slice
  float segi[kMaxSegs];   // running sums of segm in index order (inclusive)
};

// Row `r` of a device mirror (null when the launch has none).
template <typename T>
__device__ __forceinline__ T *mirror_row(void *mirror, int64_t r, int V) {
  return mirror == nullptr ? nullptr : static_cast<T *>(mirror) + r * (int64_t)V;
}

// Phase 1 of the bonus row: (max, sum-exp) of every segment of this CTA's
// slice, written to out[s] for s < nseg (an empty segment gives (-inf, 0)),
// and merged into lane 0's running statistics (the other lanes keep theirs
// empty).  Warp w reads segments w, w + kNW, ...; each tile of a segment is
// kSegLaneGroups coalesced 16-byte loads per lane.
template <typename T, bool ALIGNED>
__device__ void bonus_segment_stats(const T *row, int V, int g_lo, int g_hi, int seg_groups,
                                    int nseg, float2 *out, float &mA, float &sA, T *mir) {
  constexpr int VW = Elem<T>::kPerVec;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int s = warp; s < nseg; s += kNW) {
    const int sg_lo = g_lo + s * seg_groups;
    const int sg_hi = min(g_hi, sg_lo + seg_groups);
    float ms = -INFINITY, ss = 0.0f;
    for (int g0 = sg_lo; g0 < sg_hi; g0 += kSegGroups) {
      uint4 z[kSegLaneGroups];
#pragma unroll
      for (int u = 0; u < kSegLaneGroups; ++u) {
        const int g = g0 + u * 32 + lane;
        z[u] = g < sg_hi ? load_group<T, ALIGNED>(row, g, V) : neg_inf_group<T>();
        if (ALIGNED && mir != nullptr && g < sg_hi)
          __stcs(reinterpret_cast<uint4 *>(mir + (int64_t)g * Elem<T>::kPerVec), z[u]);
      }
      float bm = -INFINITY;
#pragma unroll
      for (int u = 0; u < kSegLaneGroups; ++u)
#pragma unroll
        for (int e = 0; e < VW; ++e) bm = fmaxf(bm, Elem<T>::get(z[u], e));
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) bm = fmaxf(bm, __shfl_xor_sync(0xffffffffu, bm, off));
      float bs = 0.0f;
      if (bm != -INFINITY) {  // warp-uniform
#pragma unroll
        for (int u = 0; u < kSegLaneGroups; ++u)
#pragma unroll
          for (int e = 0; e < VW; ++e) bs = __fadd_rn(bs, exp_shifted(Elem<T>::get(z[u], e), bm));
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) bs = __fadd_rn(bs, __shfl_xor_sync(0xffffffffu, bs, off));
      merge_stats(ms, ss, bm, bs);
    }
    if (lane == 0) {
      out[s] = make_float2(ms, ss);
      merge_stats(mA, sA, ms, ss);
    }
  }
  __threadfence();  // the segment statistics are visible device-wide before this position publishes
}

// Bonus token from the segment statistics phase 1 wrote for row K (run by
// one CTA): the mass of a segment is s_seg * exp(m_seg - mA) / S_A, the target
// softmax summed over it; block scans over the S slices' segments in index
// order give the total and route u * total to one segment, which warp 0
// walks.  Returns the token (valid in warp 0), or -1 if the row has no mass.
template <typename T, int MODE, bool ALIGNED>
__device__ int bonus_from_stats(RowsShared &sh, const RowArgs &a, const T *row, int S, int64_t b,
                                const SampleParams &sp, float u) {
  const int nseg = a.segs_per_slice;
  const int total = S * nseg;
  const float2 *st = a.ws_seg + b * (int64_t)S * nseg;
  auto mass = [&](int j) -> float {
    if (j >= total) return 0.0f;
    const float2 v = __ldcg(&st[j]);
    return v.x == -INFINITY ? 0.0f
                            : __fmul_rn(v.y, prob_from_offset(v.x, sp.nA));
  };
  float W = 0.0f;
  for (int j0 = 0; j0 < total; j0 += kNT) {
    float excl, incl, tot;
    block_scan<kNT>(sh.bs, mass(j0 + (int)threadIdx.x), excl, incl, tot);
    W = __fadd_rn(W, tot);
  }
  if (!(W > 0.0f)) return -1;
  float t = __fmul_rn(u, W);
  float base = 0.0f;
  int found = -1, lastpos = -1;
  if (threadIdx.x == 0) sh.bs.found = -1;
  for (int j0 = 0; j0 < total; j0 += kNT) {
    const int j = j0 + (int)threadIdx.x;
    const float m = mass(j);
    float excl, incl, tot;
    block_scan<kNT>(sh.bs, m, excl, incl, tot);
    const float l = __fadd_rn(base, excl), h = __fadd_rn(base, incl);
    if (j < total && l <= t && t < h) {
      sh.bs.found = j;
      sh.seg_lo = l;
    }
    if (m > 0.0f) lastpos = j;
    __syncthreads();
    found = sh.bs.found;
    __syncthreads();
    if (found >= 0) break;
    base = __fadd_rn(base, tot);
  }
  float lo = 0.0f;
  if (found >= 0) {
    lo = sh.seg_lo;
  } else {  // u * W not below the total (u >= 1): the last segment with mass, its last entry
    found = block_max_index<kNT>(sh.bs, lastpos);
    t = INFINITY;
  }
  if ((threadIdx.x >> 5) != 0 || found < 0) return -1;
  const int seg_groups = a.seg_tiles * kSegGroups;
  const int r = found / nseg, s = found - r * nseg;
  const int r_lo = r * a.groups_per_slice;
  const int r_hi = min(a.num_groups, r_lo + a.groups_per_slice);
  const int sg_lo = r_lo + s * seg_groups;
  const int sg_hi = min(r_hi, sg_lo + seg_groups);
  return segment_walk<T, MODE, ALIGNED, kSegLaneGroups>(row, row, a.V, sg_lo, sg_hi, kWBonus, sp,
                                                        lo, t);
}

// The token at one index of a sequence, by inverse CDF over the sampler
// weights of `kind` of the row(s), split over the S CTAs of the cluster (this
// CTA: groups [g_lo, g_hi) in nseg segments): segment masses, the S slice
// masses over DSMEM, the rank holding u * total routes it to a segment, one
// warp walks it; a residual of zero mass (round-off only) falls back to p~.
// Writes *out.  Every rank of the cluster calls it (cluster barriers inside).
template <typename T, int MODE, bool ALIGNED>
__device__ void draw_token(RowsShared &sh, cg::cluster_group &cluster, int S, int rank,
                           const T *sA_row, const T *sB_row, int V, int g_lo, int g_hi,
                           int seg_groups, int nseg, int kind, const SampleParams &sp, float u,
                           int32_t *out) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float R = 0.0f;
  int attempt = 0;
  for (;; ++attempt) {
    const float mass = segment_masses<T, MODE, ALIGNED, kSegLaneGroups, kNT>(
        sh, sA_row, sB_row, V, g_lo, g_hi, seg_groups, nseg, kind, sp);
    if (threadIdx.x == 0)
      for (int r = 0; r < S; ++r) cluster.map_shared_rank(sh.masses[attempt], r)[rank] = mass;
    cluster.sync();  // all slice masses exchanged
    R = 0.0f;
    for (int r = 0; r < S; ++r) R = __fadd_rn(R, sh.masses[attempt][r]);
    if (R > 0.0f || kind != kWResidual || attempt == 1) break;
    kind = kWMixture;  // zero residual mass (round-off only): draw from p~ instead
  }
  if (!(R > 0.0f)) {
    if (rank == 0 && threadIdx.x == 0) *out = -1;
    return;
  }
  const float t = __fmul_rn(u, R);
  int rstar = -1;
  float tloc = INFINITY;
  float c = 0.0f;
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
  if (rank != rstar) return;
  float lo = 0.0f;
  const int s = find_segment<kNT>(sh, nseg, tloc, &lo);
  if (warp != 0) return;
  if (s < 0) {  // no entry of positive weight in the routed slice (not reached: its mass is > 0)
    if (lane == 0) *out = -1;
    return;
  }
  const int sg_lo = g_lo + s * seg_groups;
  const int sg_hi = min(g_hi, sg_lo + seg_groups);
  const int tok = segment_walk<T, MODE, ALIGNED, kSegLaneGroups>(sA_row, sB_row, V, sg_lo, sg_hi,
                                                                  kind, sp, lo, tloc);
  if (lane == 0) *out = tok;
}

// Arrival of position (b, .) at the sequence's counter, after its statistics
// (and its own draw, if any) are written: returns 1 for the last of the K + 1
// positions, which resets the counter and the early-exit word for the next call.
__device__ __forceinline__ int arrive(const RowArgs &a, int64_t b, int K) {
  // one acquire-release atomic: this position's results (and, through the
  // cluster barrier before it, its ranks' fenced writes) before the count, and
  // for the last arrival every other position's results after it
  unsigned prev;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;"
               : "=r"(prev) : "l"(&a.ws_count[b]) : "memory");
  const int last = prev == (unsigned)K;
  if (last) {
    a.ws_count[b] = 0;  // every position has arrived: leave the counter zero for the next call
    if (a.ws_reject != nullptr) a.ws_reject[b] = 0;  // and the early-exit word
  }
  return last;
}

// Position statistics in the scratch: (mA, sA, mB, sB), with the sign of sB
// (a sum of exponentials, never negative) carrying the position's own
// decision: negative when its acceptance test rejects.
__device__ __forceinline__ float4 pack_stats(float mA, float sA, float mB, float sB, bool rejected) {
  return make_float4(mA, sA, mB, rejected ? -sB : sB);
}
__device__ __forceinline__ bool stats_rejected(const float4 &st) {
  return (__float_as_uint(st.w) >> 31) != 0u;
}
__device__ __forceinline__ PosStats stats_of(const float4 &st) {
  return PosStats{st.x, st.y, st.z, fabsf(st.w)};
}

// Sampler kind of the token at index n < K: the residual, or p~ itself when
// the residual is identically zero (lambda = 1: p~ = q in either mixture).
template <int MODE>
__device__ __forceinline__ int residual_kind(float lam) {
  return !(lam < 1.0f) ? kWMixture : kWResidual;
}

template <typename T, int MODE, bool ALIGNED, bool MIRROR = false>
__global__ void __launch_bounds__(kNT, 4) rows_kernel(RowArgs a) {
  __shared__ RowsShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int S = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t pl = (int64_t)blockIdx.x / S;  // the cluster's position in launch order
  const int K = a.K, V = a.V;
  int64_t b;
  int i;
  if (a.pos_major) {
    i = (int)(pl / a.B);
    b = pl - (int64_t)i * a.B;
  } else {
    b = pl / (K + 1);
    i = (int)(pl - b * (K + 1));
  }
  const int64_t p = b * (K + 1) + i;  // position index b*(K+1) + i
  const bool pair = i < K;
  const T *tgt = static_cast<const T *>(a.target);
  const T *dft = static_cast<const T *>(a.draft);
  const T *rowA = tgt + (b * (K + 1) + i) * (int64_t)V;
  const T *rowB = dft + (b * K + (pair ? i : 0)) * (int64_t)V;
  const int g_lo = rank * a.groups_per_slice;
  const int g_hi = min(a.num_groups, g_lo + a.groups_per_slice);
  const float lam_seq = a.lam[b];
  // Early exit (the pages' loop stops at the first rejection): a position
  // after one whose rejection is already published reads none of its rows.
  // Its partials stay empty; it never influences the outputs, since the first
  // rejection lies before it.
  bool skip = false;
  if (a.ws_reject != nullptr) {
    const unsigned v = __ldcg(&a.ws_reject[b]);
    skip = v != 0u && K + 1 - (int)v < i;
  }
  // The token-draw launch that follows (deferred sampling) may be scheduled
  // from now on; it waits for this whole grid to complete before it reads
  // anything this grid writes.
  if (a.defer_sampling) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // The inputs of this position's own acceptance test (rank 0's thread 0
  // decides): the drafted token and its uniform now, so that their latency
  // hides behind the stream; the two logits at the token right after it.
  int x_own = -1;
  float u_own = 0.0f, zt_own = 0.0f, zq_own = 0.0f;
  const bool decides = rank == 0 && threadIdx.x == 0 && pair && !skip;
  if (decides) {
    x_own = a.tokens[b * K + i];
    u_own = a.u_accept[b * K + i];
  }

  // ---------------------------------------------------------------- phase 1
  float mA = -INFINITY, sA = 0.0f, mB = -INFINITY, sB = 0.0f;
  const int seg_groups = a.seg_tiles * kSegGroups;
  const int nseg = a.segs_per_slice;
  if (skip) {
    // nothing to read: a rejection before this position is already published
  } else if (!pair && a.ws_seg != nullptr) {
    bonus_segment_stats<T, ALIGNED>(
        rowA, V, g_lo, g_hi, seg_groups, nseg, a.ws_seg + (b * S + rank) * (int64_t)nseg, mA, sA,
        MIRROR ? mirror_row<T>(a.mirror_target, b * (K + 1) + i, V) : nullptr);
  } else {
    // with early exit the stream stops when an earlier rejection is published meanwhile
    const bool stopped = slice_stats<T, MODE, ALIGNED, kNT, kUnroll>(
        rowA, rowB, pair, lam_seq, V, g_lo, g_hi, mA, sA, mB, sB,
        a.ws_reject != nullptr ? &a.ws_reject[b] : nullptr, i, K,
        MIRROR ? mirror_row<T>(a.mirror_target, b * (K + 1) + i, V) : nullptr,
        MIRROR ? mirror_row<T>(a.mirror_draft, b * K + (pair ? i : 0), V) : nullptr);
    skip = stopped;
  }
  if (decides && x_own >= 0 && x_own < V) {  // in flight during the merges below
    zt_own = Elem<T>::load(rowA + x_own);
    zq_own = Elem<T>::load(rowB + x_own);
  }
  if (a.ws_reject != nullptr) skip = __syncthreads_or(skip) != 0;  // CTA-wide: partial statistics
  block_merge_stats<kNT>(sh.bs, mA, sA, mB, sB);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) cluster.map_shared_rank(sh.part, 0)[rank] = make_float4(mA, sA, mB, sB);
  cluster.sync();  // every rank's partial is in rank 0's shared memory
  if (rank == 0 && threadIdx.x == 0) {
    float m0, s0, m1, s1;
    merge_stats2_n(S, [&](int r) { return sh.part[r]; }, m0, s0, m1, s1);
    // this position's own decision, from the merged statistics (the last
    // cluster of the sequence reads it back instead of testing again)
    bool own_reject = false;
    if (pair && !skip && x_own >= 0 && x_own < V && lambda_valid(lam_seq)) {
      const PosStats st{m0, s0, m1, s1};
      float qx = 0.0f;
      const float ratio = accept_ratio(MODE, st, zt_own, zq_own, lam_seq, nullptr, &qx);
      own_reject = !accept_test(u_own, ratio);
    }
    // early exit: publish a rejection at once
    if (own_reject && a.ws_reject != nullptr) atomicMax(&a.ws_reject[b], (unsigned)(K + 1 - i));
    a.ws_stats[p] = pack_stats(m0, s0, m1, s1, own_reject);
    const int last = arrive(a, b, K);
    for (int r = 0; r < S; ++r) *cluster.map_shared_rank(&sh.last, r) = last;
  }
  cluster.sync();  // sh.last is set in every rank; rank 0 is done reading partials
  if (!sh.last) return;

  // ---------------------------------------------------------------- phase 2
  if (rank == 0 && warp == 0) {
    __threadfence();
    const bool lam_ok = lambda_valid(lam_seq);
    bool lane_ok = true;
    int n = K;
    for (int i0 = 0; i0 < K; i0 += 32) {
      const int j = i0 + lane;
      bool rejected = false;
      if (j < K) {
        const int x = a.tokens[b * K + j];
        const bool tok_ok = x >= 0 && x < V;
        lane_ok = lane_ok && tok_ok;
        if (tok_ok && lam_ok) {
          const float4 st4 = __ldcg(&a.ws_stats[b * (K + 1) + j]);
          rejected = stats_rejected(st4);  // the position's own decision
          if (a.dbg_ptilde) {  // the debug entry point also reports p~(x), q(x)
            const float zt_x = Elem<T>::load(tgt + (b * (K + 1) + j) * (int64_t)V + x);
            const float zq_x = Elem<T>::load(dft + (b * K + j) * (int64_t)V + x);
            float px = 0.0f, qx = 0.0f;
            (void)accept_ratio(MODE, stats_of(st4), zt_x, zq_x, lam_seq, &px, &qx);
            a.dbg_ptilde[b * K + j] = px;
            if (a.dbg_q) a.dbg_q[b * K + j] = qx;
          }
        }
      }
      const unsigned rej = __ballot_sync(0xffffffffu, rejected);
      if (rej != 0u && n == K) n = i0 + __ffs(rej) - 1;
    }
    const bool all_tok = __all_sync(0xffffffffu, lane_ok);  // every lane votes
    const bool valid = lam_ok && all_tok;
    if (a.dbg_lse) {
      for (int j = lane; j <= K; j += 32) {
        const float4 st4 = __ldcg(&a.ws_stats[b * (K + 1) + j]);
        a.dbg_lse[(b * (K + 1) + j) * 2 + 0] = st4.x + lg2(st4.y) * kLn2;
        a.dbg_lse[(b * (K + 1) + j) * 2 + 1] = j < K ? st4.z + lg2(fabsf(st4.w)) * kLn2 : 0.0f;
      }
    }
    for (int j = lane; j <= K; j += 32) {
      int out = -1;
      if (valid && j < n) out = a.tokens[b * K + j];
      if (!valid || j != n) a.out_tokens[b * (K + 1) + j] = out;
    }
    if (lane == 0) {
      a.out_n[b] = valid ? n : -1;
      Broadcast bc;
      bc.n = valid ? n : -1;
      bc.u = a.u_resample[b];
      const PosStats st = stats_of(__ldcg(&a.ws_stats[b * (K + 1) + (valid ? n : 0)]));
      bc.sp = make_sample_params_rn(st.mA, st.sA, st.mB, st.sB, lam_seq);
      bc.kind = n == K ? kWBonus : residual_kind<MODE>(lam_seq);
      if (!a.defer_sampling)
        for (int r = 0; r < S; ++r) *cluster.map_shared_rank(&sh.bc, r) = bc;
    }
  }
  if (a.defer_sampling) return;  // rows_sample draws the tokens (no DSMEM traffic above)
  cluster.sync();  // broadcast visible everywhere
  const Broadcast bc = sh.bc;
  if (bc.n < 0) return;
  // the second read of the rows: from the device mirror when there is one
  const T *tsrc = MIRROR ? static_cast<const T *>(a.mirror_target) : tgt;
  const T *dsrc = MIRROR ? static_cast<const T *>(a.mirror_draft) : dft;
  const T *sA_row = tsrc + (b * (K + 1) + bc.n) * (int64_t)V;
  const T *sB_row = dsrc + (b * K + (bc.n < K ? bc.n : 0)) * (int64_t)V;
  if (bc.kind == kWBonus && a.ws_seg != nullptr) {
    // every draft accepted: the bonus row's segment statistics are in the workspace
    if (rank != 0) return;
    __threadfence();
    const int tok = bonus_from_stats<T, MODE, ALIGNED>(sh, a, sA_row, S, b, bc.sp, bc.u);
    if (threadIdx.x == 0) a.out_tokens[b * (K + 1) + bc.n] = tok;
    return;
  }
  draw_token<T, MODE, ALIGNED>(sh, cluster, S, rank, sA_row, sB_row, V, g_lo, g_hi, seg_groups,
                               nseg, bc.kind, bc.sp, bc.u, a.out_tokens + b * (K + 1) + bc.n);
}

// The deferred token draws: one cluster of S CTAs per sequence (a wider
// cluster than the statistics launch's, so that each CTA's share of the
// second read is small), after the statistics launch has written out_n and
// the position statistics.  The sampler's weight kind and parameters follow
// from out_n[b] exactly as the statistics launch's last cluster derives them.
template <typename T, int MODE, bool ALIGNED>
__global__ void __launch_bounds__(kNT, 4) rows_sample_kernel(RowArgs a) {
  __shared__ RowsShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int S = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t b = (int64_t)blockIdx.x / S;
  const int K = a.K, V = a.V;
  // launched as a programmatic dependent of the statistics launch: wait until
  // that grid has completed and its writes are visible
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n = a.out_n[b];
  if (n < 0) return;  // invalid sequence (or a timed-out copy): nothing to draw
  const float lam = a.lam[b];
  const PosStats st = stats_of(__ldcg(&a.ws_stats[b * (K + 1) + n]));
  const SampleParams sp = make_sample_params_rn(st.mA, st.sA, st.mB, st.sB, lam);
  const int kind = n == K ? kWBonus : residual_kind<MODE>(lam);
  const float u = a.u_resample[b];
  const T *tgt = static_cast<const T *>(a.target);
  const T *dft = static_cast<const T *>(a.draft);
  const T *tsrc = a.mirror_target != nullptr ? static_cast<const T *>(a.mirror_target) : tgt;
  const T *dsrc = a.mirror_draft != nullptr ? static_cast<const T *>(a.mirror_draft) : dft;
  const T *sA_row = tsrc + (b * (K + 1) + n) * (int64_t)V;
  const T *sB_row = dsrc + (b * K + (n < K ? n : 0)) * (int64_t)V;
  int32_t *out = a.out_tokens + b * (K + 1) + n;
  if (kind == kWBonus && a.ws_seg != nullptr) {
    if (rank != 0) return;
    RowArgs a1 = a;  // the statistics launch's geometry of the segment statistics
    a1.groups_per_slice = a.stats_groups_per_slice;
    a1.seg_tiles = a.stats_seg_tiles;
    a1.segs_per_slice = a.stats_segs_per_slice;
    const int tok = bonus_from_stats<T, MODE, ALIGNED>(sh, a1, sA_row, a.stats_cluster, b, sp, u);
    if (threadIdx.x == 0) *out = tok;
    return;
  }
  const int g_lo = rank * a.groups_per_slice;
  const int g_hi = min(a.num_groups, g_lo + a.groups_per_slice);
  draw_token<T, MODE, ALIGNED>(sh, cluster, S, rank, sA_row, sB_row, V, g_lo, g_hi,
                               a.seg_tiles * kSegGroups, a.segs_per_slice, kind, sp, u, out);
}

// One cluster per SEQUENCE (grid B * S; plan for grids of about one wave):
// the CTAs of the cluster stream the sequence's rows (the target and draft
// rows of positions 0..K-1, then target row K) in S contiguous parts and
// push their partial statistics of every position into rank 0's shared
// memory.  After one cluster barrier rank 0's first warp merges them (lane =
// position), takes the acceptance tests (their inputs were loaded while the
// rows streamed), finds the first rejection n and writes the outputs; the
// token at n is then drawn by the whole cluster from its slices of row pair
// n (or of target row K) -- the rows were streamed moments ago, so the second
// read hits L2 -- with no second launch, no scratch memory and no arrival
// counter.  Dynamic shared memory: the copy ring (logit rule, aligned rows;
// see seq_staged), the partials [K+1][S] of every rank (used in rank 0), then
// the drafted tokens, acceptance uniforms and the resample uniform of the
// sequence (copied in by rank 0's first warp).
extern __shared__ float4 g_seq_smem[];

// Work units of one group of a pair position against one group of the bonus
// row: the bytes (2 : 1) in the probability rule; the logit rule's mixed row
// costs about 1.6 times as much per byte (Qwen-shaped batch, B = 32, K = 5,
// V = 152064 bf16, with 2 : 1: CTAs on pair positions streamed for 26.8 us
// median, those on the bonus row 16.7 us, for equal bytes), hence 3 : 1.
template <int MODE>
constexpr int kSeqPairUnits = MODE == kLogitMix ? 3 : 2;

// The logit rule's parts of aligned rows stream through a ring of per-thread
// asynchronous copies (slice_stats_staged, kSeqDepth groups per row in
// flight), the others with batches of register loads: measured at B = 32,
// K = 5, V = 152064 bf16 (GB300, one launch per step after an L2 flush), the
// ring gave 47.6 against 51.2 us in the logit rule but 41.5 against 41.1 us
// in the probability rule, whose lighter arithmetic the one-group folds of
// the ring outweigh.
constexpr int kSeqDepth = 4;
constexpr int kSeqRing = (kSeqDepth + 1) * 2 * kNT;  // 16-byte slots of the copy ring
template <int MODE, bool ALIGNED>
__host__ __device__ constexpr bool seq_staged() { return ALIGNED && MODE == kLogitMix; }

__host__ __device__ constexpr int64_t seq_smem_bytes(int K, int S, bool staged) {
  return (staged ? (int64_t)kSeqRing * 16 : 0) + (int64_t)(K + 1) * S * 16 +
         (2 * kSeqMaxPositions + 4) * 4;
}

template <typename T, int MODE, bool ALIGNED>
__global__ void __launch_bounds__(kNT, 4) rows_seq_kernel(RowArgs a) {
  __shared__ RowsShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int S = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t b = (int64_t)blockIdx.x / S;
  const int K = a.K, V = a.V;
  const T *tgt = static_cast<const T *>(a.target) + b * (K + 1) * (int64_t)V;
  const T *dft = static_cast<const T *>(a.draft) + b * K * (int64_t)V;
  const int g_lo = rank * a.groups_per_slice;
  const int g_hi = min(a.num_groups, g_lo + a.groups_per_slice);
  const float lam = a.lam[b];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const bool decider = rank == 0 && warp == 0;
  uint4 *ring = reinterpret_cast<uint4 *>(g_seq_smem);  // [kSeqDepth + 1][2][kNT] when staged
  float4 *part = g_seq_smem + (seq_staged<MODE, ALIGNED>() ? kSeqRing : 0);  // [K+1][S]
  int *pre_x = reinterpret_cast<int *>(part + (K + 1) * S);  // [kSeqMaxPositions]
  float *pre_u = reinterpret_cast<float *>(pre_x + kSeqMaxPositions);  // [kSeqMaxPositions]
  float *pre_ur = pre_u + kSeqMaxPositions;
  // the decision inputs, copied into shared memory while the rows stream
  if (decider) {
    for (int j = lane; j < K; j += 32) {
      cp_async4(pre_x + j, a.tokens + b * K + j);
      cp_async4(pre_u + j, a.u_accept + b * K + j);
    }
    if (lane == 0) cp_async4(pre_ur, a.u_resample + b);
  }

  // ------------------------------------------------- statistics of every position
  // The sequence's rows as one range of work units (a pair position's group
  // is kSeqPairUnits units, a bonus-row group 1), cut into S equal contiguous parts: CTA
  // `rank` streams its part -- long runs of at most a few positions, like a
  // one-position cluster's slice -- and contributes a partial to every
  // position its part touches (the identity to the others).
  float4 *part0 = cluster.map_shared_rank(part, 0);
  {
    // this part: from group g_first of position i_first to group g_last
    // (exclusive) of position i_last
    const int G = a.num_groups;
    int i_first, g_first, i_last, g_last;
    {
      const int64_t total = ((int64_t)kSeqPairUnits<MODE> * K + 1) * G;
      const int64_t per = (total + S - 1) / S;
      const int64_t u_lo = min(total, (int64_t)rank * per), u_hi = min(total, u_lo + per);
      auto locate = [&](int64_t u, int &i, int &g) {  // the first group at or after unit u
        const int64_t ip = u / ((int64_t)kSeqPairUnits<MODE> * G);
        i = ip < K ? (int)ip : K;
        const int upg = i < K ? kSeqPairUnits<MODE> : 1;
        g = (int)((u - (int64_t)kSeqPairUnits<MODE> * i * G + upg - 1) / upg);
      };
      locate(u_lo, i_first, g_first);
      locate(u_hi, i_last, g_last);
      if (g_last == 0 && i_last > i_first) {  // the part ends at a position boundary
        --i_last;
        g_last = G;
      }
    }
    for (int i = (int)threadIdx.x; i <= K; i += kNT)  // positions this part does not touch
      if (i < i_first || i > i_last) part0[i * S + rank] = make_float4(-INFINITY, 0.0f, -INFINITY, 0.0f);
    for (int i = i_first; i <= i_last; ++i) {
      const int gl = i == i_first ? g_first : 0, gh = i == i_last ? g_last : G;
      // The bonus row alone streams its two halves as the two rows of a
      // plain pair (as many loads in flight as a pair position; lambda 0
      // makes the logit rule's fold the plain one), then the groups left
      // over -- an odd one, and the row's partial last group, whose bounds
      // check needs its own index -- as a single row; the statistics of the
      // pieces are merged.
      const bool bonus = i == K;
      const int gp = (bonus && gh == G && V % Elem<T>::kPerVec != 0) ? gh - 1 : gh;
      const int h = bonus ? (gp > gl ? (gp - gl) / 2 : 0) : gh - gl;
      const T *rowA = tgt + (int64_t)i * V;
      float mA = -INFINITY, sA = 0.0f, mB = -INFINITY, sB = 0.0f;
      for (int c = 0; c < (bonus ? 2 : 1); ++c) {
        const bool pr = c == 0;
        const T *rowB = bonus ? rowA + (int64_t)h * Elem<T>::kPerVec : dft + (int64_t)i * V;
        float a0 = -INFINITY, a1 = 0.0f, b0 = -INFINITY, b1 = 0.0f;
        if constexpr (seq_staged<MODE, ALIGNED>())
          slice_stats_staged<T, MODE, kNT, kSeqDepth>(rowA, rowB, pr, bonus ? 0.0f : lam,
                                                      pr ? gl : gl + 2 * h, pr ? gl + h : gh, ring,
                                                      a0, a1, b0, b1);
        else
          slice_stats<T, MODE, ALIGNED, kNT, kUnroll>(rowA, rowB, pr, bonus ? 0.0f : lam, V,
                                                    pr ? gl : gl + 2 * h, pr ? gl + h : gh, a0, a1,
                                                    b0, b1);
        if (bonus) {
          merge_stats(mA, sA, a0, a1);
          merge_stats(mA, sA, b0, b1);
        } else {
          mA = a0;
          sA = a1;
          mB = b0;
          sB = b1;
        }
      }
      block_merge_stats<kNT>(sh.bs, mA, sA, mB, sB);
      if (threadIdx.x == 0) part0[i * S + rank] = make_float4(mA, sA, mB, sB);
    }
  }
  // the logits at the first 32 drafted tokens, in flight during the barrier
  float zt_pre = 0.0f, zq_pre = 0.0f;
  if (decider) {
    cp_async_wait_all();
    __syncwarp();
    const int x = lane < K ? pre_x[lane] : -1;
    if (x >= 0 && x < V) {
      zt_pre = Elem<T>::load(tgt + (int64_t)lane * V + x);
      zq_pre = Elem<T>::load(dft + (int64_t)lane * V + x);
    }
  }
  cluster.sync();  // every rank's partials of every position are in rank 0's shared memory

  // ------------------------------------------------- decisions (rank 0, warp 0)
  if (decider) {
    const bool lam_ok = lambda_valid(lam);
    bool lane_ok = true;
    int n = K;
    float4 st0 = make_float4(-INFINITY, 0.0f, -INFINITY, 0.0f);  // position `lane`'s statistics
    for (int i0 = 0; i0 < K; i0 += 32) {
      const int j = i0 + lane;
      bool rejected = false;
      if (j < K) {
        const int x = pre_x[j];
        const bool tok_ok = x >= 0 && x < V;
        lane_ok = lane_ok && tok_ok;
        PosStats st;
        merge_stats2_n(S, [&](int r) { return part[j * S + r]; }, st.mA, st.sA, st.mB, st.sB);
        if (i0 == 0) st0 = make_float4(st.mA, st.sA, st.mB, st.sB);
        if (tok_ok && lam_ok) {
          const float zt_x = i0 == 0 ? zt_pre : Elem<T>::load(tgt + (int64_t)j * V + x);
          const float zq_x = i0 == 0 ? zq_pre : Elem<T>::load(dft + (int64_t)j * V + x);
          float px = 0.0f, qx = 0.0f;
          const float ratio =
              accept_ratio(MODE, st, zt_x, zq_x, lam, a.dbg_ptilde ? &px : nullptr, &qx);
          rejected = !accept_test(pre_u[j], ratio);
          if (a.dbg_ptilde) a.dbg_ptilde[b * K + j] = px;
          if (a.dbg_q) a.dbg_q[b * K + j] = qx;
        }
      }
      const unsigned rej = __ballot_sync(0xffffffffu, rejected);
      if (rej != 0u && n == K) n = i0 + __ffs(rej) - 1;
    }
    const bool valid = lam_ok && __all_sync(0xffffffffu, lane_ok);  // every lane votes
    if (a.dbg_lse) {
      for (int j = lane; j <= K; j += 32) {
        float m0, s0, m1, s1;
        merge_stats2_n(S, [&](int r) { return part[j * S + r]; }, m0, s0, m1, s1);
        a.dbg_lse[(b * (K + 1) + j) * 2 + 0] = m0 + lg2(s0) * kLn2;
        a.dbg_lse[(b * (K + 1) + j) * 2 + 1] = j < K ? m1 + lg2(s1) * kLn2 : 0.0f;
      }
    }
    for (int j = lane; j <= K; j += 32) {
      int out = -1;
      if (valid && j < n) out = pre_x[j];
      if (!valid || j != n) a.out_tokens[b * (K + 1) + j] = out;
    }
    // the statistics of the drawn row: lane n's (a rejected position < 32),
    // else merged again (the bonus row, or a rejection past the first 32)
    const int nd = valid ? n : 0;
    float4 sn;
    sn.x = __shfl_sync(0xffffffffu, st0.x, nd & 31);
    sn.y = __shfl_sync(0xffffffffu, st0.y, nd & 31);
    sn.z = __shfl_sync(0xffffffffu, st0.z, nd & 31);
    sn.w = __shfl_sync(0xffffffffu, st0.w, nd & 31);
    if (nd >= 32 || nd == K)
      merge_stats2_n(S, [&](int r) { return part[nd * S + r]; }, sn.x, sn.y, sn.z, sn.w);
    Broadcast bc;
    bc.n = valid ? n : -1;
    bc.u = *pre_ur;
    bc.sp = make_sample_params_rn(sn.x, sn.y, sn.z, sn.w, lam);
    bc.kind = n == K ? kWBonus : residual_kind<MODE>(lam);
    if (lane == 0) a.out_n[b] = bc.n;
    if (lane < S) *cluster.map_shared_rank(&sh.bc, lane) = bc;
  }
  cluster.sync();  // the decision is in every rank
  const Broadcast bc = sh.bc;
  if (bc.n < 0) return;  // invalid input: every output is -1 already
  const T *sA_row = tgt + (int64_t)bc.n * V;
  const T *sB_row = dft + (int64_t)(bc.n < K ? bc.n : 0) * V;
  draw_token<T, MODE, ALIGNED>(sh, cluster, S, rank, sA_row, sB_row, V, g_lo, g_hi,
                               a.seg_tiles * kSegGroups, a.segs_per_slice, bc.kind, bc.sp, bc.u,
                               a.out_tokens + b * (K + 1) + bc.n);
}

// Greedy verification with the same decomposition (one cluster per position,
// rank r streams slice r): each rank finds the argmax of the mixed logits
// w = z_t + lambda (z_q - z_t) over its slice (target row K alone at the bonus
// position), the first maximum in index order; rank 0 merges the S candidates
// in rank order and publishes (max, index).  The last cluster of the sequence
// accepts x_i iff it is the argmax of row i, stops at the first mismatch and
// emits that argmax there, or the argmax of target row K when every draft
// matches.  There is no sampling pass: each logit is read once.
template <typename T, bool ALIGNED>
__global__ void __launch_bounds__(kNT, 4) rows_greedy_kernel(RowArgs a) {
  constexpr int VW = Elem<T>::kPerVec;
  __shared__ RowsShared sh;
  cg::cluster_group cluster = cg::this_cluster();
  const int S = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int64_t pl = (int64_t)blockIdx.x / S;  // the cluster's position in launch order
  const int K = a.K, V = a.V;
  int64_t b;
  int i;
  if (a.pos_major) {
    i = (int)(pl / a.B);
    b = pl - (int64_t)i * a.B;
  } else {
    b = pl / (K + 1);
    i = (int)(pl - b * (K + 1));
  }
  const int64_t p = b * (K + 1) + i;
  const bool pair = i < K;
  const T *tgt = static_cast<const T *>(a.target);
  const T *dft = static_cast<const T *>(a.draft);
  const T *rowA = tgt + (b * (K + 1) + i) * (int64_t)V;
  const T *rowB = dft + (b * K + (pair ? i : 0)) * (int64_t)V;
  const int g_lo = rank * a.groups_per_slice;
  const int g_hi = min(a.num_groups, g_lo + a.groups_per_slice);
  const float lam = a.lam[b];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // early exit: nothing to read after a published mismatch of this sequence
  bool skip = false;
  if (a.ws_reject != nullptr) {
    const unsigned v = __ldcg(&a.ws_reject[b]);
    skip = v != 0u && K + 1 - (int)v < i;
  }

  float best = -INFINITY;
  int bidx = INT_MAX;
  // (skip: an earlier position of this sequence is already known to mismatch)
  unsigned seen = 0u;  // early exit while streaming, as in slice_stats
  int it = 0;
  for (int g0 = g_lo + (int)threadIdx.x; !skip && g0 < g_hi; g0 += kNT * kUnroll, ++it) {
    if (a.ws_reject != nullptr && it % kExitEvery == 0) {
      if (seen != 0u && K + 1 - (int)seen < i) {
        skip = true;
        break;
      }
      seen = __ldcg(&a.ws_reject[b]);
    }
    uint4 za[kUnroll], zb[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int g = g0 + u * kNT;
      if (g < g_hi) {
        za[u] = load_group<T, ALIGNED>(rowA, g, V);
        if (pair) zb[u] = load_group<T, ALIGNED>(rowB, g, V);
      }
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int g = g0 + u * kNT;
      if (g < g_hi) greedy_fold_group<T>(za[u], pair ? zb[u] : za[u], pair, lam, g * VW, best, bidx);
    }
  }
  if (a.ws_reject != nullptr) skip = __syncthreads_or(skip) != 0;  // CTA-wide: partial candidates
  warp_argmax(best, bidx);
  if (lane == 0) {
    sh.bs.red[warp][0] = best;
    sh.bs.red[warp][1] = __int_as_float(bidx);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = -INFINITY;
    int ix = INT_MAX;
    for (int w = 0; w < kNW; ++w) argmax_merge(m, ix, sh.bs.red[w][0], __float_as_int(sh.bs.red[w][1]));
    cluster.map_shared_rank(sh.part, 0)[rank] = make_float4(m, __int_as_float(ix), 0.0f, 0.0f);
  }
  cluster.sync();  // every rank's candidate is in rank 0's shared memory
  if (rank == 0 && threadIdx.x == 0) {
    float m = -INFINITY;
    int ix = INT_MAX;
    for (int r = 0; r < S; ++r) argmax_merge(m, ix, sh.part[r].x, __float_as_int(sh.part[r].y));
    if (a.ws_reject != nullptr && pair && !skip) {
      // publish this position's mismatch (the last cluster repeats the test)
      const int x = a.tokens[b * K + i];
      if (x >= 0 && x < V && lambda_valid(lam) && ix != x)
        atomicMax(&a.ws_reject[b], (unsigned)(K + 1 - i));
    }
    a.ws_stats[p] = make_float4(m, __int_as_float(ix), 0.0f, 0.0f);
    const int last = arrive(a, b, K);
    for (int r = 0; r < S; ++r) *cluster.map_shared_rank(&sh.last, r) = last;
  }
  cluster.sync();  // sh.last is set in every rank; rank 0 is done reading candidates
  if (!sh.last || rank != 0 || warp != 0) return;

  // the sequence: accept while x_i is the argmax of row i
  __threadfence();
  const bool lam_ok = lambda_valid(lam);
  bool lane_ok = true;
  int n = K;
  for (int i0 = 0; i0 < K; i0 += 32) {
    const int j = i0 + lane;
    bool rejected = false;
    if (j < K) {
      const int x = a.tokens[b * K + j];
      const bool tok_ok = x >= 0 && x < V;
      lane_ok = lane_ok && tok_ok;
      if (tok_ok && lam_ok) rejected = __float_as_int(__ldcg(&a.ws_stats[b * (K + 1) + j]).y) != x;
    }
    const unsigned rej = __ballot_sync(0xffffffffu, rejected);
    if (rej != 0u && n == K) n = i0 + __ffs(rej) - 1;
  }
  const bool valid = lam_ok && __all_sync(0xffffffffu, lane_ok);  // every lane votes
  for (int j = lane; j <= K; j += 32) {
    int out = -1;
    if (valid && j < n) out = a.tokens[b * K + j];
    if (valid && j == n) out = __float_as_int(__ldcg(&a.ws_stats[b * (K + 1) + n]).y);
    a.out_tokens[b * (K + 1) + j] = out;
  }
  if (lane == 0) a.out_n[b] = valid ? n : -1;
}

template <typename T, int MODE, bool ALIGNED, bool MIRROR = false>
constexpr void (*row_kernel_of())(RowArgs) {
  if constexpr (MODE == kGreedy)
    return rows_greedy_kernel<T, ALIGNED>;
  else
    return rows_kernel<T, MODE, ALIGNED, MIRROR>;
}

template <typename T, int MODE, bool ALIGNED>
cudaError_t launch_one(const RowArgs &a, int S, int64_t grid, cudaStream_t stream) {
  // the mirrored variant (aligned sampling rows with device copies to fill)
  constexpr bool kCanMirror = ALIGNED && MODE != kGreedy;
  void (*kern)(RowArgs) = (kCanMirror && a.mirror_target != nullptr)
                              ? row_kernel_of<T, MODE, ALIGNED, kCanMirror>()
                              : row_kernel_of<T, MODE, ALIGNED>();
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
  return cudaLaunchKernelEx(&cfg, kern, a);
}

template <typename T, int MODE, bool ALIGNED>
cudaError_t launch_sample_one(const RowArgs &a, int S, int64_t grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kNT, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  // programmatic dependent launch: scheduled while the statistics launch
  // finishes, released by its completion (griddepcontrol.wait)
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, rows_sample_kernel<T, MODE, ALIGNED>, a);
}

template <typename T, int MODE, bool ALIGNED>
cudaError_t launch_seq_one(const RowArgs &a, int S, int64_t grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid, 1, 1);
  cfg.blockDim = dim3(kNT, 1, 1);
  cfg.dynamicSmemBytes = (size_t)seq_smem_bytes(a.K, S, seq_staged<MODE, ALIGNED>());
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, rows_seq_kernel<T, MODE, ALIGNED>, a);
}

template <typename T, int MODE, bool ALIGNED>
cudaError_t prepare_one() {
  cudaError_t e = cudaFuncSetAttribute(row_kernel_of<T, MODE, ALIGNED>(),
                                       cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if constexpr (ALIGNED && MODE != kGreedy) {
    const cudaError_t e1 = cudaFuncSetAttribute(row_kernel_of<T, MODE, true, true>(),
                                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) e = e1;
  }
  if constexpr (MODE != kGreedy) {
    const cudaError_t e2 = cudaFuncSetAttribute(rows_sample_kernel<T, MODE, ALIGNED>,
                                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) e = e2;
    const cudaError_t e3 = cudaFuncSetAttribute(rows_seq_kernel<T, MODE, ALIGNED>,
                                                cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) e = e3;
    const cudaError_t e4 = cudaFuncSetAttribute(rows_seq_kernel<T, MODE, ALIGNED>,
                                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                (int)seq_smem_bytes(kSeqMaxPositions - 1, kMaxCluster, true));
    if (e == cudaSuccess) e = e4;
  }
  return e;
}

}  // namespace

cudaError_t rows_prepare() {
  cudaError_t e = cudaSuccess;
  cudaError_t r;
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
  SPECV_PREP(float, kGreedy, true)
  SPECV_PREP(float, kGreedy, false)
  SPECV_PREP(uint16_t, kGreedy, true)
  SPECV_PREP(uint16_t, kGreedy, false)
#undef SPECV_PREP
  return e;
}

cudaError_t rows_launch(const RowArgs &a, int dtype_bf16, int mode, bool aligned, int S,
                        int64_t grid, cudaStream_t stream) {
  if (mode == kGreedy) {
    if (dtype_bf16)
      return aligned ? launch_one<uint16_t, kGreedy, true>(a, S, grid, stream)
                     : launch_one<uint16_t, kGreedy, false>(a, S, grid, stream);
    return aligned ? launch_one<float, kGreedy, true>(a, S, grid, stream)
                   : launch_one<float, kGreedy, false>(a, S, grid, stream);
  }
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

namespace specv {

cudaError_t rows_sample_launch(const RowArgs &a, int dtype_bf16, int mode, bool aligned, int S,
                               int64_t grid, cudaStream_t stream) {
  if (dtype_bf16) {
    if (mode == kProbMix)
      return aligned ? launch_sample_one<uint16_t, kProbMix, true>(a, S, grid, stream)
                     : launch_sample_one<uint16_t, kProbMix, false>(a, S, grid, stream);
    return aligned ? launch_sample_one<uint16_t, kLogitMix, true>(a, S, grid, stream)
                   : launch_sample_one<uint16_t, kLogitMix, false>(a, S, grid, stream);
  }
  if (mode == kProbMix)
    return aligned ? launch_sample_one<float, kProbMix, true>(a, S, grid, stream)
                   : launch_sample_one<float, kProbMix, false>(a, S, grid, stream);
  return aligned ? launch_sample_one<float, kLogitMix, true>(a, S, grid, stream)
                 : launch_sample_one<float, kLogitMix, false>(a, S, grid, stream);
}

cudaError_t rows_seq_launch(const RowArgs &a, int dtype_bf16, int mode, bool aligned, int S,
                            cudaStream_t stream) {
  const int64_t grid = a.B * (int64_t)S;
  if (dtype_bf16) {
    if (mode == kProbMix)
      return aligned ? launch_seq_one<uint16_t, kProbMix, true>(a, S, grid, stream)
                     : launch_seq_one<uint16_t, kProbMix, false>(a, S, grid, stream);
    return aligned ? launch_seq_one<uint16_t, kLogitMix, true>(a, S, grid, stream)
                   : launch_seq_one<uint16_t, kLogitMix, false>(a, S, grid, stream);
  }
  if (mode == kProbMix)
    return aligned ? launch_seq_one<float, kProbMix, true>(a, S, grid, stream)
                   : launch_seq_one<float, kProbMix, false>(a, S, grid, stream);
  return aligned ? launch_seq_one<float, kLogitMix, true>(a, S, grid, stream)
                 : launch_seq_one<float, kLogitMix, false>(a, S, grid, stream);
}

}  // namespace specv
