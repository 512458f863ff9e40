// specv_sweep.cu -- the sweep row kernel: the verify/accept step for long
// rows that start on 16-byte boundaries, streamed by persistent CTAs.
//
// Work decomposition.  Every row is cut into chunks of chunk_groups 16-byte
// groups.  An item is chunk c of position (b, i): the chunk of target row i
// together with the same chunk of draft row i for i < K, the chunk of target
// row K alone for the bonus position.  Items are numbered position-major and
// CTA x takes items x, x + grid, x + 2 grid, ...: at any moment the running
// CTAs read one contiguous window of the logits, and the rows of a sequence
// are finished within a short stretch of the stream (so the sampler's second
// read of a row finds it in L2).
//
// Streaming.  Each CTA keeps kSweepStages items in flight: thread 0 starts a
// 1-D bulk copy (TMA) of the next item into a free stage of shared memory,
// completing on that stage's mbarrier; all threads wait on the mbarrier with
// a time limit, compute the chunk's (max, sum-exp) statistics of both rows
// from shared memory (one exp per element), and release the stage.
//
// Bookkeeping.  The chunk statistics go to the workspace; one atomic counter
// per position finds the CTA that publishes the last chunk of a row, which
// merges the row's chunk statistics in chunk order (so the result does not
// depend on arrival order) and publishes the position's statistics; one
// counter per sequence finds the CTA that publishes the last position, which
// finishes the sequence before taking its next item: the acceptance test of
// every drafted position, the first rejection n, and the token at index n by
// inverse CDF -- over the residual normalize(max(0, p~ - q)) of row n (segment
// masses, then a walk of one segment), or over the target softmax of row K
// when every draft passed (routed through the chunk statistics of row K, then
// a walk of one chunk).  Every counter is left at zero for the next launch.
//
// The target and draft chunk of a pair go through the same instructions, so
// identical rows give identical statistics (an acceptance ratio of exactly
// 1).  A copy that does not land within the time limit marks its chunk as
// failed: the CTA stops copying, every position it touches later is marked
// failed too, and the affected sequences report out_n = -2.
#include "specv_block.cuh"
#include "specv_device.cuh"
#include "specv_internal.h"
#include "specv_segments.cuh"

namespace specv {

namespace {

constexpr int kNT = kSweepThreads;
constexpr int kNW = kNT / 32;
constexpr int kNS = kSweepStages;
constexpr int kGPT = 4;  // groups per thread per pass over a chunk

struct SweepBroadcast {
  int n;       // first rejected position (K if none), -1 if nothing is sampled
  int kind;    // sampler weight kind
  SampleParams sp;
  float u;     // u_resample[b]
};

struct __align__(16) SweepShared {
  BlockScratch<kNT> bs;
  float4 wpart[kNW];   // per-warp chunk statistics
  long long finish;    // sequence to finish after the current item, -1 if none
  SweepBroadcast bc;
  float seg_lo;
  float segm[kMaxSegs];
  float segi[kMaxSegs];
};

// Statistics (mA, sA, mB, sB) with sA < 0 mark a chunk or position whose copy
// failed.
__device__ __forceinline__ float4 failed_stats() {
  return make_float4(-INFINITY, -1.0f, -INFINITY, -1.0f);
}

// Warp reduction of per-lane (m, s) statistics: the warp max first, then each
// lane's sum rescaled to it and summed by a butterfly in a fixed order.  Every
// lane ends with the result; empty statistics are (-inf, 0).
__device__ __forceinline__ void warp_stats(float &m, float &s) {
  float mw = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) mw = fmaxf(mw, __shfl_xor_sync(0xffffffffu, mw, off));
  float sc = (m == mw) ? s : (m == -INFINITY ? 0.0f : __fmul_rn(s, exp_shifted(m, mw)));
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sc = __fadd_rn(sc, __shfl_xor_sync(0xffffffffu, sc, off));
  m = mw;
  s = sc;
}

// One CTA walks the groups [g_lo, g_hi) of the row(s) in index order from
// running sum c0 and returns the first entry at which the running sum of the
// sampler weights exceeds t (every thread gets it); if round-off leaves no
// crossing, the last entry of positive weight (-1 if none).  Thread j of a
// tile owns kGPT consecutive groups; a block scan routes t to one thread.
template <typename T, int MODE>
__device__ int block_walk(SweepShared &sh, const T *rowA, const T *rowB, int V, int g_lo, int g_hi,
                          int kind, const SampleParams &sp, float c0, float t) {
  constexpr int VW = Elem<T>::kPerVec;
  float base = c0;
  int lastpos = -1;
  if (threadIdx.x == 0) sh.bs.found = -1;
  for (int tb = g_lo; tb < g_hi; tb += kNT * kGPT) {
    const int gs = tb + (int)threadIdx.x * kGPT;
    float w[kGPT][VW];
    float s = 0.0f;
#pragma unroll
    for (int u = 0; u < kGPT; ++u) {
      const int g = gs + u;
      if (g < g_hi) {
        const uint4 za = load_group<T, true, true>(rowA, g, V);
        const uint4 zb = kind != kWBonus ? load_group<T, true, true>(rowB, g, V) : za;
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          w[u][e] = sample_weight(MODE, kind, sp, Elem<T>::get(za, e), Elem<T>::get(zb, e));
          s = __fadd_rn(s, w[u][e]);
          if (w[u][e] > 0.0f) lastpos = g * VW + e;
        }
      } else {
#pragma unroll
        for (int e = 0; e < VW; ++e) w[u][e] = 0.0f;
      }
    }
    float excl, incl, total;
    block_scan<kNT>(sh.bs, s, excl, incl, total);
    const float lo = __fadd_rn(base, excl), hi = __fadd_rn(base, incl);
    if (lo <= t && t < hi) {  // one thread at most: the intervals are disjoint
      float c = lo;
      int pick = -1, lastg = -1;
#pragma unroll
      for (int u = 0; u < kGPT; ++u)
#pragma unroll
        for (int e = 0; e < VW; ++e) {
          c = __fadd_rn(c, w[u][e]);
          if (w[u][e] > 0.0f) lastg = (gs + u) * VW + e;
          if (pick < 0 && c > t) pick = (gs + u) * VW + e;
        }
      sh.bs.found = pick >= 0 ? pick : lastg;
    }
    __syncthreads();
    const int f = sh.bs.found;
    __syncthreads();
    if (f >= 0) return f;
    base = __fadd_rn(base, total);
  }
  return block_max_index<kNT>(sh.bs, lastpos);
}

// Bonus token: the mass of chunk c of row K is s_c * exp(m_c - mA) / S_A (the
// target softmax summed over the chunk); block scans over the chunks in index
// order give the total and route u * total to one chunk, which the CTA walks.
template <typename T, int MODE>
__device__ int bonus_token(SweepShared &sh, const SweepArgs &a, int64_t p, const T *row,
                           const SampleParams &sp, float u) {
  const int C = a.chunks;
  const float4 *st = a.ws_chunk + p * C;
  auto mass = [&](int c) -> float {
    if (c >= C) return 0.0f;
    const float4 v = __ldcg(&st[c]);
    return v.x == -INFINITY ? 0.0f
                            : __fmul_rn(v.y, prob_from_offset(v.x, sp.nA));
  };
  float W = 0.0f;
  for (int c0 = 0; c0 < C; c0 += kNT) {
    float excl, incl, tot;
    block_scan<kNT>(sh.bs, mass(c0 + (int)threadIdx.x), excl, incl, tot);
    W = __fadd_rn(W, tot);
  }
  if (!(W > 0.0f)) return -1;
  float t = __fmul_rn(u, W);
  float base = 0.0f;
  int found = -1, lastpos = -1;
  if (threadIdx.x == 0) sh.bs.found = -1;
  for (int c0 = 0; c0 < C; c0 += kNT) {
    const int c = c0 + (int)threadIdx.x;
    const float m = mass(c);
    float excl, incl, tot;
    block_scan<kNT>(sh.bs, m, excl, incl, tot);
    const float l = __fadd_rn(base, excl), h = __fadd_rn(base, incl);
    if (c < C && l <= t && t < h) {
      sh.bs.found = c;
      sh.seg_lo = l;
    }
    if (m > 0.0f) lastpos = c;
    __syncthreads();
    found = sh.bs.found;
    __syncthreads();
    if (found >= 0) break;
    base = __fadd_rn(base, tot);
  }
  float lo = 0.0f;
  if (found >= 0) {
    lo = sh.seg_lo;
  } else {  // u * W not below the total (u >= 1): the last chunk with mass, its last entry
    found = block_max_index<kNT>(sh.bs, lastpos);
    t = INFINITY;
  }
  if (found < 0) return -1;
  const int g_lo = found * a.chunk_groups;
  const int g_hi = min(a.num_groups, g_lo + a.chunk_groups);
  return block_walk<T, MODE>(sh, row, row, a.V, g_lo, g_hi, kWBonus, sp, lo, t);
}

// Residual (or mixture) token of row pair n: segment masses over the whole
// row, the segment holding u * total, and a warp's walk of that segment.  A
// residual of zero mass (round-off only) falls back to p~.  The token is
// valid in warp 0.
template <typename T, int MODE>
__device__ int residual_token(SweepShared &sh, const SweepArgs &a, const T *rowA, const T *rowB,
                              int kind, const SampleParams &sp, float u) {
  const int G = a.num_groups, nseg = a.nseg;
  const int seg_groups = a.seg_tiles * kSweepSegGroups;
  float R = 0.0f;
  for (int attempt = 0;; ++attempt) {
    R = segment_masses<T, MODE, true, kSweepLaneGroups, kNT>(sh, rowA, rowB, a.V, 0, G,
                                                             seg_groups, nseg, kind, sp);
    if (R > 0.0f || kind != kWResidual || attempt == 1) break;
    kind = kWMixture;
  }
  if (!(R > 0.0f)) return -1;
  float t = __fmul_rn(u, R);
  float lo = 0.0f;
  const int s = find_segment<kNT>(sh, nseg, t, &lo);
  if ((threadIdx.x >> 5) != 0 || s < 0) return -1;
  const int sg_lo = s * seg_groups;
  const int sg_hi = min(G, sg_lo + seg_groups);
  return segment_walk<T, MODE, true, kSweepLaneGroups>(rowA, rowB, a.V, sg_lo, sg_hi, kind, sp, lo,
                                                       t);
}

// Finish sequence b once every position has published (whole CTA): warp 0
// runs the acceptance tests (the pages' loop: accept x_i iff
// u_i < min(1, p~(x_i)/q(x_i)), stop at the first rejection) and writes the
// accepted prefix; then the CTA draws the token at index n.
template <typename T, int MODE>
__device__ void finish_sequence(SweepShared &sh, const SweepArgs &a, int64_t b) {
  const int K = a.K, V = a.V;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const T *tgt = static_cast<const T *>(a.target);
  const T *dft = static_cast<const T *>(a.draft);
  __threadfence();
  if (warp == 0) {
    const float lam = a.lam[b];
    const bool lam_ok = lambda_valid(lam);
    bool lane_ok = true, lane_failed = false;
    int n = K;
    for (int i0 = 0; i0 < K; i0 += 32) {
      const int j = i0 + lane;
      bool rejected = false;
      if (j < K) {
        const int x = a.tokens[b * K + j];
        const bool tok_ok = x >= 0 && x < V;
        const float4 st4 = __ldcg(&a.ws_stats[b * (K + 1) + j]);
        const bool st_ok = st4.y >= 0.0f;
        lane_ok = lane_ok && tok_ok;
        lane_failed = lane_failed || !st_ok;
        if (tok_ok && lam_ok && st_ok) {
          const PosStats st{st4.x, st4.y, st4.z, st4.w};
          const float zt_x = Elem<T>::load(tgt + (b * (K + 1) + j) * (int64_t)V + x);
          const float zq_x = Elem<T>::load(dft + (b * K + j) * (int64_t)V + x);
          float px = 0.0f, qx = 0.0f;
          const float ratio =
              accept_ratio(MODE, st, zt_x, zq_x, lam, a.dbg_ptilde ? &px : nullptr, &qx);
          rejected = !accept_test(a.u_accept[b * K + j], ratio);
          if (a.dbg_ptilde) a.dbg_ptilde[b * K + j] = px;
          if (a.dbg_q) a.dbg_q[b * K + j] = qx;
        }
      }
      const unsigned rej = __ballot_sync(0xffffffffu, rejected);
      if (rej != 0u && n == K) n = i0 + __ffs(rej) - 1;
    }
    if (lane == 0 && !(__ldcg(&a.ws_stats[b * (K + 1) + K]).y >= 0.0f)) lane_failed = true;
    const bool all_tok = __all_sync(0xffffffffu, lane_ok);  // every lane votes
    const bool failed = __any_sync(0xffffffffu, lane_failed);
    const bool valid = lam_ok && all_tok && !failed;
    if (a.dbg_lse) {
      for (int j = lane; j <= K; j += 32) {
        const float4 st4 = __ldcg(&a.ws_stats[b * (K + 1) + j]);
        a.dbg_lse[(b * (K + 1) + j) * 2 + 0] = st4.x + lg2(st4.y) * kLn2;
        a.dbg_lse[(b * (K + 1) + j) * 2 + 1] = j < K ? st4.z + lg2(st4.w) * kLn2 : 0.0f;
      }
    }
    for (int j = lane; j <= K; j += 32) {
      int out = -1;
      if (valid && j < n) out = a.tokens[b * K + j];
      if (!valid || j != n) a.out_tokens[b * (K + 1) + j] = out;
    }
    if (lane == 0) {
      a.out_n[b] = failed ? -2 : (valid ? n : -1);
      SweepBroadcast bc;
      bc.n = valid ? n : -1;
      bc.u = a.u_resample[b];
      const float4 st4 = __ldcg(&a.ws_stats[b * (K + 1) + (valid ? n : 0)]);
      bc.sp = make_sample_params_rn(st4.x, st4.y, st4.z, st4.w, lam);
      if (n == K)
        bc.kind = kWBonus;
      else if (MODE == kProbMix && !(lam < 1.0f))
        bc.kind = kWMixture;  // p~ = q: the residual is identically zero
      else
        bc.kind = kWResidual;
      sh.bc = bc;
    }
  }
  __syncthreads();
  const SweepBroadcast bc = sh.bc;
  if (bc.n < 0) return;
  const int64_t pn = b * (K + 1) + bc.n;
  const T *rowA = tgt + pn * (int64_t)V;
  const T *rowB = dft + (b * K + (bc.n < K ? bc.n : 0)) * (int64_t)V;
  const int tok = bc.kind == kWBonus ? bonus_token<T, MODE>(sh, a, pn, rowA, bc.sp, bc.u)
                                     : residual_token<T, MODE>(sh, a, rowA, rowB, bc.kind, bc.sp,
                                                               bc.u);
  if (threadIdx.x == 0) a.out_tokens[pn] = tok;
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kNT, 2) sweep_kernel(SweepArgs a) {
  constexpr int VW = Elem<T>::kPerVec;
  extern __shared__ __align__(128) unsigned char stage_mem[];
  __shared__ __align__(8) uint64_t full[kNS];
  __shared__ SweepShared sh;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K, G = a.num_groups, CG = a.chunk_groups, C = a.chunks;
  const int CH = CG * 16;  // bytes of one row's chunk
  const char *tgt = static_cast<const char *>(a.target);
  const char *dft = static_cast<const char *>(a.draft);
  const int64_t grid = gridDim.x;

  // Start the bulk copies of item number k of this CTA into stage k % kNS.
  auto issue = [&](int64_t k) {
    const int64_t j = (int64_t)blockIdx.x + k * grid;
    if (j >= a.items) return;
    const int64_t p = j / C;
    const int c = (int)(j - p * C);
    const int64_t b = p / (K + 1);
    const int i = (int)(p - b * (K + 1));
    const int g_lo = c * CG;
    const uint32_t bytes = (uint32_t)min(CG, G - g_lo) * 16u;
    const int s = (int)(k % kNS);
    unsigned char *dst = stage_mem + (size_t)s * 2 * CH;
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");  // earlier reads of the stage
    mbar_arrive_expect_tx(&full[s], i < K ? 2 * bytes : bytes);
    tma_load_1d(dst, tgt + (p * (int64_t)G + g_lo) * 16, bytes, &full[s]);
    if (i < K) tma_load_1d(dst + CH, dft + ((b * K + i) * (int64_t)G + g_lo) * 16, bytes, &full[s]);
  };

  if (tid == 0) {
    for (int s = 0; s < kNS; ++s) mbar_init(&full[s], 1);
    mbar_fence_init();
    sh.finish = -1;
  }
  __syncthreads();
  int64_t next_issue = 0;  // thread 0's count of items started
  if (tid == 0)
    for (; next_issue < kNS; ++next_issue) issue(next_issue);

  bool dead = false;
  int64_t k_dead = -1;
  for (int64_t k = 0;; ++k) {
    const int64_t j = (int64_t)blockIdx.x + k * grid;
    if (j >= a.items) break;
    const int64_t p = j / C;
    const int c = (int)(j - p * C);
    const int64_t b = p / (K + 1);
    const int i = (int)(p - b * (K + 1));
    const bool pair = i < K;
    const int ng = min(CG, G - c * CG);
    const float lam = (MODE == kLogitMix && pair) ? a.lam[b] : 0.0f;
    const int s = (int)(k % kNS);
    const uint32_t parity = (uint32_t)((k / kNS) & 1);
    const bool got = __syncthreads_and(dead ? 0 : (mbar_wait(&full[s], parity) ? 1 : 0)) != 0;
    if (!got && !dead) {
      dead = true;
      k_dead = k;
    }

    // ------------------------------------------------ chunk statistics
    float mA = -INFINITY, sA = 0.0f, mB = -INFINITY, sB = 0.0f;
    if (got) {
      const uint4 *Av = reinterpret_cast<const uint4 *>(stage_mem + (size_t)s * 2 * CH);
      const uint4 *Bv = Av + CG;
      for (int q0 = 0; q0 < ng; q0 += kNT * kGPT) {
        uint4 za[kGPT], zb[kGPT];
#pragma unroll
        for (int u = 0; u < kGPT; ++u) {
          const int g = q0 + u * kNT + tid;
          za[u] = g < ng ? Av[g] : neg_inf_group<T>();
          zb[u] = (pair && g < ng) ? Bv[g] : neg_inf_group<T>();
        }
        // A-row value: the target logit, or in logit mode the mixed logit
        auto a_val = [&](int u, int e) -> float {
          const float zt = Elem<T>::get(za[u], e);
          if (MODE == kLogitMix && pair) {
            const float zq = Elem<T>::get(zb[u], e);
            return zq == -INFINITY ? -INFINITY : mix_logit(zt, zq, lam);
          }
          return zt;
        };
        float bmA = -INFINITY, bmB = -INFINITY;
#pragma unroll
        for (int u = 0; u < kGPT; ++u)
#pragma unroll
          for (int e = 0; e < VW; ++e) {
            bmA = fmaxf(bmA, a_val(u, e));
            bmB = fmaxf(bmB, Elem<T>::get(zb[u], e));
          }
        if (bmA > mA) {
          sA = __fmul_rn(sA, exp_shifted(mA, bmA));
          mA = bmA;
        }
        if (bmB > mB) {
          sB = __fmul_rn(sB, exp_shifted(mB, bmB));
          mB = bmB;
        }
        if (mA != -INFINITY) {
#pragma unroll
          for (int u = 0; u < kGPT; ++u)
#pragma unroll
            for (int e = 0; e < VW; ++e) sA = __fadd_rn(sA, exp_shifted(a_val(u, e), mA));
        }
        if (mB != -INFINITY) {
#pragma unroll
          for (int u = 0; u < kGPT; ++u)
#pragma unroll
            for (int e = 0; e < VW; ++e) sB = __fadd_rn(sB, exp_shifted(Elem<T>::get(zb[u], e), mB));
        }
      }
    }
    warp_stats(mA, sA);
    warp_stats(mB, sB);
    if (lane == 0) sh.wpart[warp] = got ? make_float4(mA, sA, mB, sB) : failed_stats();
    __syncthreads();  // stage s is consumed; warp partials are visible
    if (tid == 0 && !dead) {
      issue(next_issue);
      ++next_issue;
    }

    // ------------------------------------------------ publish
    if (warp == 0) {
      const float4 v = lane < kNW ? sh.wpart[lane] : make_float4(-INFINITY, 0.0f, -INFINITY, 0.0f);
      const bool bad = __any_sync(0xffffffffu, v.y < 0.0f);
      float cmA = v.x, csA = v.y, cmB = v.z, csB = v.w;
      warp_stats(cmA, csA);
      warp_stats(cmB, csB);
      int row_done = 0;
      if (lane == 0) {
        a.ws_chunk[j] = bad ? failed_stats() : make_float4(cmA, csA, cmB, csB);
        __threadfence();
        const unsigned prev = atomicAdd(&a.row_count[p], 1u);
        row_done = prev == (unsigned)(C - 1);
        if (row_done) a.row_count[p] = 0;  // every chunk has arrived: leave it zero
      }
      row_done = __shfl_sync(0xffffffffu, row_done, 0);
      if (row_done) {
        __threadfence();
        // the row's statistics: chunk statistics merged in chunk order
        float rmA = -INFINITY, rsA = 0.0f, rmB = -INFINITY, rsB = 0.0f;
        bool rbad = false;
        for (int cc = lane; cc < C; cc += 32) {
          const float4 w = __ldcg(&a.ws_chunk[p * C + cc]);
          if (w.y < 0.0f) {
            rbad = true;
          } else {
            merge_stats(rmA, rsA, w.x, w.y);
            merge_stats(rmB, rsB, w.z, w.w);
          }
        }
        rbad = __any_sync(0xffffffffu, rbad);
        warp_stats(rmA, rsA);
        warp_stats(rmB, rsB);
        if (lane == 0) {
          a.ws_stats[p] = rbad ? failed_stats() : make_float4(rmA, rsA, rmB, rsB);
          __threadfence();
          const unsigned prev = atomicAdd(&a.seq_count[b], 1u);
          if (prev == (unsigned)K) {
            a.seq_count[b] = 0;
            sh.finish = b;
          }
        }
      }
    }
    __syncthreads();
    const long long fin = sh.finish;
    if (fin >= 0) {  // CTA-uniform
      finish_sequence<T, MODE>(sh, a, fin);
      __syncthreads();
      if (tid == 0) sh.finish = -1;
      __syncthreads();
    }
  }

  // After a failed wait, copies started earlier may still be landing in this
  // CTA's shared memory: wait for them (with the same time limit) before exiting.
  if (dead && tid == 0)
    for (int64_t k2 = k_dead; k2 < next_issue; ++k2)
      (void)mbar_wait(&full[k2 % kNS], (uint32_t)((k2 / kNS) & 1));
}

template <typename T, int MODE>
cudaError_t launch_one(const SweepArgs &a, int64_t grid, int smem, cudaStream_t stream) {
  sweep_kernel<T, MODE><<<(unsigned)grid, kNT, (size_t)smem, stream>>>(a);
  return cudaGetLastError();
}

template <typename T, int MODE>
cudaError_t prepare_one(int max_smem) {
  return cudaFuncSetAttribute(sweep_kernel<T, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              max_smem);
}

template <typename T, int MODE>
int per_sm(int smem) {
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sweep_kernel<T, MODE>, kNT, (size_t)smem) !=
      cudaSuccess) {
    (void)cudaGetLastError();
    return 1;
  }
  return n > 0 ? n : 1;
}

}  // namespace

cudaError_t sweep_prepare(int max_smem_bytes) {
  cudaError_t e = cudaSuccess, r;
  if ((r = prepare_one<float, kProbMix>(max_smem_bytes)) != cudaSuccess) e = r;
  if ((r = prepare_one<float, kLogitMix>(max_smem_bytes)) != cudaSuccess) e = r;
  if ((r = prepare_one<uint16_t, kProbMix>(max_smem_bytes)) != cudaSuccess) e = r;
  if ((r = prepare_one<uint16_t, kLogitMix>(max_smem_bytes)) != cudaSuccess) e = r;
  return e;
}

int sweep_blocks_per_sm(int dtype_bf16, int mode, int smem_bytes) {
  if (dtype_bf16)
    return mode == kProbMix ? per_sm<uint16_t, kProbMix>(smem_bytes)
                            : per_sm<uint16_t, kLogitMix>(smem_bytes);
  return mode == kProbMix ? per_sm<float, kProbMix>(smem_bytes)
                          : per_sm<float, kLogitMix>(smem_bytes);
}

cudaError_t sweep_launch(const SweepArgs &a, int dtype_bf16, int mode, int64_t grid, int smem_bytes,
                         cudaStream_t stream) {
  if (dtype_bf16)
    return mode == kProbMix ? launch_one<uint16_t, kProbMix>(a, grid, smem_bytes, stream)
                            : launch_one<uint16_t, kLogitMix>(a, grid, smem_bytes, stream);
  return mode == kProbMix ? launch_one<float, kProbMix>(a, grid, smem_bytes, stream)
                          : launch_one<float, kLogitMix>(a, grid, smem_bytes, stream);
}

}  // namespace specv
