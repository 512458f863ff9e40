// specv_tile_tma.cu -- the small-vocabulary kernel with TMA-staged tiles.
//
// For short rows (V up to a few hundred entries, 16-byte aligned) a CTA owns
// whole sequences.  The target rows [s][K+1][V] and draft rows [s][K][V] of a
// tile of sequences are contiguous in HBM, so one 1-D TMA bulk copy each
// brings a tile into shared memory; two tile buffers alternate, so the next
// tile is in flight while this one is processed.  Per tile:
//   stage A: one thread per row computes (max, sum-exp) of the p~ source
//            row (target, or mixed in logit mode) or of the draft row in one
//            pass of 16-byte shared-memory reads; the walk starts at a
//            per-position offset (the same for the target and draft row of a
//            position, so identical rows give identical statistics) that
//            spreads simultaneous reads over the banks;
//   stage B: a group of kLanes lanes per sequence (kLanes = 4; eight
//            sequences per warp in lockstep): lanes 0..K-1 of the group test
//            positions 0..K-1 (in rounds of kLanes), a ballot gives the first
//            rejection, and the inverse CDF is a segmented scan across the
//            group, each lane owning a contiguous run of 16-byte groups of
//            the row.  Measured at B = 10^6, K = 4, V = 32 fp32 against 8
//            lanes per sequence: probability 239.2 vs 252.3 us, logit 281.7
//            vs 297.5 us, greedy 228.7 vs 231.0 us (the per-lane fixed work
//            of a sequence -- sampler parameters, scan, ballots -- is done by
//            half as many lanes).
// The per-sequence scalars (tokens, uniforms, lambda) are loaded into
// registers before stage A so their latency overlaps it.  No scratch memory.
#include <climits>

#include "specv_block.cuh"
#include "specv_device.cuh"
#include "specv_internal.h"

namespace specv {

namespace {

constexpr int kNT = kTmaTileThreads;
constexpr int kLanes = kTmaTileLanes;          // lanes per sequence in stage B

template <typename T>
__device__ __forceinline__ float sval(const T *p);
template <>
__device__ __forceinline__ float sval<float>(const float *p) {
  return *p;
}
template <>
__device__ __forceinline__ float sval<uint16_t>(const uint16_t *p) {
  return bf16_bits_to_float(*p);
}

// (max, sum-exp) of one staged row (or the mixed row of a pair) of G groups,
// one pass from group `rot` onwards: a per-group max, a rescale when it
// grows, and 2^(z*log2e - m*log2e) with one FFMA per entry (the rounding of
// m*log2e is a common factor of the row and cancels in every probability).
template <typename T, int MODE>
__device__ __forceinline__ float2 row_stats(const uint4 *ra, const uint4 *rb, int G, int rot,
                                            bool mixed, float lam) {
  constexpr int VW = Elem<T>::kPerVec;
  // lambda = 0 or 1: the mixed row is the target or the draft row itself
  if (MODE == kLogitMix && mixed && !(lam > 0.0f && lam < 1.0f))
    return row_stats<T, kProbMix>(lam == 0.0f ? ra : rb, rb, G, rot, false, 0.0f);
  // mL starts finite so that masked (-inf) entries before the first finite
  // one add 2^(-inf) = 0 rather than NaN; s is still 0 when m first grows, and
  // the rescale exponent is clamped at 0 so that 0 * 2^x stays 0
  float m = -INFINITY, mL = 0.0f, s = 0.0f;
  int g = rot;
  for (int k = 0; k < G; ++k) {
    float z[VW];
    const uint4 va = ra[g];
    if (MODE == kLogitMix && mixed) {
      const uint4 vb = rb[g];
#pragma unroll
      for (int e = 0; e < VW; ++e)
        z[e] = mix_logit_interior(Elem<T>::get(va, e), Elem<T>::get(vb, e), lam);
    } else {
#pragma unroll
      for (int e = 0; e < VW; ++e) z[e] = Elem<T>::get(va, e);
    }
    float bm = z[0];
#pragma unroll
    for (int e = 1; e < VW; ++e) bm = fmaxf(bm, z[e]);
    if (bm > m) {
      const float nmL = __fmul_rn(bm, kLog2e);
      s = __fmul_rn(s, ex2(fminf(__fsub_rn(mL, nmL), 0.0f)));
      m = bm;
      mL = nmL;
    }
#pragma unroll
    for (int e = 0; e < VW; ++e) s = __fadd_rn(s, ex2(__fmaf_rn(z[e], kLog2e, -mL)));
    g = (g + 1 == G) ? 0 : g + 1;
  }
  return make_float2(m, s);
}

// Greedy: (max, index) of the mixed logits w of one staged row (target row
// alone at the bonus position), the first maximum in index order; the index
// is returned in the bits of the second component.
template <typename T>
__device__ __forceinline__ float2 row_argmax(const uint4 *ra, const uint4 *rb, int G, int rot,
                                             bool mixed, float lam) {
  constexpr int VW = Elem<T>::kPerVec;
  float best = -INFINITY;
  int bidx = INT_MAX;
  int g = rot;
  for (int k = 0; k < G; ++k) {
    const uint4 va = ra[g];
    const uint4 vb = mixed ? rb[g] : va;
#pragma unroll
    for (int e = 0; e < VW; ++e) {
      const float zt = Elem<T>::get(va, e);
      const float w = mixed ? greedy_score(zt, Elem<T>::get(vb, e), lam) : zt;
      argmax_merge(best, bidx, w, g * VW + e);
    }
    g = (g + 1 == G) ? 0 : g + 1;
  }
  return make_float2(best, __int_as_float(bidx));
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kNT) tile_tma_kernel(TileArgs a) {
  constexpr bool GREEDY = MODE == kGreedy;  // argmax per row; no draft-row tasks, no sampling
  constexpr int VW = Elem<T>::kPerVec;
  // stage-B groups per lane whose weights are kept in registers (two fp32
  // groups fit the 64 registers of four CTAs per SM; two bf16 groups do not)
  constexpr int kCacheC = sizeof(T) == 4 ? 2 : 1;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
  const int K = a.K, V = a.V, TS = a.tile_seqs;
  const int G = V / VW;                      // 16-byte groups per row
  const int C = (G + kLanes - 1) / kLanes;   // groups per lane in stage B
  const int stage_bytes = a.smem_target_bytes + a.smem_draft_bytes;
  unsigned char *stage0 = smem + 128;
  float *st_s = reinterpret_cast<float *>(stage0 + 2 * stage_bytes);  // [TS][K+1][4]
  const T *tgt = static_cast<const T *>(a.target);
  const T *dft = static_cast<const T *>(a.draft);
  const int lane = threadIdx.x & 31;
  const int gl = lane % kLanes;                         // lane within the sequence group
  const int gsh = lane - gl;                            // first lane of the group
  const unsigned gmask = ((1u << kLanes) - 1u) << gsh;  // the group's lanes
  const int sq = threadIdx.x / kLanes;                  // stage-B sequence of this thread

  if (threadIdx.x == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    mbar_fence_init();
  }
  __syncthreads();
  auto issue = [&](int64_t tile, int stage) {
    const int64_t b0 = tile * TS;
    const int64_t nseq = (a.B - b0) < TS ? (a.B - b0) : TS;
    const uint32_t bt = (uint32_t)(nseq * (K + 1) * V * (int64_t)sizeof(T));
    const uint32_t bd = (uint32_t)(nseq * K * V * (int64_t)sizeof(T));
    unsigned char *dst = stage0 + stage * stage_bytes;
    mbar_arrive_expect_tx(&bar[stage], bt + bd);
    tma_load_1d(dst, tgt + b0 * (K + 1) * (int64_t)V, bt, &bar[stage]);
    tma_load_1d(dst + a.smem_target_bytes, dft + b0 * K * (int64_t)V, bd, &bar[stage]);
  };
  const int64_t first = blockIdx.x;
  if (threadIdx.x == 0) {
    if (first < a.num_tiles) issue(first, 0);
    if (first + gridDim.x < a.num_tiles) issue(first + gridDim.x, 1);
  }

  // This thread's first stage-A task of a full tile (the same in every full
  // tile): computed once, so full tiles need no integer division per row.
  const int fA = TS * (K + 1), fB = GREEDY ? 0 : TS * K;
  const bool has_task = (int)threadIdx.x < fA + fB;
  int t_pos = 0, t_rd = 0, t_rot = 0, t_s = 0;
  bool t_isA = false, t_mixed = false;
  if (has_task) {
    int s_, i_;
    t_isA = (int)threadIdx.x < fA;
    if (t_isA) {
      t_pos = threadIdx.x;
      s_ = t_pos / (K + 1);
      i_ = t_pos - s_ * (K + 1);
    } else {
      const int t2 = threadIdx.x - fA;
      s_ = t2 / K;
      i_ = t2 - s_ * K;
      t_pos = s_ * (K + 1) + i_;
    }
    t_s = s_;
    t_mixed = t_isA && i_ < K;
    t_rd = (s_ * K + (i_ < K ? i_ : 0)) * V;
    t_rot = t_pos % G;
  }

  int k = 0;
  bool dead = false;  // a copy of this CTA timed out: no more waits, report -2
  for (int64_t tile = first; tile < a.num_tiles; tile += gridDim.x, ++k) {
    const int stage = k & 1;
    const uint32_t parity = (uint32_t)((k >> 1) & 1);
    const int64_t b0 = tile * TS;
    const int nseq = (int)((a.B - b0) < TS ? (a.B - b0) : TS);
    const T *st_t = reinterpret_cast<const T *>(stage0 + stage * stage_bytes);
    const T *st_d = reinterpret_cast<const T *>(stage0 + stage * stage_bytes + a.smem_target_bytes);
    const bool mine = sq < nseq;  // this thread's group has a sequence in stage B
    const int64_t b = b0 + (mine ? sq : 0);

    // prefetch this group's per-sequence scalars (lane j < K of the group: x_j, u_j)
    float p_lam = 0.0f, p_ur = 0.0f, p_ua = 0.0f;
    int p_tok = 0;
    if (mine) {
      p_lam = a.lam[b];
      p_ur = a.u_resample[b];
      if (gl < K) {
        p_tok = a.tokens[b * K + gl];
        p_ua = a.u_accept[b * K + gl];
      }
    }

    const bool ok = __syncthreads_and(dead ? 0 : (int)mbar_wait(&bar[stage], parity)) != 0;
    dead = !ok;

    // stage A: one thread per row; A-rows (p~ source) of all positions first,
    // then the draft rows
    const int nA = ok ? nseq * (K + 1) : 0, nB = (ok && !GREEDY) ? nseq * K : 0;
    const bool full = nseq == TS;
    if (ok && full && has_task) {
      const uint4 *rt = reinterpret_cast<const uint4 *>(st_t + (int64_t)t_pos * V);
      const uint4 *rd = reinterpret_cast<const uint4 *>(st_d + t_rd);
      float2 r;
      if constexpr (GREEDY)
        r = row_argmax<T>(rt, rd, G, t_rot, t_mixed, a.lam[b0 + t_s]);
      else if (t_isA)
        r = row_stats<T, MODE>(rt, rd, G, t_rot, t_mixed, a.lam[b0 + t_s]);
      else
        r = row_stats<T, kProbMix>(rd, rd, G, t_rot, false, 0.0f);
      st_s[t_pos * 4 + (t_isA ? 0 : 2)] = r.x;
      st_s[t_pos * 4 + (t_isA ? 1 : 3)] = r.y;
    }
    // remaining tasks (several per thread, or the last, partial tile)
    for (int task = full ? threadIdx.x + kNT : threadIdx.x; task < nA + nB; task += kNT) {
      int pos, s, i;
      const bool isA = task < nA;
      if (isA) {
        pos = task;
        s = pos / (K + 1);
        i = pos - s * (K + 1);
      } else {
        const int t2 = task - nA;
        s = t2 / K;
        i = t2 - s * K;
        pos = s * (K + 1) + i;
      }
      const int rot = pos % G;
      const uint4 *rt = reinterpret_cast<const uint4 *>(st_t + (int64_t)pos * V);
      const uint4 *rd = reinterpret_cast<const uint4 *>(st_d + ((int64_t)s * K + (i < K ? i : 0)) * V);
      float2 r;
      if constexpr (GREEDY)
        r = row_argmax<T>(rt, rd, G, rot, i < K, a.lam[b0 + s]);
      else if (isA)
        r = row_stats<T, MODE>(rt, rd, G, rot, i < K, a.lam[b0 + s]);
      else
        r = row_stats<T, kProbMix>(rd, rd, G, rot, false, 0.0f);
      st_s[pos * 4 + (isA ? 0 : 2)] = r.x;
      st_s[pos * 4 + (isA ? 1 : 3)] = r.y;
    }
    __syncthreads();

    // stage B: kLanes lanes per sequence (all lanes of a warp stay converged;
    // groups without a sequence compute on placeholders and write nothing)
    const bool warp_busy = __any_sync(0xffffffffu, mine);  // warp-uniform
    if (!warp_busy) {
      // no sequence of this tile in this warp
    } else if (!ok) {
      if (mine) {
        for (int j = gl; j <= K; j += kLanes) a.out_tokens[b * (K + 1) + j] = -1;
        if (gl == 0) a.out_n[b] = -2;
      }
    } else if constexpr (GREEDY) {
      // accept while x_j is the argmax of row j; emit the argmax at the first
      // mismatch (or of row K when every draft matches)
      const int sl = mine ? sq : 0;
      const bool lam_ok = lambda_valid(p_lam);
      bool lane_ok = true;
      int n = K;
      for (int i0 = 0; i0 < K; i0 += kLanes) {
        const int j = i0 + gl;
        bool rejected = false;
        if (j < K) {
          const int x = i0 == 0 ? p_tok : a.tokens[b * K + j];
          const bool tok_ok = x >= 0 && x < V;
          lane_ok = lane_ok && tok_ok;
          if (tok_ok && lam_ok) rejected = __float_as_int(st_s[(sl * (K + 1) + j) * 4 + 1]) != x;
        }
        const unsigned rej = (__ballot_sync(0xffffffffu, rejected) & gmask) >> gsh;
        if (rej != 0u && n == K) n = i0 + __ffs(rej) - 1;
      }
      const unsigned bad_tok = __ballot_sync(0xffffffffu, !lane_ok) & gmask;
      const bool valid = lam_ok && bad_tok == 0u;
      if (mine) {
        for (int j = gl; j <= K; j += kLanes) {
          int out = -1;
          if (valid && j < n) out = j == gl ? p_tok : a.tokens[b * K + j];
          if (valid && j == n) out = __float_as_int(st_s[(sl * (K + 1) + n) * 4 + 1]);
          a.out_tokens[b * (K + 1) + j] = out;
        }
        if (gl == 0) a.out_n[b] = valid ? n : -1;
      }
    } else {
      const int sl = mine ? sq : 0;  // staged sequence slot (a valid one for idle groups)
      const float lam = p_lam;
      const bool lam_ok = lambda_valid(lam);
      bool lane_ok = true;
      int n = K;
      for (int i0 = 0; i0 < K; i0 += kLanes) {
        const int j = i0 + gl;
        bool rejected = false;
        if (j < K) {
          const int x = i0 == 0 ? p_tok : a.tokens[b * K + j];
          const float u = i0 == 0 ? p_ua : a.u_accept[b * K + j];
          const bool tok_ok = x >= 0 && x < V;
          lane_ok = lane_ok && tok_ok;
          if (tok_ok && lam_ok) {
            const int pos = sl * (K + 1) + j;
            const float4 st4 = reinterpret_cast<const float4 *>(st_s)[pos];
            const PosStats st{st4.x, st4.y, st4.z, st4.w};
            const float zt_x = sval<T>(st_t + (int64_t)pos * V + x);
            const float zq_x = sval<T>(st_d + ((int64_t)sl * K + j) * V + x);
            float px = 0.0f, qx = 0.0f;
            const bool dbg = mine && a.dbg_ptilde != nullptr;
            const float ratio = accept_ratio(MODE, st, zt_x, zq_x, lam, dbg ? &px : nullptr, &qx);
            rejected = !accept_test(u, ratio);
            if (dbg) {
              a.dbg_ptilde[b * K + j] = px;
              a.dbg_q[b * K + j] = qx;
            }
          }
        }
        const unsigned rej = (__ballot_sync(0xffffffffu, rejected) & gmask) >> gsh;
        if (rej != 0u && n == K) n = i0 + __ffs(rej) - 1;
      }
      // the ballot runs on every lane: groups differ in lam_ok (no short-circuit)
      const unsigned bad_tok = __ballot_sync(0xffffffffu, !lane_ok) & gmask;
      const bool valid = lam_ok && bad_tok == 0u;
      if (mine && a.dbg_lse) {
        for (int j = gl; j <= K; j += kLanes) {
          const int pos = sl * (K + 1) + j;
          a.dbg_lse[(b * (K + 1) + j) * 2 + 0] = st_s[pos * 4 + 0] + lg2(st_s[pos * 4 + 1]) * kLn2;
          a.dbg_lse[(b * (K + 1) + j) * 2 + 1] =
              j < K ? st_s[pos * 4 + 2] + lg2(st_s[pos * 4 + 3]) * kLn2 : 0.0f;
        }
      }
      if (mine) {
        for (int j = gl; j <= K; j += kLanes) {
          int out = -1;
          if (valid && j < n) out = j == gl ? p_tok : a.tokens[b * K + j];  // lane j prefetched x_j
          if (!valid || j != n) a.out_tokens[b * (K + 1) + j] = out;
        }
        if (gl == 0) a.out_n[b] = valid ? n : -1;
      }
      // sampling: lane gl owns groups [gl*C, gl*C + C) of the row (pair) at n
      const int nn = valid ? n : 0;
      const int pos = sl * (K + 1) + nn;
      const float4 st4 = reinterpret_cast<const float4 *>(st_s)[pos];
      const SampleParams sp = make_sample_params(st4.x, st4.y, st4.z, st4.w, lam);
      int kind = (nn == K) ? kWBonus
                           : (!(lam < 1.0f) ? kWMixture : kWResidual);
      const uint4 *ra = reinterpret_cast<const uint4 *>(st_t + (int64_t)pos * V);
      const uint4 *rb = reinterpret_cast<const uint4 *>(st_d + ((int64_t)sl * K + (nn < K ? nn : 0)) * V);
      int tok = -1;
      // weights of the lane's first kCacheC groups, kept in registers for the
      // owner's walk (short rows: every group of the lane)
      float wc[kCacheC][VW];
      for (int attempt = 0; attempt < 2; ++attempt) {
        float mysum = 0.0f;
        int mylast = -1;
#pragma unroll
        for (int c = 0; c < kCacheC; ++c) {
          const int g = gl * C + c;
          if (c < C && g < G) {
            const uint4 za = ra[g];
            const uint4 zb = kind != kWBonus ? rb[g] : za;
#pragma unroll
            for (int e = 0; e < VW; ++e) {
              const float w = sample_weight_sel(MODE, kind, sp, Elem<T>::get(za, e), Elem<T>::get(zb, e));
              wc[c][e] = w;
              mysum = __fadd_rn(mysum, w);
              if (w > 0.0f) mylast = g * VW + e;
            }
          }
        }
        for (int c = kCacheC; c < C; ++c) {
          const int g = gl * C + c;
          if (g < G) {
            const uint4 za = ra[g];
            const uint4 zb = kind != kWBonus ? rb[g] : za;
#pragma unroll
            for (int e = 0; e < VW; ++e) {
              const float w = sample_weight_sel(MODE, kind, sp, Elem<T>::get(za, e), Elem<T>::get(zb, e));
              mysum = __fadd_rn(mysum, w);
              if (w > 0.0f) mylast = g * VW + e;
            }
          }
        }
        // segmented inclusive scan of the lane sums over the group
        float incl = mysum;
#pragma unroll
        for (int off = 1; off < kLanes; off <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, incl, off, kLanes);
          if (gl >= off) incl = __fadd_rn(incl, y);
        }
        float excl = __shfl_up_sync(0xffffffffu, incl, 1, kLanes);
        if (gl == 0) excl = 0.0f;
        const float R = __shfl_sync(0xffffffffu, incl, kLanes - 1, kLanes);
        const bool retry = !(R > 0.0f) && kind == kWResidual;
        // Every ballot and shuffle below runs on all 32 lanes (the four groups
        // of a warp differ in R, retry and owner); results are selected after.
        const bool have = R > 0.0f;
        const float t = __fmul_rn(p_ur, R);
        const bool own = have && excl <= t && t < incl;  // at most one lane of a group
        int pick = -1;
        if (own) {  // walk this lane's entries in order (no warp collectives inside)
          float c0 = excl;
          int lastg = -1;
#pragma unroll
          for (int c = 0; c < kCacheC; ++c) {
            const int g = gl * C + c;
            if (c < C && g < G && pick < 0) {
#pragma unroll
              for (int e = 0; e < VW; ++e) {
                const float w = wc[c][e];
                c0 = __fadd_rn(c0, w);
                if (w > 0.0f) lastg = g * VW + e;
                if (pick < 0 && c0 > t) pick = g * VW + e;
              }
            }
          }
          for (int c = kCacheC; c < C && pick < 0; ++c) {
            const int g = gl * C + c;
            if (g < G) {
              const uint4 za = ra[g];
              const uint4 zb = kind != kWBonus ? rb[g] : za;
#pragma unroll
              for (int e = 0; e < VW; ++e) {
                const float w =
                    sample_weight_sel(MODE, kind, sp, Elem<T>::get(za, e), Elem<T>::get(zb, e));
                c0 = __fadd_rn(c0, w);
                if (w > 0.0f) lastg = g * VW + e;
                if (pick < 0 && c0 > t) pick = g * VW + e;
              }
            }
          }
          if (pick < 0) pick = lastg;
        }
        const unsigned owner = (__ballot_sync(0xffffffffu, own) & gmask) >> gsh;
        const int picked = __shfl_sync(0xffffffffu, pick, owner != 0u ? __ffs(owner) - 1 : 0, kLanes);
        int lastpos = mylast;  // u*R not below the total (round-off): the last entry with mass
#pragma unroll
        for (int off = kLanes / 2; off > 0; off >>= 1)
          lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, off, kLanes));
        if (!retry && have) tok = owner != 0u ? picked : lastpos;
        if (!__any_sync(0xffffffffu, retry)) break;
        if (retry) kind = kWMixture;  // zero residual mass (round-off only): p~ instead
      }
      if (mine && valid && gl == 0) a.out_tokens[b * (K + 1) + n] = tok;
    }
    __syncthreads();  // every thread is done with this stage's rows and stats
    if (threadIdx.x == 0 && !dead && tile + 2 * (int64_t)gridDim.x < a.num_tiles) {
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      issue(tile + 2 * (int64_t)gridDim.x, stage);
    }
  }
}

template <typename T, int MODE>
cudaError_t prep(int max_smem) {
  return cudaFuncSetAttribute(tile_tma_kernel<T, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              max_smem);
}

template <typename T, int MODE>
int occ(int smem) {
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, tile_tma_kernel<T, MODE>, kNT, smem) !=
      cudaSuccess)
    return 1;
  return nb > 0 ? nb : 1;
}

}  // namespace

cudaError_t tile_tma_prepare(int max_smem_bytes) {
  cudaError_t e = cudaSuccess, r;
  if ((r = prep<float, kProbMix>(max_smem_bytes)) != cudaSuccess) e = r;
  if ((r = prep<float, kLogitMix>(max_smem_bytes)) != cudaSuccess) e = r;
  if ((r = prep<uint16_t, kProbMix>(max_smem_bytes)) != cudaSuccess) e = r;
  if ((r = prep<uint16_t, kLogitMix>(max_smem_bytes)) != cudaSuccess) e = r;
  if ((r = prep<float, kGreedy>(max_smem_bytes)) != cudaSuccess) e = r;
  if ((r = prep<uint16_t, kGreedy>(max_smem_bytes)) != cudaSuccess) e = r;
  return e;
}

int tile_tma_blocks_per_sm(int dtype_bf16, int mode, int smem_bytes) {
  if (mode == kGreedy)
    return dtype_bf16 ? occ<uint16_t, kGreedy>(smem_bytes) : occ<float, kGreedy>(smem_bytes);
  if (dtype_bf16) return mode == kProbMix ? occ<uint16_t, kProbMix>(smem_bytes)
                                          : occ<uint16_t, kLogitMix>(smem_bytes);
  return mode == kProbMix ? occ<float, kProbMix>(smem_bytes) : occ<float, kLogitMix>(smem_bytes);
}

cudaError_t tile_tma_launch(const TileArgs &a, int dtype_bf16, int mode, int64_t grid,
                            int smem_bytes, cudaStream_t stream) {
  const dim3 g((unsigned)grid), blk(kNT);
  if (mode == kGreedy) {
    if (dtype_bf16)
      tile_tma_kernel<uint16_t, kGreedy><<<g, blk, smem_bytes, stream>>>(a);
    else
      tile_tma_kernel<float, kGreedy><<<g, blk, smem_bytes, stream>>>(a);
    return cudaGetLastError();
  }
  if (dtype_bf16) {
    if (mode == kProbMix)
      tile_tma_kernel<uint16_t, kProbMix><<<g, blk, smem_bytes, stream>>>(a);
    else
      tile_tma_kernel<uint16_t, kLogitMix><<<g, blk, smem_bytes, stream>>>(a);
  } else {
    if (mode == kProbMix)
      tile_tma_kernel<float, kProbMix><<<g, blk, smem_bytes, stream>>>(a);
    else
      tile_tma_kernel<float, kLogitMix><<<g, blk, smem_bytes, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace specv
