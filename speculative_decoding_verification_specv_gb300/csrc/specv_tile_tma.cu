// specv_tile_tma.cu -- the small-vocabulary kernel with TMA-staged tiles.
//
// For short rows (V up to a few hundred entries, 16-byte aligned) a CTA owns
// whole sequences.  The target rows [s][K+1][V] and draft rows [s][K][V] of a
// tile of sequences are contiguous in HBM, so one 1-D TMA bulk copy each
// brings a tile into shared memory; two tile buffers alternate, so the next
// tile is in flight while this one is processed.  Per tile:
//   stage A: one thread per row computes (max, sum-exp) of the p~ source
//            row (target, or mixed in logit mode) or of the draft row with
//            16-byte shared-memory reads; the walk over a row starts at a
//            per-position offset (the same for the target and draft row of a
//            position, so identical rows give identical statistics) that
//            spreads simultaneous reads over the banks;
//   stage B: one warp per sequence: lane j tests position j, a ballot gives
//            the first rejection, and the inverse CDF runs as a warp scan
//            (one pass when V <= 32: the scan total is the mass and the
//            crossing lane is the token).
// The per-sequence scalars (tokens, uniforms, lambda) are loaded into
// registers before stage A so their latency overlaps it.  No scratch memory.
#include "specv_block.cuh"
#include "specv_device.cuh"
#include "specv_internal.h"

namespace specv {

namespace {

constexpr int kNT = kTileThreads;
constexpr int kNW = kNT / 32;
constexpr int kSeqPerWarp = kTmaTileMaxSeqs / kNW;  // prefetched sequences per warp

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
// walked from group `rot` onwards.
template <typename T, int MODE>
__device__ __forceinline__ float2 row_stats(const uint4 *ra, const uint4 *rb, int G, int rot,
                                            bool mixed, float lam) {
  constexpr int VW = Elem<T>::kPerVec;
  float m = -INFINITY;
  for (int k = 0; k < G; ++k) {
    int g = k + rot;
    g = g >= G ? g - G : g;
    const uint4 va = ra[g];
    if (MODE == kLogitMix && mixed) {
      const uint4 vb = rb[g];
#pragma unroll
      for (int e = 0; e < VW; ++e)
        m = fmaxf(m, mix_logit(Elem<T>::get(va, e), Elem<T>::get(vb, e), lam));
    } else {
#pragma unroll
      for (int e = 0; e < VW; ++e) m = fmaxf(m, Elem<T>::get(va, e));
    }
  }
  float s = 0.0f;
  for (int k = 0; k < G; ++k) {
    int g = k + rot;
    g = g >= G ? g - G : g;
    const uint4 va = ra[g];
    if (MODE == kLogitMix && mixed) {
      const uint4 vb = rb[g];
#pragma unroll
      for (int e = 0; e < VW; ++e)
        s = __fadd_rn(s, exp_shifted(mix_logit(Elem<T>::get(va, e), Elem<T>::get(vb, e), lam), m));
    } else {
#pragma unroll
      for (int e = 0; e < VW; ++e) s = __fadd_rn(s, exp_shifted(Elem<T>::get(va, e), m));
    }
  }
  return make_float2(m, s);
}

__device__ __forceinline__ float warp_incl_scan(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v = __fadd_rn(v, y);
  }
  return v;
}

// Inverse CDF over one staged row (pair) by one warp, entries in index order
// in tiles of 32 (lane l takes entry v0 + l).  Returns the token, or -1 if the
// weights have no mass; *mass receives the total.  For V <= 32 the mass and
// the search are one scan; otherwise a mass scan precedes the search scan,
// both accumulating identically.
template <typename T, int MODE>
__device__ int warp_sample(const T *ra, const T *rb, int V, int kind, const SampleParams &sp,
                           float u, float *mass) {
  const int lane = threadIdx.x & 31;
  if (V <= 32) {
    float w = 0.0f;
    if (lane < V) w = sample_weight(MODE, kind, sp, sval<T>(ra + lane), kind != kWBonus ? sval<T>(rb + lane) : 0.0f);
    const float incl = warp_incl_scan(w);
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.0f;
    const float R = __shfl_sync(0xffffffffu, incl, 31);
    *mass = R;
    if (!(R > 0.0f)) return -1;
    const float t = __fmul_rn(u, R);
    const unsigned hit = __ballot_sync(0xffffffffu, lane < V && excl <= t && t < incl);
    if (hit) return __ffs(hit) - 1;
    const unsigned pos = __ballot_sync(0xffffffffu, w > 0.0f);
    return 31 - __clz(pos);  // u*R not below the total: the last entry with mass
  }
  float R = 0.0f;
  for (int v0 = 0; v0 < V; v0 += 32) {
    const int v = v0 + lane;
    float w = 0.0f;
    if (v < V) w = sample_weight(MODE, kind, sp, sval<T>(ra + v), kind != kWBonus ? sval<T>(rb + v) : 0.0f);
    R = __fadd_rn(R, __shfl_sync(0xffffffffu, warp_incl_scan(w), 31));
  }
  *mass = R;
  if (!(R > 0.0f)) return -1;
  const float t = __fmul_rn(u, R);
  float base = 0.0f;
  int lastpos = -1;
  for (int v0 = 0; v0 < V; v0 += 32) {
    const int v = v0 + lane;
    float w = 0.0f;
    if (v < V) w = sample_weight(MODE, kind, sp, sval<T>(ra + v), kind != kWBonus ? sval<T>(rb + v) : 0.0f);
    if (w > 0.0f) lastpos = v;
    const float incl = warp_incl_scan(w);
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.0f;
    const float lo = __fadd_rn(base, excl), hi = __fadd_rn(base, incl);
    const unsigned hit = __ballot_sync(0xffffffffu, v < V && lo <= t && t < hi);
    if (hit) return v0 + __ffs(hit) - 1;
    base = __fadd_rn(base, __shfl_sync(0xffffffffu, incl, 31));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, off));
  return lastpos;
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kNT) tile_tma_kernel(TileArgs a) {
  constexpr int VW = Elem<T>::kPerVec;
  extern __shared__ __align__(128) unsigned char smem[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(smem);
  const int K = a.K, V = a.V, TS = a.tile_seqs;
  const int G = V / VW;  // 16-byte groups per row
  const int stage_bytes = a.smem_target_bytes + a.smem_draft_bytes;
  unsigned char *stage0 = smem + 128;
  float *st_s = reinterpret_cast<float *>(stage0 + 2 * stage_bytes);  // [TS][K+1][4]
  const T *tgt = static_cast<const T *>(a.target);
  const T *dft = static_cast<const T *>(a.draft);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

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

  int k = 0;
  bool dead = false;  // a copy of this CTA timed out: no more waits, report -2
  for (int64_t tile = first; tile < a.num_tiles; tile += gridDim.x, ++k) {
    const int stage = k & 1;
    const uint32_t parity = (uint32_t)((k >> 1) & 1);
    const int64_t b0 = tile * TS;
    const int nseq = (int)((a.B - b0) < TS ? (a.B - b0) : TS);
    const T *st_t = reinterpret_cast<const T *>(stage0 + stage * stage_bytes);
    const T *st_d = reinterpret_cast<const T *>(stage0 + stage * stage_bytes + a.smem_target_bytes);

    // prefetch the per-sequence scalars of this warp's sequences
    float p_lam[kSeqPerWarp], p_ur[kSeqPerWarp], p_ua[kSeqPerWarp];
    int p_tok[kSeqPerWarp];
#pragma unroll
    for (int m = 0; m < kSeqPerWarp; ++m) {
      const int s = warp + m * kNW;
      p_lam[m] = p_ur[m] = p_ua[m] = 0.0f;
      p_tok[m] = 0;
      if (s < nseq) {
        const int64_t b = b0 + s;
        p_lam[m] = a.lam[b];
        p_ur[m] = a.u_resample[b];
        if (lane < K) {
          p_tok[m] = a.tokens[b * K + lane];
          p_ua[m] = a.u_accept[b * K + lane];
        }
      }
    }

    const bool ok = !dead && __syncthreads_and(mbar_wait(&bar[stage], parity)) != 0;
    dead = !ok;

    // stage A: one thread per row; A-rows (p~ source) of all positions first,
    // then the draft rows
    const int nA = ok ? nseq * (K + 1) : 0, nB = ok ? nseq * K : 0;
    for (int task = threadIdx.x; task < nA + nB; task += kNT) {
      int pos, s, i;
      bool isA = task < nA;
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
      const float lam = a.lam[b0 + s];
      float2 r;
      if (isA)
        r = row_stats<T, MODE>(rt, rd, G, rot, i < K, lam);
      else
        r = row_stats<T, kProbMix>(rd, rd, G, rot, false, lam);
      st_s[pos * 4 + (isA ? 0 : 2)] = r.x;
      st_s[pos * 4 + (isA ? 1 : 3)] = r.y;
    }
    __syncthreads();

    // stage B: one warp per sequence (unrolled: the prefetched scalars stay in registers)
#pragma unroll
    for (int m = 0; m < kSeqPerWarp; ++m) {
      const int s = warp + m * kNW;
      if (s >= nseq) break;
      const int64_t b = b0 + s;
      const float lam = p_lam[m];
      if (!ok) {  // a copy did not complete in time: report, skip
        for (int j = lane; j <= K; j += 32) a.out_tokens[b * (K + 1) + j] = -1;
        if (lane == 0) a.out_n[b] = -2;
        continue;
      }
      const bool lam_ok = lambda_valid(lam);
      bool lane_ok = true;
      int n = K;
      for (int i0 = 0; i0 < K; i0 += 32) {
        const int j = i0 + lane;
        bool rejected = false;
        if (j < K) {
          const int x = i0 == 0 ? p_tok[m] : a.tokens[b * K + j];
          const float u = i0 == 0 ? p_ua[m] : a.u_accept[b * K + j];
          const bool tok_ok = x >= 0 && x < V;
          lane_ok = lane_ok && tok_ok;
          if (tok_ok && lam_ok) {
            const int pos = s * (K + 1) + j;
            const PosStats st{st_s[pos * 4 + 0], st_s[pos * 4 + 1], st_s[pos * 4 + 2],
                              st_s[pos * 4 + 3]};
            const float zt_x = sval<T>(st_t + (int64_t)pos * V + x);
            const float zq_x = sval<T>(st_d + ((int64_t)s * K + j) * V + x);
            float px = 0.0f, qx = 0.0f;
            const float ratio =
                accept_ratio(MODE, st, zt_x, zq_x, lam, a.dbg_ptilde ? &px : nullptr, &qx);
            rejected = !accept_test(u, ratio);
            if (a.dbg_ptilde) {
              a.dbg_ptilde[b * K + j] = px;
              a.dbg_q[b * K + j] = qx;
            }
          }
        }
        const unsigned rej = __ballot_sync(0xffffffffu, rejected);
        if (rej != 0u && n == K) n = i0 + __ffs(rej) - 1;
      }
      const bool valid = lam_ok && __all_sync(0xffffffffu, lane_ok);
      if (a.dbg_lse) {
        for (int j = lane; j <= K; j += 32) {
          const int pos = s * (K + 1) + j;
          a.dbg_lse[(b * (K + 1) + j) * 2 + 0] = st_s[pos * 4 + 0] + lg2(st_s[pos * 4 + 1]) * kLn2;
          a.dbg_lse[(b * (K + 1) + j) * 2 + 1] =
              j < K ? st_s[pos * 4 + 2] + lg2(st_s[pos * 4 + 3]) * kLn2 : 0.0f;
        }
      }
      for (int j = lane; j <= K; j += 32) {
        int out = -1;
        if (valid && j < n) out = j == lane ? p_tok[m] : a.tokens[b * K + j];  // lane j prefetched x_j
        if (!valid || j != n) a.out_tokens[b * (K + 1) + j] = out;
      }
      if (lane == 0) a.out_n[b] = valid ? n : -1;
      if (!valid) continue;
      const int pos = s * (K + 1) + n;
      SampleParams sp;
      sp.mA = st_s[pos * 4 + 0];
      sp.invSA = __fdiv_rn(1.0f, st_s[pos * 4 + 1]);
      sp.mB = st_s[pos * 4 + 2];
      sp.invSB = __fdiv_rn(1.0f, st_s[pos * 4 + 3]);
      sp.lam = lam;
      int kind = (n == K) ? kWBonus
                          : ((MODE == kProbMix && !(lam < 1.0f)) ? kWMixture : kWResidual);
      const T *ra = st_t + (int64_t)pos * V;
      const T *rb = st_d + ((int64_t)s * K + (n < K ? n : 0)) * V;
      float R = 0.0f;
      int tok = warp_sample<T, MODE>(ra, rb, V, kind, sp, p_ur[m], &R);
      if (!(R > 0.0f) && kind == kWResidual)  // zero residual mass (round-off only): p~ instead
        tok = warp_sample<T, MODE>(ra, rb, V, kWMixture, sp, p_ur[m], &R);
      if (lane == 0) a.out_tokens[b * (K + 1) + n] = tok;
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
  return e;
}

int tile_tma_blocks_per_sm(int dtype_bf16, int mode, int smem_bytes) {
  if (dtype_bf16) return mode == kProbMix ? occ<uint16_t, kProbMix>(smem_bytes)
                                          : occ<uint16_t, kLogitMix>(smem_bytes);
  return mode == kProbMix ? occ<float, kProbMix>(smem_bytes) : occ<float, kLogitMix>(smem_bytes);
}

cudaError_t tile_tma_launch(const TileArgs &a, int dtype_bf16, int mode, int64_t grid,
                            int smem_bytes, cudaStream_t stream) {
  const dim3 g((unsigned)grid), blk(kNT);
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
