// specv_tile.cu -- the small-vocabulary kernel: whole sequences per CTA.
//
// For short rows (V up to a few hundred) a cluster per position would spend
// more time on barriers than on bytes.  Here a CTA stages a tile of whole
// sequences -- their (K+1) target rows and K draft rows are contiguous in
// HBM -- into shared memory with coalesced 16-byte loads, then:
//   stage A: one thread per position computes the row statistics (max, then
//            sum of exp) of the p~ source row and of the draft row from
//            shared memory;
//   stage B: one warp per sequence evaluates the acceptance test of each
//            drafted position (lane j takes position j), finds the first
//            rejection with a ballot, writes the accepted prefix, and draws
//            the replacement or bonus token by inverse CDF with a warp scan
//            over the row (lane l takes entry v0 + l).
// The CTA loops over tiles (grid sized to the resident CTAs of the GPU).
// No scratch memory: everything between the stages lives in shared memory.
#include "specv_device.cuh"
#include "specv_internal.h"

namespace specv {

namespace {

constexpr int kNT = kTileThreads;
constexpr int kNW = kNT / 32;

template <typename T>
__device__ __forceinline__ float smem_val(const T *p);
template <>
__device__ __forceinline__ float smem_val<float>(const float *p) {
  return *p;
}
template <>
__device__ __forceinline__ float smem_val<uint16_t>(const uint16_t *p) {
  return bf16_bits_to_float(*p);
}

// Copy `count` elements from global to shared memory, 16 bytes at a time when
// both ends are 16-byte aligned and the byte count is a multiple of 16.
template <typename T>
__device__ __forceinline__ void stage_copy(T *dst, const T *src, int64_t count, bool vec) {
  if (vec) {
    const int64_t n16 = count * (int64_t)sizeof(T) / 16;
    const uint4 *s = reinterpret_cast<const uint4 *>(src);
    uint4 *d = reinterpret_cast<uint4 *>(dst);
    int64_t k = threadIdx.x;
    for (; k + 3 * kNT < n16; k += 4 * kNT) {
      uint4 v0 = ld_stream16(s + k), v1 = ld_stream16(s + k + kNT);
      uint4 v2 = ld_stream16(s + k + 2 * kNT), v3 = ld_stream16(s + k + 3 * kNT);
      d[k] = v0;
      d[k + kNT] = v1;
      d[k + 2 * kNT] = v2;
      d[k + 3 * kNT] = v3;
    }
    for (; k < n16; k += kNT) d[k] = ld_stream16(s + k);
  } else {
    for (int64_t k = threadIdx.x; k < count; k += kNT) dst[k] = src[k];
  }
}

// Warp inclusive scan (fixed order); every lane gets its inclusive prefix.
__device__ __forceinline__ float warp_incl_scan(float v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    float y = __shfl_up_sync(0xffffffffu, v, off);
    if (lane >= off) v = __fadd_rn(v, y);
  }
  return v;
}

// Warp traversal of one staged row pair in tiles of 32 entries, index order.
// Returns the mass in *mass when t = +inf; otherwise the smallest index whose
// running sum exceeds t, or the largest index with positive weight if
// round-off leaves none (-1 if the row has no positive weight).
template <typename T, int MODE>
__device__ int warp_traverse(const T *ra, const T *rb, int V, int kind, const SampleParams &sp,
                             float t, float *mass) {
  const int lane = threadIdx.x & 31;
  float base = 0.0f;
  int lastpos = -1;
  for (int v0 = 0; v0 < V; v0 += 32) {
    const int v = v0 + lane;
    float w = 0.0f;
    if (v < V) {
      const float za = smem_val<T>(ra + v);
      const float zb = kind != kWBonus ? smem_val<T>(rb + v) : 0.0f;
      w = sample_weight(MODE, kind, sp, za, zb);
      if (w > 0.0f) lastpos = v;
    }
    const float incl = warp_incl_scan(w);
    float excl = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) excl = 0.0f;
    const float total = __shfl_sync(0xffffffffu, incl, 31);
    const float lo = __fadd_rn(base, excl), hi = __fadd_rn(base, incl);
    const unsigned hit = __ballot_sync(0xffffffffu, v < V && lo <= t && t < hi);
    if (hit) return v0 + __ffs(hit) - 1;
    base = __fadd_rn(base, total);
  }
  if (mass != nullptr) *mass = base;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, off));
  return lastpos;
}

template <typename T, int MODE>
__global__ void __launch_bounds__(kNT) tile_kernel(TileArgs a) {
  extern __shared__ __align__(16) unsigned char smem[];
  const int K = a.K, V = a.V, TS = a.tile_seqs;
  T *st_t = reinterpret_cast<T *>(smem);
  T *st_d = reinterpret_cast<T *>(smem + a.smem_target_bytes);
  float4 *st_s = reinterpret_cast<float4 *>(smem + a.smem_target_bytes + a.smem_draft_bytes);
  const T *tgt = static_cast<const T *>(a.target);
  const T *dft = static_cast<const T *>(a.draft);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;

  for (int64_t tile = blockIdx.x; tile < a.num_tiles; tile += gridDim.x) {
    const int64_t b0 = tile * TS;
    const int nseq = (int)((a.B - b0) < TS ? (a.B - b0) : TS);
    stage_copy<T>(st_t, tgt + b0 * (K + 1) * (int64_t)V, (int64_t)nseq * (K + 1) * V, a.vec_copy);
    stage_copy<T>(st_d, dft + b0 * K * (int64_t)V, (int64_t)nseq * K * V, a.vec_copy);
    __syncthreads();

    // stage A: statistics of every position of the tile
    for (int task = threadIdx.x; task < nseq * (K + 1); task += kNT) {
      const int s = task / (K + 1), i = task - s * (K + 1);
      const bool pair = i < K;
      const T *ra = st_t + ((int64_t)s * (K + 1) + i) * V;
      const T *rb = st_d + ((int64_t)s * K + (pair ? i : 0)) * V;
      const float lam = a.lam[b0 + s];
      const int rot = lane % V;  // staggered start: lanes hit different banks
      float mA = -INFINITY, mB = -INFINITY;
      for (int k = 0; k < V; ++k) {
        int v = k + rot;
        v = v >= V ? v - V : v;
        float za = smem_val<T>(ra + v);
        if (pair) {
          const float zb = smem_val<T>(rb + v);
          if (MODE == kLogitMix) za = mix_logit(za, zb, lam);
          mB = fmaxf(mB, zb);
        }
        mA = fmaxf(mA, za);
      }
      float sA = 0.0f, sB = 0.0f;
      for (int k = 0; k < V; ++k) {
        int v = k + rot;
        v = v >= V ? v - V : v;
        float za = smem_val<T>(ra + v);
        if (pair) {
          const float zb = smem_val<T>(rb + v);
          if (MODE == kLogitMix) za = mix_logit(za, zb, lam);
          sB = __fadd_rn(sB, exp_shifted(zb, mB));
        }
        sA = __fadd_rn(sA, exp_shifted(za, mA));
      }
      st_s[s * (K + 1) + i] = make_float4(mA, sA, mB, sB);
    }
    __syncthreads();

    // stage B: one warp per sequence
    for (int s = warp; s < nseq; s += kNW) {
      const int64_t b = b0 + s;
      const float lam = a.lam[b];
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
          if (tok_ok && lam_ok) {
            const float4 st4 = st_s[s * (K + 1) + j];
            const PosStats st{st4.x, st4.y, st4.z, st4.w};
            const float zt_x = smem_val<T>(st_t + ((int64_t)s * (K + 1) + j) * V + x);
            const float zq_x = smem_val<T>(st_d + ((int64_t)s * K + j) * V + x);
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
      const bool all_tok = __all_sync(0xffffffffu, lane_ok);  // every lane votes
      const bool valid = lam_ok && all_tok;
      if (a.dbg_lse) {
        for (int j = lane; j <= K; j += 32) {
          const float4 st4 = st_s[s * (K + 1) + j];
          a.dbg_lse[(b * (K + 1) + j) * 2 + 0] = st4.x + lg2(st4.y) * kLn2;
          a.dbg_lse[(b * (K + 1) + j) * 2 + 1] = j < K ? st4.z + lg2(st4.w) * kLn2 : 0.0f;
        }
      }
      for (int j = lane; j <= K; j += 32) {
        int out = -1;
        if (valid && j < n) out = a.tokens[b * K + j];
        if (!valid || j != n) a.out_tokens[b * (K + 1) + j] = out;
      }
      if (lane == 0) a.out_n[b] = valid ? n : -1;
      if (!valid) continue;

      const float4 st4 = st_s[s * (K + 1) + n];
      const SampleParams sp = make_sample_params_rn(st4.x, st4.y, st4.z, st4.w, lam);
      int kind = (n == K) ? kWBonus
                          : (!(lam < 1.0f) ? kWMixture : kWResidual);
      const T *ra = st_t + ((int64_t)s * (K + 1) + n) * V;
      const T *rb = st_d + ((int64_t)s * K + (n < K ? n : 0)) * V;
      float R = 0.0f;
      warp_traverse<T, MODE>(ra, rb, V, kind, sp, INFINITY, &R);
      if (!(R > 0.0f) && kind == kWResidual) {
        kind = kWMixture;  // zero residual mass (round-off only): draw from p~ instead
        warp_traverse<T, MODE>(ra, rb, V, kind, sp, INFINITY, &R);
      }
      int tok = -1;
      if (R > 0.0f) {
        const float t = __fmul_rn(a.u_resample[b], R);
        tok = warp_traverse<T, MODE>(ra, rb, V, kind, sp, t, nullptr);
      }
      if (lane == 0) a.out_tokens[b * (K + 1) + n] = tok;
    }
    __syncthreads();  // the next tile overwrites the staged rows
  }
}

template <typename T, int MODE>
cudaError_t prep(int max_smem) {
  return cudaFuncSetAttribute(tile_kernel<T, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              max_smem);
}

template <typename T, int MODE>
int occ(int smem) {
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, tile_kernel<T, MODE>, kNT, smem) !=
      cudaSuccess)
    return 1;
  return nb > 0 ? nb : 1;
}

}  // namespace

cudaError_t tile_prepare(int max_smem_bytes) {
  cudaError_t e = cudaSuccess, r;
  if ((r = prep<float, kProbMix>(max_smem_bytes)) != cudaSuccess) e = r;
  if ((r = prep<float, kLogitMix>(max_smem_bytes)) != cudaSuccess) e = r;
  if ((r = prep<uint16_t, kProbMix>(max_smem_bytes)) != cudaSuccess) e = r;
  if ((r = prep<uint16_t, kLogitMix>(max_smem_bytes)) != cudaSuccess) e = r;
  return e;
}

int tile_blocks_per_sm(int dtype_bf16, int mode, int smem_bytes) {
  if (dtype_bf16) return mode == kProbMix ? occ<uint16_t, kProbMix>(smem_bytes)
                                          : occ<uint16_t, kLogitMix>(smem_bytes);
  return mode == kProbMix ? occ<float, kProbMix>(smem_bytes) : occ<float, kLogitMix>(smem_bytes);
}

cudaError_t tile_launch(const TileArgs &a, int dtype_bf16, int mode, int64_t grid, int smem_bytes,
                        cudaStream_t stream) {
  const dim3 g((unsigned)grid), blk(kNT);
  if (dtype_bf16) {
    if (mode == kProbMix)
      tile_kernel<uint16_t, kProbMix><<<g, blk, smem_bytes, stream>>>(a);
    else
      tile_kernel<uint16_t, kLogitMix><<<g, blk, smem_bytes, stream>>>(a);
  } else {
    if (mode == kProbMix)
      tile_kernel<float, kProbMix><<<g, blk, smem_bytes, stream>>>(a);
    else
      tile_kernel<float, kLogitMix><<<g, blk, smem_bytes, stream>>>(a);
  }
  return cudaGetLastError();
}

}  // namespace specv
