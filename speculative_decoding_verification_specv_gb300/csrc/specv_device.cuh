// specv_device.cuh -- device helpers shared by the verify kernels (sm_103a).
//
// Row statistics are kept as (m, S): m = max_v z_v and S = sum_v exp(z_v - m),
// both fp32.  A probability is exp(z - m) / S.  Ratios of probabilities are
// formed from differences (z_x - m), which are exact or nearly so for the
// likely tokens, so the acceptance ratio keeps fp32 accuracy even when the
// logits are large.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace specv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Verification modes: the two mixtures of the sampling rule, and greedy
// verification (accept x_i iff it is the argmax of the mixed logits).
enum : int { kProbMix = 0, kLogitMix = 1, kGreedy = 2 };

// 2^x and log2(x) on the special-function unit (PTX ex2/lg2, flush-to-zero).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// exp(z - m) computed as 2^((z - m) * log2 e); the subtraction is done first
// (exact for z near m) and rounded operations are spelled out so that every
// call site rounds identically.
__device__ __forceinline__ float exp_shifted(float z, float m) {
  return ex2(__fmul_rn(__fsub_rn(z, m), kLog2e));
}

// Logit-mode mixture (1 - l) z_t + l z_q, written as z_t + l (z_q - z_t):
// equal in exact arithmetic, and exactly z_t whenever z_q == z_t.  A term of
// weight zero drops out, so l = 0 gives z_t and l = 1 gives z_q exactly,
// whatever the other row holds.  Masked logits (-inf, e.g. a padded
// vocabulary or a grammar mask): a masked entry of a row with positive weight
// masks the mixed entry.  For 0 < l < 1 the expression is -inf when z_q is,
// and NaN when z_t is -inf (inf - inf); fmaxf turns that NaN into -inf and
// leaves every other value alone.
__device__ __forceinline__ float mix_logit_interior(float zt, float zq, float lam) {
  return fmaxf(__fmaf_rn(lam, __fsub_rn(zq, zt), zt), -INFINITY);
}
__device__ __forceinline__ float mix_logit(float zt, float zq, float lam) {
  return lam == 0.0f ? zt : (lam == 1.0f ? zq : mix_logit_interior(zt, zq, lam));
}

// The exponent offset -m log2e of a running maximum m, or 0 while m is -inf
// (every entry folded so far is masked): then the masked entries give
// 2^(-inf) = 0 instead of 2^(-inf + inf) = NaN.
__device__ __forceinline__ float neg_scaled_max(float m) {
  return m == -INFINITY ? 0.0f : -__fmul_rn(m, kLog2e);
}

// bf16 bits -> fp32 (exact).
__device__ __forceinline__ float bf16_bits_to_float(uint32_t bits16) {
  return __uint_as_float(bits16 << 16);
}

// Element access for the two logit types.  A 16-byte vector holds kPerVec
// elements; get(v, e) widens element e to fp32 (exact for both types).
template <typename T>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kPerVec = 4;  // elements per 16-byte vector
  static constexpr uint32_t kNegInfBits = 0xff800000u;
  __device__ __forceinline__ static float load(const float *p) { return __ldg(p); }
  __device__ __forceinline__ static uint32_t load_bits(const float *p) {
    return __float_as_uint(__ldg(p));
  }
  __device__ __forceinline__ static float get(const uint4 &v, int e) {
    const uint32_t w = e == 0 ? v.x : e == 1 ? v.y : e == 2 ? v.z : v.w;
    return __uint_as_float(w);
  }
  // element e of a vector assembled from scalar loads
  __device__ __forceinline__ static void put_bits(uint4 &v, int e, uint32_t bits) {
    if (e == 0) v.x = bits;
    else if (e == 1) v.y = bits;
    else if (e == 2) v.z = bits;
    else v.w = bits;
  }
};
template <>
struct Elem<uint16_t> {  // bfloat16 storage
  static constexpr int kPerVec = 8;
  static constexpr uint32_t kNegInfBits = 0xff80u;
  __device__ __forceinline__ static float load(const uint16_t *p) {
    return bf16_bits_to_float(__ldg(p));
  }
  __device__ __forceinline__ static uint32_t load_bits(const uint16_t *p) { return __ldg(p); }
  __device__ __forceinline__ static float get(const uint4 &v, int e) {
    const uint32_t w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  }
  __device__ __forceinline__ static void put_bits(uint4 &v, int e, uint32_t bits) {
    uint32_t &w = (e >> 1) == 0 ? v.x : (e >> 1) == 1 ? v.y : (e >> 1) == 2 ? v.z : v.w;
    w = (e & 1) ? ((w & 0x0000ffffu) | (bits << 16)) : ((w & 0xffff0000u) | bits);
  }
};

// 16-byte streaming load: read-only path, no L1 allocation (each byte is
// used once by this CTA); L2 keeps its normal policy so that the sampler's
// re-read of the rejected row can hit in L2.
__device__ __forceinline__ uint4 ld_stream16(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Merge two (m, S) partial statistics.  Empty partials are (-inf, 0).
__device__ __forceinline__ void merge_stats(float &m, float &s, float m2, float s2) {
  float mn = fmaxf(m, m2);
  if (mn == -INFINITY) return;  // both empty
  float a = (m == mn) ? s : __fmul_rn(s, exp_shifted(m, mn));
  float b = (m2 == mn) ? s2 : __fmul_rn(s2, exp_shifted(m2, mn));
  m = mn;
  s = __fadd_rn(a, b);
}

// Merge of n partial statistics of two rows at once; get(r) returns
// (mA, sA, mB, sB) of partial r.  The maxima come first, then every partial is
// scaled to them and summed in index order, so the n exponentials are
// independent of one another (a pairwise merge would chain n rescales).
// Empty partials are (-inf, 0) and add nothing.
template <typename Get>
__device__ __forceinline__ void merge_stats2_n(int n, Get get, float &mA, float &sA, float &mB,
                                               float &sB) {
  float MA = -INFINITY, MB = -INFINITY;
  for (int r = 0; r < n; ++r) {
    const float4 q = get(r);
    MA = fmaxf(MA, q.x);
    MB = fmaxf(MB, q.z);
  }
  float SA = 0.0f, SB = 0.0f;
  for (int r = 0; r < n; ++r) {
    const float4 q = get(r);
    SA = __fadd_rn(SA, q.x == MA ? q.y : __fmul_rn(q.y, exp_shifted(q.x, MA)));
    SB = __fadd_rn(SB, q.z == MB ? q.w : __fmul_rn(q.w, exp_shifted(q.z, MB)));
  }
  mA = MA;
  sA = SA;
  mB = MB;
  sB = SB;
}

// Merge across a warp: the warp's maximum by a butterfly, then every lane's
// sum scaled to it and added by a butterfly (one exponential per lane instead
// of one per level).  Addition is commutative, so every lane ends with the
// same result, and the combination order is fixed.
__device__ __forceinline__ void warp_merge_stats(float &m, float &s) {
  float M = m;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float t = m == M ? s : __fmul_rn(s, exp_shifted(m, M));  // an empty lane (-inf, 0) adds 0
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) t = __fadd_rn(t, __shfl_xor_sync(0xffffffffu, t, off));
  m = M;
  s = t;
}

// Greedy: of two (value, index) candidates keep the larger value, and the
// smaller index among equal values (the first maximum in index order).  An
// empty candidate is (-inf, INT_MAX).
__device__ __forceinline__ void argmax_merge(float &w, int &idx, float w2, int idx2) {
  if (w2 > w || (w2 == w && idx2 < idx)) {
    w = w2;
    idx = idx2;
  }
}

// Butterfly argmax across a warp; every lane ends with the result.
__device__ __forceinline__ void warp_argmax(float &w, int &idx) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    const float w2 = __shfl_xor_sync(0xffffffffu, w, off);
    const int i2 = __shfl_xor_sync(0xffffffffu, idx, off);
    argmax_merge(w, idx, w2, i2);
  }
}

// Greedy score of one entry: the mixed logit z_t + l (z_q - z_t), with the
// masking rule of mix_logit.
__device__ __forceinline__ float greedy_score(float zt, float zq, float lam) {
  return mix_logit(zt, zq, lam);
}

// Statistics of one position: A = source row of p~ (target row in
// probability mode and at the bonus position, mixed row in logit mode),
// B = draft row.
struct PosStats {
  float mA, sA, mB, sB;
};

// Acceptance ratio p~(x)/q(x) of one drafted position, and optionally p~(x)
// and q(x) themselves.
//   prob:  r = p_t(x)/q(x) = e^{(zt_x - mA) - (zq_x - mB)} * sB / sA and
//          p~/q = 1 + (1 - l)(r - 1), which is exactly 1 when r == 1 or l == 1.
//   logit: p~/q = e^{(w_x - mA) - (zq_x - mB)} * sB / sA, w_x = mix_logit(.).
//   q(x) = 0 (the drafted token is masked in the draft row): the ratio is
//   +inf (accept) if p~(x) > 0, else 0 (reject).
__device__ __forceinline__ float accept_ratio(int mode, const PosStats &st, float zt_x, float zq_x,
                                              float lam, float *ptilde_x, float *q_x) {
  float a_x = (mode == kProbMix) ? zt_x : mix_logit(zt_x, zq_x, lam);
  float da = __fsub_rn(a_x, st.mA);
  float db = __fsub_rn(zq_x, st.mB);
  if (ptilde_x != nullptr) {
    float q = __fdividef(ex2(__fmul_rn(db, kLog2e)), st.sB);
    float pa = __fdividef(ex2(__fmul_rn(da, kLog2e)), st.sA);
    *q_x = q;
    *ptilde_x = (mode == kProbMix) ? __fmaf_rn(lam, q, __fmul_rn(__fsub_rn(1.0f, lam), pa)) : pa;
  }
  if (zq_x == -INFINITY) {
    const bool pos = (mode == kProbMix) ? (lam < 1.0f && zt_x != -INFINITY) : (a_x != -INFINITY);
    return pos ? INFINITY : 0.0f;
  }
  float d = __fsub_rn(da, db);
  float e = (d == 0.0f) ? 1.0f : ex2(__fmul_rn(d, kLog2e));
  // sB / sA with the SFU reciprocal (a few ulp); exactly 1 for equal sums
  float r = __fmul_rn(e, st.sB == st.sA ? 1.0f : __fdividef(st.sB, st.sA));
  if (mode == kProbMix) r = __fmaf_rn(__fsub_rn(1.0f, lam), __fsub_rn(r, 1.0f), 1.0f);
  return r;
}

// The acceptance test r < min(1, ratio) (strict, as printed in the pages' loop).
__device__ __forceinline__ bool accept_test(float u, float ratio) {
  return u < fminf(1.0f, ratio);
}

__device__ __forceinline__ bool lambda_valid(float lam) { return lam >= 0.0f && lam <= 1.0f; }

// Weight of vocabulary entry v in the sampler.  What selects the weight:
//   kWResidual : max(0, p~_v - q_v) up to the constant factor (1 - l) in
//                probability mode (p~ - q = (1 - l)(p_t - q) there), exactly
//                in logit mode;
//   kWBonus    : p~_v at the bonus position = target softmax of row K;
//   kWMixture  : p~_v itself (fallback when the residual has zero mass);
//   kWResidualC: max(0, p~_v - c q_v), the residual after rejections of
//                several independent drafts of one node (tree verification;
//                c = 1 is the residual of the first rejection).
enum : int { kWResidual = 0, kWBonus = 1, kWMixture = 2, kWResidualC = 3 };

struct SampleParams {
  float mA, invSA, mB, invSB, lam;
  float c;       // threshold of kWResidualC
  float nA, nB;  // -(m log2e + log2 S): a probability is 2^(z log2e + n) = exp(z - m) / S
};

// The exponent offsets nA, nB from the statistics: one fused multiply-add and
// the SFU's 2^x per probability in the sampler.  log2 S comes from the SFU
// (absolute error near 2^-22: a common factor within 2e-7 of 1 on a row's
// probabilities).  Equal statistics give equal offsets (a residual of
// identical rows stays exactly zero).
__device__ __forceinline__ void set_exponent_offsets(SampleParams &p, float sA, float sB) {
  p.nA = -__fmaf_rn(p.mA, kLog2e, lg2(sA));
  p.nB = -__fmaf_rn(p.mB, kLog2e, lg2(sB));
}

// Sampler parameters of a position from its statistics.  The reciprocals are
// SFU approximations: a common factor on a weight vector does not move its
// normalised CDF beyond round-off, and equal sums give equal reciprocals.
__device__ __forceinline__ SampleParams make_sample_params(float mA, float sA, float mB, float sB,
                                                           float lam) {
  SampleParams p;
  p.mA = mA;
  p.invSA = __fdividef(1.0f, sA);
  p.mB = mB;
  p.invSB = __fdividef(1.0f, sB);
  p.lam = lam;
  p.c = 1.0f;
  set_exponent_offsets(p, sA, sB);
  return p;
}

// The same with correctly rounded reciprocals.
__device__ __forceinline__ SampleParams make_sample_params_rn(float mA, float sA, float mB,
                                                              float sB, float lam) {
  SampleParams p;
  p.mA = mA;
  p.invSA = __fdiv_rn(1.0f, sA);
  p.mB = mB;
  p.invSB = __fdiv_rn(1.0f, sB);
  p.lam = lam;
  p.c = 1.0f;
  set_exponent_offsets(p, sA, sB);
  return p;
}

// A probability exp(z - m) / S from the exponent offset n of its row.
__device__ __forceinline__ float prob_from_offset(float z, float n) {
  return ex2(__fmaf_rn(z, kLog2e, n));
}

__device__ __forceinline__ float sample_weight(int mode, int kind, const SampleParams &p, float zt,
                                               float zq) {
  if (kind == kWBonus) return prob_from_offset(zt, p.nA);
  float a = (mode == kProbMix) ? zt : mix_logit(zt, zq, p.lam);
  float pa = prob_from_offset(a, p.nA);
  float pq = prob_from_offset(zq, p.nB);
  if (kind == kWResidual) return fmaxf(0.0f, __fsub_rn(pa, pq));
  const float pt = (mode == kProbMix) ? __fmaf_rn(p.lam, pq, __fmul_rn(__fsub_rn(1.0f, p.lam), pa))
                                      : pa;
  if (kind == kWResidualC) return fmaxf(0.0f, __fsub_rn(pt, __fmul_rn(p.c, pq)));
  return pt;  // kWMixture
}

// sample_weight without branches on `kind`: every candidate is computed and
// one is selected, for warps whose lanes serve sequences of different kinds
// (a bonus sequence next to a residual one).  Same values as sample_weight;
// the candidates not selected may be non-finite and are discarded.  For the
// bonus kind the caller passes zq = zt (there is no draft row at K + 1): the
// mixed logit is then zt itself (mix_logit(zt, zt, l) == zt in every case,
// masked entries included), so pa is the bonus weight in both modes.
__device__ __forceinline__ float sample_weight_sel(int mode, int kind, const SampleParams &p,
                                                   float zt, float zq) {
  const float a = (mode == kProbMix) ? zt : mix_logit(zt, zq, p.lam);
  const float pa = prob_from_offset(a, p.nA);
  const float pq = prob_from_offset(zq, p.nB);
  const float resid = fmaxf(0.0f, __fsub_rn(pa, pq));
  const float mixed =
      (mode == kProbMix) ? __fmaf_rn(p.lam, pq, __fmul_rn(__fsub_rn(1.0f, p.lam), pa)) : pa;
  return kind == kWBonus ? pa : (kind == kWResidual ? resid : mixed);
}

}  // namespace specv
