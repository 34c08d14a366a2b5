// Renormalised softmax weights of the kept logits, w_r = exp(l_r - m) /
// sum_i exp(l_i - m) with m the largest kept logit, computed in
// double-float arithmetic: a value is an unevaluated sum hi + lo of two fp32
// numbers (Dekker 1971, "A floating-point technique for extending the
// available precision"; error-free TwoSum and, with a fused multiply-add,
// TwoProduct), which carries about 44 bits.  The result rounded to fp32 is
// the fp32 rounding of the exact weight, or its neighbour when the exact
// value lies within 2^-44 of a rounding boundary: so within one ulp of the
// weight computed in fp64, without fp64 arithmetic (a small fraction of the
// fp32 rate on this GPU).
// exp: Cody and Waite's range reduction d = k ln2 + r, |r| <= ln2 / 2, with
// ln2 split so that k * LN2_HI is exact for |k| < 256, then the Taylor series
// of exp(r) to degree 11 (next term below 2^-47 relative), then * 2^k.
// Constants: 1/n! and ln2 rounded to fp32 pairs hi + lo from their exact
// values.
#pragma once
#include <cuda_runtime.h>

namespace moe {

struct dflt {
  float hi, lo;
};

__device__ __forceinline__ dflt df_two_sum(float a, float b) {
  const float s = a + b;
  const float bb = s - a;
  return {s, (a - (s - bb)) + (b - bb)};
}
// |a| >= |b|
__device__ __forceinline__ dflt df_quick_two_sum(float a, float b) {
  const float s = a + b;
  return {s, b - (s - a)};
}
__device__ __forceinline__ dflt df_two_prod(float a, float b) {
  const float p = a * b;
  return {p, fmaf(a, b, -p)};
}
__device__ __forceinline__ dflt df_add(dflt a, dflt b) {
  dflt s = df_two_sum(a.hi, b.hi);
  s.lo += a.lo + b.lo;
  return df_quick_two_sum(s.hi, s.lo);
}
__device__ __forceinline__ dflt df_mul(dflt a, dflt b) {
  dflt p = df_two_prod(a.hi, b.hi);
  p.lo = fmaf(a.hi, b.lo, fmaf(a.lo, b.hi, p.lo));
  return df_quick_two_sum(p.hi, p.lo);
}
__device__ __forceinline__ dflt df_div(dflt a, dflt b) {
  const float q1 = a.hi / b.hi;
  const dflt p = df_mul(b, dflt{q1, 0.0f});
  const dflt r = df_add(a, dflt{-p.hi, -p.lo});
  const float q2 = r.hi / b.hi;
  return df_quick_two_sum(q1, q2);
}

// exp(dh + dl) for -150 < dh <= 0 (|dl| <= ulp(dh) / 2)
__device__ __forceinline__ dflt df_exp_nonpos(float dh, float dl) {
  constexpr float kInvLn2 = 0x1.715476p+0f;
  constexpr float kLn2Hi = 0x1.62e4p-1f;  // 16 significant bits
  constexpr float kLn2LoHi = 0x1.7f7d1cp-20f, kLn2LoLo = 0x1.ef357ap-45f;
  // 1/n!, n = 0..11, as hi + lo
  constexpr float kHi[12] = {0x1p+0f,        0x1p+0f,        0x1p-1f,        0x1.555556p-3f,
                             0x1.555556p-5f, 0x1.111112p-7f, 0x1.6c16c2p-10f, 0x1.a01a02p-13f,
                             0x1.a01a02p-16f, 0x1.71de3ap-19f, 0x1.27e4fcp-22f, 0x1.ae6456p-26f};
  constexpr float kLo[12] = {0.0f,          0.0f,           0.0f,           -0x1.555556p-28f,
                             -0x1.555556p-30f, -0x1.dddddep-32f, -0x1.27d27ep-35f, -0x1.7f97fap-39f,
                             -0x1.7f97fap-42f, 0x1.55b1ccp-45f, -0x1.10ec14p-47f, 0x1.fd5138p-52f};
  const float k = rintf(dh * kInvLn2);
  const float rh = fmaf(-k, kLn2Hi, dh);  // exact: k has at most 8 significant bits
  const dflt kl = df_two_prod(k, kLn2LoHi);
  dflt r = df_add(dflt{rh, 0.0f}, dflt{-kl.hi, -(kl.lo + k * kLn2LoLo)});
  r = df_add(r, dflt{dl, 0.0f});
  dflt p{kHi[11], kLo[11]};
#pragma unroll
  for (int n = 10; n >= 0; --n) p = df_add(df_mul(p, r), dflt{kHi[n], kLo[n]});
  // * 2^k, k in [-217, 0], as two power-of-two factors (each a normal float)
  const int ki = (int)k;
  const int a = ki / 2, b = ki - a;
  const float fa = __int_as_float((a + 127) << 23), fb = __int_as_float((b + 127) << 23);
  return {p.hi * fa * fb, p.lo * fa * fb};
}

// exp(v - m) with the limits of the infinite cases (+inf logits share
// equally; if every kept logit is -inf they share equally), as hi + lo
__device__ __forceinline__ dflt df_softmax_term(float v, float m) {
  if (m == INFINITY) return {v == INFINITY ? 1.0f : 0.0f, 0.0f};
  if (m == -INFINITY) return {1.0f, 0.0f};
  if (v == -INFINITY) return {0.0f, 0.0f};
  const dflt dd = df_two_sum(v, -m);  // exact
  if (dd.hi < -150.0f) return {0.0f, 0.0f};
  return df_exp_nonpos(dd.hi, dd.lo);
}

}  // namespace moe
