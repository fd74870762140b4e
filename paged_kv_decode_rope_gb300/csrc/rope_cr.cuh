// rope_cr.cuh -- correctly rounded fp64 cos and sin of RoPE angles (sm_103a).
//
// "手写LLM推理引擎：Tokenizer、Transformer与Detokenizer三段式实现" section 3.2
// rotates by the angle m theta_j; this library forms that angle in fp64 as one
// rounded product a = fl(pos * inv_freq_j). The new key it stores is the bf16
// rounding of an fp64 rotation by cos(a) and sin(a), so those two fp64 values
// must be fixed exactly, independently of any math library: they are the fp64
// numbers nearest to the true cos(a) and sin(a) (correct rounding).
//
// Evaluation in double-double arithmetic (a value is the unevaluated sum
// hi + lo of two doubles, about 106 significant bits), one function value per
// thread:
//  * cos(a) or sin(a) is +-cos(r) or +-sin(r) of the reduced argument
//    r = a - k pi/2, k the integer nearest to a 2/pi, |r| <= pi/4 (+ a few
//    ulps); sin(a) = cos(a - pi/2) shifts the quadrant k mod 4 by one.
//  * Reduction after Cody and Waite: pi/2 is written as three 30-bit parts
//    C1 + C2 + C3 followed by two full doubles C4 + C5 (together pi/2 to
//    about 2^-203 relative). Each k Ci is formed exactly as a two-product with
//    an FMA, and the differences are accumulated in double-double.
//  * Taylor series of cos r and sin r in nested (Horner) form, z = r^2:
//      cos r = 1 - z/(1*2) (1 - z/(3*4) (1 - ...)),
//      sin r = r (1 - z/(2*3) (1 - z/(4*5) (1 - ...))),
//    fifteen factors each, the innermost seven in plain fp64 (an error there
//    reaches the result scaled by less than 2^-49) and the eight outer ones
//    in double-double,
//    with the reciprocals 1/((2n-1)(2n)) and 1/((2n)(2n+1)) as double-double
//    constants. A lane picks the cos or sin coefficients by value (no branch),
//    so a warp that mixes the two series does not diverge.
//  * Rounding test (Ziv): the double-double result v is within
//    eps = 2^-90 |v| + k 2^-128 of the true value (series and arithmetic
//    errors, about 2^-100 |v|; the reduction's, below k 2^-130, and none
//    when k = 0). When no midpoint between neighbouring doubles lies within eps
//    of v, v.hi is the correctly rounded value. Otherwise the function still
//    returns v.hi (within half an ulp plus eps) and reports the value as
//    undecided; for an angle that is not special this happens with a
//    probability of about 2^-37.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace pkv {

// Double-double reciprocals of the Taylor factors: index n = 1..15 holds
// 1/((2n-1)(2n)) (cos) and 1/((2n)(2n+1)) (sin); built on the host once
// (rope_series_coef) and passed to kernels by value.
struct RopeSeriesCoef {
  double cos_hi[16], cos_lo[16];
  double sin_hi[16], sin_lo[16];
};

// Host: hi = 1/d rounded, lo = (1 - hi d)/d rounded, the remainder 1 - hi d
// being exact with an FMA; hi + lo is 1/d to about 2^-106.
RopeSeriesCoef rope_series_coef();

struct Dd {
  double hi, lo;
};

// Knuth's two-sum: hi + lo = a + b exactly.
__device__ __forceinline__ Dd dd_two_sum(double a, double b) {
  const double s = __dadd_rn(a, b);
  const double bv = __dsub_rn(s, a);
  const double av = __dsub_rn(s, bv);
  return {s, __dadd_rn(__dsub_rn(a, av), __dsub_rn(b, bv))};
}

// Dekker's fast two-sum, for |a| >= |b| or a == 0.
__device__ __forceinline__ Dd dd_fast_sum(double a, double b) {
  const double s = __dadd_rn(a, b);
  return {s, __dsub_rn(b, __dsub_rn(s, a))};
}

// hi + lo = a b exactly (an FMA gives the product's rounding error).
__device__ __forceinline__ Dd dd_two_prod(double a, double b) {
  const double p = __dmul_rn(a, b);
  return {p, __fma_rn(a, b, -p)};
}

// x + y, relative error about 3 2^-106 whatever the signs.
__device__ __forceinline__ Dd dd_add(Dd x, Dd y) {
  Dd s = dd_two_sum(x.hi, y.hi);
  const Dd t = dd_two_sum(x.lo, y.lo);
  s = dd_fast_sum(s.hi, __dadd_rn(s.lo, t.hi));
  return dd_fast_sum(s.hi, __dadd_rn(s.lo, t.lo));
}

__device__ __forceinline__ Dd dd_neg(Dd x) { return {-x.hi, -x.lo}; }

// x y, relative error about 2^-104.
__device__ __forceinline__ Dd dd_mul(Dd x, Dd y) {
  const Dd p = dd_two_prod(x.hi, y.hi);
  const double c = __fma_rn(x.hi, y.lo, __dmul_rn(x.lo, y.hi));
  return dd_fast_sum(p.hi, __dadd_rn(p.lo, c));
}

// pi/2 = C1 + C2 + C3 + C4 + C5 (C1..C3 of 30 significant bits, C4 and C5
// the following two doubles), and 2/pi rounded to fp64.
constexpr double kHalfPiC1 = 0x1.921fb54000000p+0;
constexpr double kHalfPiC2 = 0x1.10b4611800000p-30;
constexpr double kHalfPiC3 = 0x1.313198a000000p-61;
constexpr double kHalfPiC4 = 0x1.701b839a25205p-92;
constexpr double kHalfPiC5 = -0x1.8fbbacc19c5ffp-146;
constexpr double kTwoOverPi = 0x1.45f306dc9c883p-1;

// Whether v.hi is the fp64 value nearest to every real within eps of
// hi + lo (v normalised: hi = fl(hi + lo)).
__device__ __forceinline__ bool dd_rounds_to_hi(Dd v, double eps) {
  if (v.hi == 0.0) return v.lo == 0.0 && eps == 0.0;
  const uint64_t bits = static_cast<uint64_t>(__double_as_longlong(v.hi)) & 0x7fffffffffffffffull;
  const int e = static_cast<int>(bits >> 52);
  if (e == 0 || e == 0x7ff) return false;  // subnormal or non-finite: not for RoPE angles
  const double ulp = __longlong_as_double(static_cast<long long>(e - 52) << 52);  // 2^(exp - 52)
  // the gap on lo's side: below a power of two (away from zero) it is half as wide
  const bool toward_zero = (v.lo < 0.0) == (v.hi > 0.0);
  const bool pow2 = (bits & 0x000fffffffffffffull) == 0;
  const double half_gap = (toward_zero && pow2) ? 0.25 * ulp : 0.5 * ulp;
  return __dadd_ru(fabs(v.lo), eps) < half_gap;
}

// cos(a) (want_sin = false) or sin(a) (want_sin = true), correctly rounded to
// fp64; *certain is false when the rounding test could not decide (the value
// returned is then within half an ulp plus eps). a must be finite and
// |a| < 2^52.
__device__ __forceinline__ double rope_cos_or_sin_cr(double a, bool want_sin,
                                                     const RopeSeriesCoef& cf, bool* certain) {
  const bool neg = signbit(a);
  const double x = fabs(a);
  const double k = rint(__dmul_rn(x, kTwoOverPi));
  // r = x - k pi/2 in double-double
  Dd r = dd_add({x, 0.0}, dd_neg(dd_two_prod(k, kHalfPiC1)));
  r = dd_add(r, dd_neg(dd_two_prod(k, kHalfPiC2)));
  r = dd_add(r, dd_neg(dd_two_prod(k, kHalfPiC3)));
  r = dd_add(r, dd_neg(dd_two_prod(k, kHalfPiC4)));
  r = dd_add(r, {-__dmul_rn(k, kHalfPiC5), 0.0});
  // quadrant of the cos evaluation: sin(x) = cos(x - pi/2)
  const int q = static_cast<int>((static_cast<long long>(k) + (want_sin ? 3 : 0)) & 3);
  const bool odd = q & 1;  // +-sin r, else +-cos r
  const Dd z = dd_mul(r, r);
  double t = 1.0;
#pragma unroll
  for (int n = 15; n >= 9; --n)
    t = __fma_rn(-__dmul_rn(z.hi, odd ? cf.sin_hi[n] : cf.cos_hi[n]), t, 1.0);
  Dd tt = {t, 0.0};
#pragma unroll
  for (int n = 8; n >= 1; --n) {
    const Dd c = odd ? Dd{cf.sin_hi[n], cf.sin_lo[n]} : Dd{cf.cos_hi[n], cf.cos_lo[n]};
    const Dd w = dd_mul(dd_mul(z, tt), c);
    const Dd s = dd_two_sum(1.0, -w.hi);
    tt = dd_fast_sum(s.hi, __dsub_rn(s.lo, w.lo));
  }
  Dd v = odd ? dd_mul(r, tt) : tt;
  if ((q == 1 || q == 2) != (want_sin && neg)) v = dd_neg(v);
  const double eps = __fma_rn(fabs(v.hi), 0x1p-90, __dmul_rn(k, 0x1p-128));
  *certain = (x == 0.0) || dd_rounds_to_hi(v, eps);
  return v.hi;
}

}  // namespace pkv
