// Double-float ("df32") arithmetic: a value is the unevaluated sum hi + lo of
// two floats with |lo| <= ulp(hi) / 2, about 48 significant bits.  The error-
// free transformations are Knuth's TwoSum and Dekker's Fast2Sum, and the exact
// product split uses one fused multiply-add (Dekker 1971, "A floating-point
// technique for extending the available precision"; the fma form is the one
// in Muller et al., "Handbook of Floating-Point Arithmetic", ch. 4).
//
// The explicit __fadd_rn / __fsub_rn / __fmul_rn calls keep the compiler from
// contracting or reassociating the steps whose rounding errors are captured.
#pragma once

#include <cstdint>

namespace sv {

struct Df {
  float hi, lo;
};

// a + b = s + e exactly (any magnitudes).
__device__ __forceinline__ void two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// a + b = s + e exactly when |a| >= |b| (or a == 0).
__device__ __forceinline__ void fast_two_sum(float a, float b, float &s, float &e) {
  s = __fadd_rn(a, b);
  e = __fsub_rn(b, __fsub_rn(s, a));
}

__device__ __forceinline__ Df df_norm(float hi, float lo) {
  Df r;
  fast_two_sum(hi, lo, r.hi, r.lo);
  return r;
}

__device__ __forceinline__ Df df_add(Df a, Df b) {
  float s, e;
  two_sum(a.hi, b.hi, s, e);
  e = __fadd_rn(e, __fadd_rn(a.lo, b.lo));
  return df_norm(s, e);
}

__device__ __forceinline__ Df df_sub(Df a, Df b) {
  b.hi = -b.hi;
  b.lo = -b.lo;
  return df_add(a, b);
}

__device__ __forceinline__ Df df_mul(Df a, Df b) {
  const float p = __fmul_rn(a.hi, b.hi);
  const float e = fmaf(a.hi, b.hi, -p);  // exact rounding error of the product
  const float t = fmaf(a.hi, b.lo, __fmul_rn(a.lo, b.hi));
  return df_norm(p, __fadd_rn(e, t));
}

__device__ __forceinline__ double df_to_double(Df a) {
  return static_cast<double>(a.hi) + static_cast<double>(a.lo);
}

__device__ __forceinline__ Df df_from_double(double x) {
  Df r;
  r.hi = static_cast<float>(x);
  r.lo = static_cast<float>(x - static_cast<double>(r.hi));
  return r;
}

// 2^(j/64), j = 0..63, as double-float pairs (filled on the host from a
// double-precision exp2).
struct Exp2Table {
  float hi[64];
  float lo[64];
};

constexpr double kLn2d = 0.69314718055994530941723212145818;
constexpr float kLn2Hi = static_cast<float>(kLn2d);
constexpr float kLn2Lo = static_cast<float>(kLn2d - static_cast<double>(kLn2Hi));

// 2^t for a double-float t <= 0 (relative error below 1e-11):
//   t = n/64 + r with n = rint(64 t_hi), |r| <= 1/128 + |t_lo|;
//   2^t = 2^(n div 64) * 2^((n mod 64)/64) * e^(r ln 2), the middle factor
//   from the table and e^y = 1 + y + y^2/2 + ... + y^5/120 for |y| < 0.006
//   (truncation below 1e-15), the terms after y carried in single precision.
// Results below 2^-126 flush to zero.  Branch-free (the out-of-range case is
// computed on a stand-in argument and selected away), so that the compiler can
// interleave the independent evaluations of an unrolled loop.
__device__ __forceinline__ Df df_exp2(Df t, const float *tab_hi, const float *tab_lo) {
  const float nf0 = rintf(__fmul_rn(t.hi, 64.f));
  const bool under = !(nf0 >= -64.f * 126.f);  // also -inf and NaN
  if (under) t = Df{0.f, 0.f};
  const float nf = under ? 0.f : nf0;
  const float rh = fmaf(nf, -0.015625f, t.hi);  // exact: t.hi - nf / 64
  float r_hi, r_lo;
  two_sum(rh, t.lo, r_hi, r_lo);
  const int n = static_cast<int>(nf);
  const int j = n & 63;
  const int e = n >> 6;  // floor(n / 64)
  // y = r ln 2 as a double-float
  const float yh = __fmul_rn(r_hi, kLn2Hi);
  const float yl = __fadd_rn(fmaf(r_hi, kLn2Hi, -yh), fmaf(r_hi, kLn2Lo, __fmul_rn(r_lo, kLn2Hi)));
  // e^y - 1 = yh + (yl + q), q the terms of degree >= 2 (|q| < 2e-5)
  const float p5 = fmaf(yh, 1.f / 120.f, 1.f / 24.f);
  const float p4 = fmaf(yh, p5, 1.f / 6.f);
  const float p3 = fmaf(yh, p4, 0.5f);
  const float q = fmaf(__fmul_rn(yh, yh), p3, __fmul_rn(yh, yl));
  const float lo = __fadd_rn(yl, q);
  // T (1 + yh + lo), T = Th + Tl from the table
  const float Th = tab_hi[j], Tl = tab_lo[j];
  const float ph = __fmul_rn(Th, yh);
  const float pe = fmaf(Th, yh, -ph);
  float s, se;
  two_sum(Th, ph, s, se);
  const float tail = __fadd_rn(__fadd_rn(se, pe), fmaf(Th, lo, fmaf(Tl, yh, Tl)));
  Df r = df_norm(s, tail);
  const float scale = __int_as_float((e + 127) << 23);  // 2^e, -126 <= e <= 0
  r.hi = under ? 0.f : __fmul_rn(r.hi, scale);
  r.lo = under ? 0.f : __fmul_rn(r.lo, scale);
  return r;
}

}  // namespace sv
