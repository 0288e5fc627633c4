// Double-float row arithmetic of the precise redraw: exp((z - max) / T) of
// one logit in double-float precision, and the 8-entry logit loads the
// redraw passes use.
#pragma once

#include "ops.cuh"
#include "precise.cuh"
#include "verify_units.cuh"

namespace sv {

struct HpRow {
  float m;         // row maximum
  float khi, klo;  // log2(e) / T as a double-float
  float thr;       // top-k threshold (-inf: none)
};

__device__ __forceinline__ HpRow hp_row(const RowDesc &d, float T) {
  HpRow r;
  r.m = d.m;
  // log2(e) / T as a double-float: the quotient, then the exact remainder of
  // the rounded division (plus the low part of log2(e)) divided by T
  const float l2e_hi = 1.44269502162933349609375f;      // log2(e) rounded to float
  const float l2e_lo = 1.9259629911266175e-8f;  // log2(e) - l2e_hi, rounded
  const float q = __fdiv_rn(l2e_hi, T);
  const float rem = fmaf(-q, T, l2e_hi);
  r.khi = q;
  r.klo = __fdiv_rn(__fadd_rn(rem, l2e_lo), T);
  r.thr = d.thr;
  return r;
}

// exp((z - max) / T) as a double-float; 0 below the top-k threshold.
// Branch-free like df_exp2 (an excluded entry is computed as z = max and
// selected away).
__device__ __forceinline__ Df hp_exp(const HpRow &r, float z, const float *th, const float *tl) {
  const bool zero = !(z > -INFINITY) || z < r.thr;
  const float zz = zero ? r.m : z;
  float dh, dl;
  two_sum(zz, -r.m, dh, dl);  // z - max exactly
  const float t_hi = __fmul_rn(dh, r.khi);
  const float t_lo =
      __fadd_rn(fmaf(dh, r.khi, -t_hi), fmaf(dh, r.klo, __fmul_rn(dl, r.khi)));
  const Df v = df_exp2(df_norm(t_hi, t_lo), th, tl);
  return zero ? Df{0.f, 0.f} : v;
}

// Logits of the 8 entries from `base` (a multiple of 8); -inf at or past `end`.
template <typename TE>
__device__ __forceinline__ void hp_load8(const TE *g, int base, int end, bool vec, float z[8]) {
  if (vec && base + 8 <= end) {
    if (sizeof(TE) == 2) {
      const uint4 w = *reinterpret_cast<const uint4 *>(g + base);
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        z[2 * i] = __uint_as_float(ws[i] << 16);
        z[2 * i + 1] = __uint_as_float(ws[i] & 0xFFFF0000u);
      }
    } else {
      const float4 a = *reinterpret_cast<const float4 *>(g + base);
      const float4 b = *reinterpret_cast<const float4 *>(g + base + 4);
      z[0] = a.x; z[1] = a.y; z[2] = a.z; z[3] = a.w;
      z[4] = b.x; z[5] = b.y; z[6] = b.z; z[7] = b.w;
    }
    return;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) z[e] = base + e < end ? to_f32(g[base + e]) : -INFINITY;
}

}  // namespace sv
