// Device helpers shared by the verification kernels (sm_103a).
#pragma once

#include <cooperative_groups.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "specverify.h"

namespace sv {

namespace cg = cooperative_groups;

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxCluster = 16;
constexpr float kLog2e = 1.4426950408889634f;

// ---------------------------------------------------------------------------
// element access: fp32 is stored as float, bf16 as its raw 16 bits
// ---------------------------------------------------------------------------

__device__ __forceinline__ float to_f32(float x) { return x; }
// A float that holds a value of the element type back in that type (exact).
template <typename TE>
__device__ __forceinline__ TE from_f32(float x);
template <>
__device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ uint16_t from_f32<uint16_t>(float x) {
  return static_cast<uint16_t>(__float_as_uint(x) >> 16);
}
__device__ __forceinline__ float to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Order-preserving unsigned key of a logit (larger key <=> larger value,
// except that -0 sorts just below +0).
__device__ __forceinline__ uint32_t order_key(float x) {
  uint32_t b = __float_as_uint(x);
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ uint32_t order_key(uint16_t b) {
  uint32_t x = b;
  return (x & 0x8000u) ? (~x & 0xFFFFu) : (x | 0x8000u);
}
__device__ __forceinline__ float key_value_f32(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}
__device__ __forceinline__ float key_value_bf16(uint32_t k) {
  uint32_t b = (k & 0x8000u) ? (k & 0x7FFFu) : (~k & 0xFFFFu);
  return __uint_as_float(b << 16);
}

// 2^x on the special-function unit (relative error about 2^-22; results below
// the smallest normal float flush to zero).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy
// as 1, 2, 3", SC'11): ten rounds of two 32x32->64 multiplies mixed with the
// key, the key advanced by two Weyl constants after each round.
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t philox_word0(uint32_t c0, uint32_t c1, uint32_t c2,
                                                 uint32_t c3, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int round = 0; round < 10; ++round) {
    const uint32_t lo_a = 0xD2511F53u * c0;
    const uint32_t hi_a = __umulhi(0xD2511F53u, c0);
    const uint32_t lo_b = 0xCD9E8D57u * c2;
    const uint32_t hi_b = __umulhi(0xCD9E8D57u, c2);
    const uint32_t n0 = hi_b ^ c1 ^ k0;
    const uint32_t n2 = hi_a ^ c3 ^ k1;
    c0 = n0;
    c1 = lo_b;
    c2 = n2;
    c3 = lo_a;
    k0 += 0x9E3779B9u;
    k1 += 0xBB67AE85u;
  }
  return c0;
}

// Uniform in [0, 1) on the 2^-24 grid for the key (seed, seq, pos, draw).
__device__ __forceinline__ float philox_uniform(unsigned long long seed, uint32_t seq,
                                                uint32_t pos, uint32_t draw) {
  const uint32_t w0 = philox_word0(seq, pos, draw, 0u, static_cast<uint32_t>(seed),
                                   static_cast<uint32_t>(seed >> 32));
  return static_cast<float>(w0 >> 8) * 5.9604644775390625e-08f;  // 2^-24
}

// ---------------------------------------------------------------------------
// warp / block reductions
// ---------------------------------------------------------------------------

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}
__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
  return v;
}
__device__ __forceinline__ uint32_t warp_or(uint32_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v |= __shfl_xor_sync(0xFFFFFFFFu, v, o);
  return v;
}

// Online (max, scaled sum) pair: S is the sum of 2^((z - m) * k).
__device__ __forceinline__ void online_merge(float &m, float &S, float m2, float S2, float k) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    S = S2;
    return;
  }
  const float M = fmaxf(m, m2);
  S = S * fast_exp2((m - M) * k) + S2 * fast_exp2((m2 - M) * k);
  m = M;
}

// (value, index) argmax with the lowest index winning ties.
__device__ __forceinline__ void argmax_merge(float &v, int &i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

}  // namespace sv
