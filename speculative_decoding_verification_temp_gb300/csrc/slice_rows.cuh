// Row slices read in groups of 8 entries, for the kernels that split one
// vocabulary row over the CTAs of a cluster (overlap.cu, typical.cu).
#pragma once

#include <climits>

#include "common.cuh"
#include "ops.cuh"

namespace sv {

// Eight consecutive entries of a row as raw words (-inf outside the slice).
template <typename TE> struct Group;
template <> struct Group<uint16_t> {
  uint32_t w[4];
};
template <> struct Group<float> {
  float f[8];
};

template <typename TE>
__device__ __forceinline__ Group<TE> load_group(const TE *g, int base, int n, bool fast);

template <>
__device__ __forceinline__ Group<uint16_t> load_group<uint16_t>(const uint16_t *g, int base, int n,
                                                                bool fast) {
  Group<uint16_t> r;
  if (fast) {
    const uint4 v = *reinterpret_cast<const uint4 *>(g + base);
    r.w[0] = v.x; r.w[1] = v.y; r.w[2] = v.z; r.w[3] = v.w;
    return r;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = base + 2 * i < n ? g[base + 2 * i] : 0xFF80u;
    const uint32_t hi = base + 2 * i + 1 < n ? g[base + 2 * i + 1] : 0xFF80u;
    r.w[i] = lo | (hi << 16);
  }
  return r;
}

template <>
__device__ __forceinline__ Group<float> load_group<float>(const float *g, int base, int n,
                                                          bool fast) {
  Group<float> r;
  if (fast) {
    const float4 a = *reinterpret_cast<const float4 *>(g + base);
    const float4 b = *reinterpret_cast<const float4 *>(g + base + 4);
    r.f[0] = a.x; r.f[1] = a.y; r.f[2] = a.z; r.f[3] = a.w;
    r.f[4] = b.x; r.f[5] = b.y; r.f[6] = b.z; r.f[7] = b.w;
    return r;
  }
#pragma unroll
  for (int e = 0; e < 8; ++e) r.f[e] = base + e < n ? g[base + e] : -INFINITY;
  return r;
}

// The group's entries i and i + 1 (i even) as an fp32 pair, and its max.
__device__ __forceinline__ uint64_t pair_of(const Group<uint16_t> &x, int i) {
  return bf16x2_to_pair(x.w[i / 2]);
}
__device__ __forceinline__ uint64_t pair_of(const Group<float> &x, int i) {
  return pack2(x.f[i], x.f[i + 1]);
}
__device__ __forceinline__ float group_max(const Group<uint16_t> &x) {
  const uint32_t h = bf16x2_max(bf16x2_max(x.w[0], x.w[1]), bf16x2_max(x.w[2], x.w[3]));
  return fmaxf(__uint_as_float(h << 16), __uint_as_float(h & 0xFFFF0000u));
}
__device__ __forceinline__ float group_max(const Group<float> &x) {
  return fmaxf(fmaxf(fmaxf(x.f[0], x.f[1]), fmaxf(x.f[2], x.f[3])),
               fmaxf(fmaxf(x.f[4], x.f[5]), fmaxf(x.f[6], x.f[7])));
}
__device__ __forceinline__ float entry(const Group<uint16_t> &x, int e) {
  const uint32_t w = x.w[e / 2];
  return __uint_as_float((e & 1) ? (w & 0xFFFF0000u) : (w << 16));
}
__device__ __forceinline__ float entry(const Group<float> &x, int e) { return x.f[e]; }

// Finite argmax (lowest index among equals; ai = INT_MAX when there is no
// finite entry) and non-finite flag (a NaN or +inf) of one thread's groups
// t, t + kThreads, ... of a slice of n entries whose first entry is
// vocabulary index lo.
struct ArgStat {
  float av;
  int ai;
  int bad;
};

template <typename TE>
__device__ ArgStat slice_argmax(const TE *g, int n, int lo, bool vec) {
  ArgStat r{-INFINITY, INT_MAX, 0};
  const int ngroups = (n + 7) / 8;
  for (int j = threadIdx.x; j < ngroups; j += kThreads) {
    const Group<TE> x = load_group<TE>(g, 8 * j, n, vec && 8 * j + 8 <= n);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float z = entry(x, e);
      if (z != z || z == INFINITY) {
        r.bad = 1;  // the fill beyond n is -inf, never NaN or +inf
      } else if (z > r.av) {
        r.av = z;
        r.ai = lo + 8 * j + e;
      }
    }
  }
  return r;
}

// Arrival on the cluster barrier with no memory ordering (paired with a
// later cluster_wait, e.g. to know every CTA of the cluster has started).
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}

}  // namespace sv
