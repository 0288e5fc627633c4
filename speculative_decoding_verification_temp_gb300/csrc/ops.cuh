// Device building blocks shared by the resident and the streaming
// verification kernels: PTX wrappers (mbarrier, bulk copies, cluster barrier
// halves, packed fp32 pairs), per-element probabilities, per-thread row
// statistics, CTA reductions, the cluster-wide top-k select and the
// inverse-CDF search over a shared-memory slice.
#pragma once

#include <climits>

#include "verify_units.cuh"

namespace sv {

// Barrier over the 256 compute threads (named barrier 1).  In the resident
// kernel these are all the block's threads; the streaming kernel adds a
// producer warp that never takes part.
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }

// Upper bound of one bounded wait on a TMA completion barrier (about two
// seconds at the GB300 clock); a wait that runs out sets SPEC_FLAG_TIMEOUT.
constexpr long long kWaitLimitCycles = 4000000000ll;

template <typename TE>
struct Elem;
template <>
struct Elem<float> {
  static constexpr int kKeyRounds = 4;
  static constexpr int kPerVec = 4;
};
template <>
struct Elem<uint16_t> {
  static constexpr int kKeyRounds = 2;
  static constexpr int kPerVec = 8;
};

// ---------------------------------------------------------------------------
// PTX helpers: mbarrier, bulk copies, cluster barrier halves, packed fp32 pairs
// ---------------------------------------------------------------------------

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(unsigned long long *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(unsigned long long *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         unsigned long long *bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_g2s_plain(void *dst, const void *src, uint32_t bytes,
                                               unsigned long long *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(unsigned long long *bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}

// One non-blocking test of a phase.
__device__ __forceinline__ bool mbar_test_wait(unsigned long long *bar, uint32_t phase) {
  uint32_t ok;
  asm volatile(
      "{ .reg .pred p; mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2; "
      "selp.u32 %0, 1, 0, p; }"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(phase)
      : "memory");
  return ok != 0;
}

// A wait that gives up after `limit` cycles (limit <= 0: one non-blocking
// test).  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait_limit(unsigned long long *bar, uint32_t phase,
                                                long long limit) {
  if (limit <= 0) return mbar_test_wait(bar, phase);
  if (mbar_try_wait(bar, phase)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, phase))
    if (clock64() - t0 > limit) return false;
  return true;
}

// Returns false when the wait gave up.
__device__ __forceinline__ bool mbar_wait_bounded(unsigned long long *bar, uint32_t phase) {
  if (mbar_try_wait(bar, phase)) return true;
  const long long t0 = clock64();
  while (!mbar_try_wait(bar, phase))
    if (clock64() - t0 > kWaitLimitCycles) return false;
  return true;
}

__device__ __forceinline__ void cluster_arrive() {
  asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_sync_all() {
  cluster_arrive();
  cluster_wait();
}

__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fadd2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ uint64_t ex2_pair(uint64_t v) {
  float a, b;
  unpack2(v, a, b);
  return pack2(fast_exp2(a), fast_exp2(b));
}
__device__ __forceinline__ float hsum2(uint64_t v) {
  float a, b;
  unpack2(v, a, b);
  return a + b;
}
// Two bf16 logits of one 32-bit word as an fp32 pair (low element first).
__device__ __forceinline__ uint64_t bf16x2_to_pair(uint32_t w) {
  return pack2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

// ---------------------------------------------------------------------------
// per-element probability and draw weight
// ---------------------------------------------------------------------------

__device__ __forceinline__ float prob(const RowDesc &d, float z, int v) {
  if (d.onehot) return v == d.a ? 1.f : 0.f;
  return z >= d.thr ? fast_exp2(fmaf(z, d.k, d.nmk)) * d.invS : 0.f;
}

// Weight of vocabulary entry v in the distribution the node currently holds:
// p itself, or the repeated residual [p - c q]_+ (unnormalised).
__device__ __forceinline__ float weight(const RowDesc &dp, const RowDesc &dq, int residual,
                                        float c, float zp, float zq, int v) {
  const float pv = prob(dp, zp, v);
  if (!residual) return pv;
  return fmaxf(fmaf(-c, prob(dq, zq, v), pv), 0.f);
}

// ---------------------------------------------------------------------------
// shared-memory element access
// ---------------------------------------------------------------------------

// Eight consecutive shared-memory entries starting at `base` (a multiple of 8);
// entries at or beyond len read as -inf.
template <typename TE>
__device__ __forceinline__ void load8(const TE *s, int base, int len, float z[8]);

template <>
__device__ __forceinline__ void load8<uint16_t>(const uint16_t *s, int base, int len, float z[8]) {
  if (base + 8 <= len) {
    const uint4 w = *reinterpret_cast<const uint4 *>(s + base);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      z[2 * j] = __uint_as_float(ws[j] << 16);
      z[2 * j + 1] = __uint_as_float(ws[j] & 0xFFFF0000u);
    }
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) z[e] = base + e < len ? to_f32(s[base + e]) : -INFINITY;
  }
}

template <>
__device__ __forceinline__ void load8<float>(const float *s, int base, int len, float z[8]) {
  if (base + 8 <= len) {
    const float4 a = *reinterpret_cast<const float4 *>(s + base);
    const float4 b = *reinterpret_cast<const float4 *>(s + base + 4);
    z[0] = a.x; z[1] = a.y; z[2] = a.z; z[3] = a.w;
    z[4] = b.x; z[5] = b.y; z[6] = b.z; z[7] = b.w;
  } else {
#pragma unroll
    for (int e = 0; e < 8; ++e) z[e] = base + e < len ? s[base + e] : -INFINITY;
  }
}

// ---------------------------------------------------------------------------
// per-thread row statistics over 16-byte vectors of the slice
// ---------------------------------------------------------------------------

struct RowAcc {
  float m, S;  // running max and sum of 2^((z - m) k)
  float bv;    // argmax value / index
  int bi;
  int fl;      // bit 0: NaN, bit 1: +inf, bit 2: timeout
};

__device__ __forceinline__ void acc_init(RowAcc &a) {
  a.m = -INFINITY;
  a.S = 0.f;
  a.bv = -INFINITY;
  a.bi = INT_MAX;
  a.fl = 0;
}

__device__ __forceinline__ void acc_scalar_softmax(RowAcc &a, float z, float k) {
  if (z != z) {
    a.fl |= 1;
    return;
  }
  if (z == -INFINITY) return;
  if (z > a.m) {
    a.S = a.S * fast_exp2((a.m - z) * k);
    a.m = z;
  }
  a.S += fast_exp2(fmaf(z, k, -a.m * k));
}

__device__ __forceinline__ void acc_scalar_argmax(RowAcc &a, float z, int v) {
  if (z != z) {
    a.fl |= 1;
  } else if (z == INFINITY) {
    a.fl |= 2;
  } else if (z > a.bv) {
    a.bv = z;
    a.bi = v;
  }
}

// Vectors [vb, ve) of a bf16 slice, thread-strided: running max / exp-sum.
__device__ __forceinline__ void stage_softmax(const uint16_t *s, int vb, int ve, float k,
                                              RowAcc &a) {
  const uint4 *s4 = reinterpret_cast<const uint4 *>(s);
  uint32_t hm = 0xFF80FF80u;
  for (int i = vb + threadIdx.x; i < ve; i += kThreads) {
    const uint4 w = s4[i];
    hm = bf16x2_max(hm, bf16x2_max(bf16x2_max(w.x, w.y), bf16x2_max(w.z, w.w)));
  }
  const float vm = fmaxf(__uint_as_float(hm << 16), __uint_as_float(hm & 0xFFFF0000u));
  if (vm > a.m) {
    a.S *= fast_exp2((a.m - vm) * k);
    a.m = vm;
  }
  if (a.m == -INFINITY) {  // nothing but -inf or NaN so far: look for NaN
    for (int i = vb + threadIdx.x; i < ve; i += kThreads) {
      const uint4 w = s4[i];
      const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if ((ws[j] & 0x7FFFu) > 0x7F80u || (ws[j] & 0x7FFF0000u) > 0x7F800000u) a.fl |= 1;
      }
    }
    return;
  }
  const float nmk = -a.m * k;
  const uint64_t k2 = pack2(k, k), n2 = pack2(nmk, nmk);
  uint64_t acc0 = 0ull, acc1 = 0ull;
  for (int i = vb + threadIdx.x; i < ve; i += kThreads) {
    const uint4 w = s4[i];
    acc0 = fadd2(acc0, ex2_pair(ffma2(bf16x2_to_pair(w.x), k2, n2)));
    acc1 = fadd2(acc1, ex2_pair(ffma2(bf16x2_to_pair(w.y), k2, n2)));
    acc0 = fadd2(acc0, ex2_pair(ffma2(bf16x2_to_pair(w.z), k2, n2)));
    acc1 = fadd2(acc1, ex2_pair(ffma2(bf16x2_to_pair(w.w), k2, n2)));
  }
  a.S += hsum2(fadd2(acc0, acc1));
}

// fp32 slices: vectors of four.
__device__ __forceinline__ void stage_softmax(const float *s, int vb, int ve, float k, RowAcc &a) {
  const float4 *s4 = reinterpret_cast<const float4 *>(s);
  float vm = -INFINITY;
  for (int i = vb + threadIdx.x; i < ve; i += kThreads) {
    const float4 w = s4[i];
    vm = fmaxf(vm, fmaxf(fmaxf(w.x, w.y), fmaxf(w.z, w.w)));
  }
  if (vm > a.m) {
    a.S *= fast_exp2((a.m - vm) * k);
    a.m = vm;
  }
  if (a.m == -INFINITY) {
    for (int i = vb + threadIdx.x; i < ve; i += kThreads) {
      const float4 w = s4[i];
      if (w.x != w.x || w.y != w.y || w.z != w.z || w.w != w.w) a.fl |= 1;
    }
    return;
  }
  const float nmk = -a.m * k;
  const uint64_t k2 = pack2(k, k), n2 = pack2(nmk, nmk);
  uint64_t acc0 = 0ull, acc1 = 0ull;
  const uint4 *u4 = reinterpret_cast<const uint4 *>(s);
  for (int i = vb + threadIdx.x; i < ve; i += kThreads) {
    const uint4 w = u4[i];
    const uint64_t lo = (static_cast<uint64_t>(w.y) << 32) | w.x;
    const uint64_t hi = (static_cast<uint64_t>(w.w) << 32) | w.z;
    acc0 = fadd2(acc0, ex2_pair(ffma2(lo, k2, n2)));
    acc1 = fadd2(acc1, ex2_pair(ffma2(hi, k2, n2)));
  }
  a.S += hsum2(fadd2(acc0, acc1));
}

// Generic per-element passes (argmax rows, top-k masked rows, tails).
template <typename TE>
__device__ __forceinline__ void stage_argmax(const TE *s, int eb, int ee, int v0, RowAcc &a) {
  constexpr int P = Elem<TE>::kPerVec;
  for (int i = eb / P + threadIdx.x; i * P < ee; i += kThreads) {
#pragma unroll
    for (int e = 0; e < P; ++e) {
      const int idx = i * P + e;
      if (idx < ee) acc_scalar_argmax(a, to_f32(s[idx]), v0 + idx);
    }
  }
}

template <typename TE>
__device__ __forceinline__ void stage_softmax_masked(const TE *s, int eb, int ee, float k,
                                                     float thr, RowAcc &a) {
  constexpr int P = Elem<TE>::kPerVec;
  for (int i = eb / P + threadIdx.x; i * P < ee; i += kThreads) {
#pragma unroll
    for (int e = 0; e < P; ++e) {
      const int idx = i * P + e;
      if (idx < ee) {
        const float z = to_f32(s[idx]);
        if (z != z) a.fl |= 1;
        else if (z >= thr) acc_scalar_softmax(a, z, k);
      }
    }
  }
}

// ---------------------------------------------------------------------------
// CTA reductions
// ---------------------------------------------------------------------------

static __device__ void block_online(float &m, float &S, int &fl, float k, RedScratch &ctl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xFFFFFFFFu, m, o);
    const float S2 = __shfl_xor_sync(0xFFFFFFFFu, S, o);
    online_merge(m, S, m2, S2, k);
    fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, o);
  }
  if (lane == 0) {
    ctl.red_f[0][warp] = m;
    ctl.red_f[1][warp] = S;
    ctl.red_i[0][warp] = fl;
  }
  csync();
  m = -INFINITY;
  S = 0.f;
  fl = 0;
  for (int w = 0; w < kWarps; ++w) {
    online_merge(m, S, ctl.red_f[0][w], ctl.red_f[1][w], k);
    fl |= ctl.red_i[0][w];
  }
  csync();
}

static __device__ void block_argmax(float &bv, int &bi, int &fl, RedScratch &ctl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xFFFFFFFFu, bv, o);
    const int i2 = __shfl_xor_sync(0xFFFFFFFFu, bi, o);
    argmax_merge(bv, bi, v2, i2);
    fl |= __shfl_xor_sync(0xFFFFFFFFu, fl, o);
  }
  if (lane == 0) {
    ctl.red_f[0][warp] = bv;
    ctl.red_i[0][warp] = bi;
    ctl.red_i[1][warp] = fl;
  }
  csync();
  bv = -INFINITY;
  bi = INT_MAX;
  fl = 0;
  for (int w = 0; w < kWarps; ++w) {
    argmax_merge(bv, bi, ctl.red_f[0][w], ctl.red_i[0][w]);
    fl |= ctl.red_i[1][w];
  }
  csync();
}

static __device__ float block_sum(float v, RedScratch &ctl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum(v);
  if (lane == 0) ctl.red_f[0][warp] = v;
  csync();
  float r = 0.f;
  for (int w = 0; w < kWarps; ++w) r += ctl.red_f[0][w];
  csync();
  return r;
}

// ---------------------------------------------------------------------------
// cluster-wide top-k threshold: radix select on order keys, 8 bits per round
// ---------------------------------------------------------------------------

// Mass-histogram adds of one warp (every lane calls; bin < 0: nothing to
// add): the lanes that share a bin are summed first, so each distinct bin of
// the warp takes one 64-bit shared-memory atomic.  The radix rounds' keys
// concentrate in a few bins (the high byte of an order key is mostly the
// exponent), where per-lane 64-bit atomics on one address serialise.  Integer
// sums: the result does not depend on the grouping.
__device__ __forceinline__ void warp_hist_mass(unsigned long long *hist, int bin,
                                               unsigned long long x) {
  const int lane = threadIdx.x & 31;
  unsigned pend = __ballot_sync(0xFFFFFFFFu, bin >= 0);
  while (pend) {
    const int leader = __ffs(pend) - 1;
    const int b = __shfl_sync(0xFFFFFFFFu, bin, leader);
    const unsigned grp = __ballot_sync(0xFFFFFFFFu, bin == b);
    unsigned long long v = bin == b ? x : 0ull;
    if (__popc(grp) > 1) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, off);
    }
    if (lane == leader) atomicAdd(&hist[b], v);
    pend &= ~grp;
  }
}

template <typename TE>
__device__ void topk_thresholds(const TE *sp, const TE *sq, int len, bool do_p, bool do_q,
                                int kp, int kq, Ctl &ctl, TopkScratch &tk,
                                cg::cluster_group &cluster, int C, float &thr_p, float &thr_q) {
  constexpr int R = Elem<TE>::kKeyRounds;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 2) {
    ctl.prefix[tid] = 0u;
    ctl.kk[tid] = tid == 0 ? kp : kq;
  }
  for (int round = 0; round < R; ++round) {
    const int buf = round & 1;
    const int shift = (R - 1 - round) * 8;
    for (int i = tid; i < 512; i += kThreads) (&tk.hist[buf][0][0])[i] = 0;
    csync();
    const uint32_t hmask = static_cast<uint32_t>(~0ull << (shift + 8));
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      if (row == 0 ? !do_p : !do_q) continue;
      const TE *s = row == 0 ? sp : sq;
      const uint32_t want =
          static_cast<uint32_t>(static_cast<unsigned long long>(ctl.prefix[row]) << (shift + 8));
      for (int v = tid; v < len; v += kThreads) {
        const uint32_t key = order_key(s[v]);
        if ((key & hmask) == want) atomicAdd(&tk.hist[buf][row][(key >> shift) & 255u], 1);
      }
    }
    csync();
    cluster_sync_all();
    for (int i = tid; i < 512; i += kThreads) {
      int g = 0;
      for (int r = 0; r < C; ++r) g += cluster.map_shared_rank(&tk.hist[buf][0][0], r)[i];
      (&tk.ghist[0][0])[i] = g;
    }
    csync();
    if (warp < 2 && (warp == 0 ? do_p : do_q)) {
      const int row = warp;
      int cnt[8];
      int s = 0;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = tk.ghist[row][255 - 8 * lane - j];
        s += cnt[j];
      }
      int incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      const int kk = ctl.kk[row];
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, incl >= kk);
      const int first = __ffs(bal) - 1;
      if (lane == first) {
        int acc = incl - s;
        int d = 255 - 8 * lane - 7, knew = kk - acc;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc + cnt[j] >= kk) {
            d = 255 - 8 * lane - j;
            knew = kk - acc;
            break;
          }
          acc += cnt[j];
        }
        ctl.prefix[row] = (ctl.prefix[row] << 8) | static_cast<uint32_t>(d);
        ctl.kk[row] = knew;
      }
    }
    csync();
  }
  if (sizeof(TE) == 2) {
    thr_p = key_value_bf16(ctl.prefix[0]);
    thr_q = key_value_bf16(ctl.prefix[1]);
  } else {
    thr_p = key_value_f32(ctl.prefix[0]);
    thr_q = key_value_f32(ctl.prefix[1]);
  }
  csync();
}

// ---------------------------------------------------------------------------
// cluster-wide top-p threshold: radix select on order keys weighted by mass
// ---------------------------------------------------------------------------

// Masses are fixed point (w * 2^40, w = 2^((z - m) k) <= 1) so that the
// histogram sums are exact and independent of the order of the atomics.
constexpr float kMassScale = 1099511627776.0f;  // 2^40, exact in float

// w * 2^40 is exact in float (a power-of-two scale); the conversion rounds to
// the nearest integer, an error below 2^-41 of the row maximum per entry.
__device__ __forceinline__ unsigned long long mass_fixed(float z, float m, float k) {
  return __float2ull_rn(fast_exp2(__fmul_rn(__fsub_rn(z, m), k)) * kMassScale);
}

// Top-p boundary of the rows p (do_p) and q (do_q): the largest logit value
// thr such that the entries >= thr (among those >= cut, the threshold already
// in force) hold at least top_p of the kept mass.  Every entry tied with the
// boundary is kept.  One radix round per 8 bits of the order key; per round a
// mass histogram of the entries under the current prefix, summed over the
// cluster, and a scan from the top digit by one warp per row.
//
// hcut[row] >= cut[row] restricts the histograms to the entries at or above
// it (the min-p boundary, when min-p applies too): the final kept set is
// {z >= max(top-p boundary, hcut)}, so a top-p boundary below hcut need not be
// found - when the entries at or above hcut hold less than top_p of the mass
// the result is -inf.  The total mass (all entries at or above cut) is summed
// separately in round 0.
template <typename TE>
__device__ void topp_thresholds(const TE *sp, const TE *sq, int len, bool do_p, bool do_q,
                                const float cut[2], const float hcut[2], const float m[2],
                                const float k[2], const float top_p[2], Ctl &ctl,
                                MassScratch &ms, cg::cluster_group &cluster, int C,
                                float thr[2]) {
  constexpr int R = Elem<TE>::kKeyRounds;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  if (tid < 2) {
    ctl.prefix[tid] = 0u;
    ms.remaining[tid] = 0ull;  // set from the total in round 0
    ms.below[tid] = 0;
  }
  for (int round = 0; round < R; ++round) {
    const int buf = round & 1;
    const int shift = (R - 1 - round) * 8;
    for (int i = tid; i < 512; i += kThreads) (&ms.hist[buf][0][0])[i] = 0ull;
    csync();
    const uint32_t hmask = static_cast<uint32_t>(~0ull << (shift + 8));
#pragma unroll
    for (int row = 0; row < 2; ++row) {
      if (row == 0 ? !do_p : !do_q) continue;
      const TE *s = row == 0 ? sp : sq;
      const uint32_t want =
          static_cast<uint32_t>(static_cast<unsigned long long>(ctl.prefix[row]) << (shift + 8));
      unsigned long long tot = 0ull;  // round 0: the mass of every entry at or above cut
      for (int v0 = tid - lane; v0 < len; v0 += kThreads) {  // warp-uniform trip count
        const int v = v0 + lane;
        int bin = -1;
        unsigned long long x = 0ull;
        if (v < len) {
          const float z = to_f32(s[v]);
          const uint32_t key = order_key(s[v]);
          if (round == 0 ? z >= cut[row] : z >= hcut[row] && (key & hmask) == want) {
            x = mass_fixed(z, m[row], k[row]);
            tot += x;
            if (z >= hcut[row]) bin = static_cast<int>((key >> shift) & 255u);
          }
        }
        warp_hist_mass(ms.hist[buf][row], bin, bin >= 0 ? x : 0ull);
      }
      if (round == 0) {
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xFFFFFFFFu, tot, off);
        if (lane == 0) ms.wtot[warp][row] = tot;
      }
    }
    csync();
    if (round == 0 && tid < 2) {
      unsigned long long t = 0ull;
      for (int x = 0; x < kWarps; ++x) t += ms.wtot[x][tid];
      ms.ctot[tid] = t;
    }
    csync();
    cluster_sync_all();
    for (int i = tid; i < 512; i += kThreads) {
      unsigned long long g = 0ull;
      for (int r = 0; r < C; ++r) g += cluster.map_shared_rank(&ms.hist[buf][0][0], r)[i];
      (&ms.ghist[0][0])[i] = g;
    }
    if (round == 0 && tid < 2) {
      unsigned long long g = 0ull;
      for (int r = 0; r < C; ++r) g += cluster.map_shared_rank(&ms.ctot[0], r)[tid];
      ms.gtot[tid] = g;
    }
    csync();
    if (warp < 2 && (warp == 0 ? do_p : do_q)) {
      const int row = warp;
      // lane l owns digits 255 - 8 l - j, j = 0..7 (descending values)
      unsigned long long cnt[8];
      unsigned long long s = 0ull;
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        cnt[j] = ms.ghist[row][255 - 8 * lane - j];
        s += cnt[j];
      }
      unsigned long long incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += t;
      }
      if (round == 0) {
        // the target: top_p of the kept mass (at least one unit, so that
        // top_p = 0 keeps the largest value); below hcut when the entries at
        // or above it do not reach it
        const unsigned long long total = ms.gtot[row];
        const unsigned long long hsum = __shfl_sync(0xFFFFFFFFu, incl, 31);
        double t = static_cast<double>(top_p[row]) * static_cast<double>(total);
        unsigned long long tg = static_cast<unsigned long long>(t);
        if (static_cast<double>(tg) < t) ++tg;  // ceil: the mass must reach top_p
        if (tg == 0ull) tg = 1ull;
        if (lane == 0) {
          ms.remaining[row] = tg;
          if (hsum < tg) ms.below[row] = 1;
        }
        __syncwarp();
      }
      const unsigned long long need = ms.remaining[row];
      const bool below = ms.below[row] != 0;
      const unsigned bal = below ? 0u : __ballot_sync(0xFFFFFFFFu, incl >= need);
      const int first = bal ? __ffs(bal) - 1 : 31;
      if (!below && lane == first) {
        unsigned long long acc = incl - s;
        int d = 255 - 8 * lane - 7;
        unsigned long long left = need - (acc < need ? acc : need);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          if (acc + cnt[j] >= need) {
            d = 255 - 8 * lane - j;
            left = need - acc;
            break;
          }
          acc += cnt[j];
        }
        ctl.prefix[row] = (ctl.prefix[row] << 8) | static_cast<uint32_t>(d);
        ms.remaining[row] = left;
      }
    }
    csync();
  }
#pragma unroll
  for (int row = 0; row < 2; ++row)
    thr[row] = ms.below[row] ? -INFINITY
               : sizeof(TE) == 2 ? key_value_bf16(ctl.prefix[row])
                                 : key_value_f32(ctl.prefix[row]);
  csync();
}

// ---------------------------------------------------------------------------
// draw weights: per-CTA totals and the inverse-CDF search
// ---------------------------------------------------------------------------

// Sum over this CTA's slice of the current draw weights (p, or [p - c q]_+).
template <typename TE>
__device__ float slice_total(const RowDesc &dp, const RowDesc &dq, int residual, float c,
                             const TE *sp, const TE *sq, int v0, int len) {
  float acc = 0.f;
  const bool fast = !dp.onehot && dp.thr == -INFINITY &&
                    (!residual || (!dq.onehot && dq.thr == -INFINITY)) && sizeof(TE) == 2;
  if (fast) {
    // bf16, no masks: packed pairs
    const uint4 *p4 = reinterpret_cast<const uint4 *>(sp);
    const uint4 *q4 = reinterpret_cast<const uint4 *>(sq);
    const int nv = len / 8;
    const uint64_t kp2 = pack2(dp.k, dp.k), np2 = pack2(dp.nmk, dp.nmk);
    if (!residual) {
      uint64_t a0 = 0ull, a1 = 0ull;
      for (int i = threadIdx.x; i < nv; i += kThreads) {
        const uint4 w = p4[i];
        a0 = fadd2(a0, ex2_pair(ffma2(bf16x2_to_pair(w.x), kp2, np2)));
        a1 = fadd2(a1, ex2_pair(ffma2(bf16x2_to_pair(w.y), kp2, np2)));
        a0 = fadd2(a0, ex2_pair(ffma2(bf16x2_to_pair(w.z), kp2, np2)));
        a1 = fadd2(a1, ex2_pair(ffma2(bf16x2_to_pair(w.w), kp2, np2)));
      }
      acc = hsum2(fadd2(a0, a1)) * dp.invS;
    } else {
      const uint64_t kq2 = pack2(dq.k, dq.k), nq2 = pack2(dq.nmk, dq.nmk);
      const uint64_t ia2 = pack2(dp.invS, dp.invS), ib2 = pack2(dq.invS, dq.invS);
      const uint64_t nc2 = pack2(-c, -c);
      for (int i = threadIdx.x; i < nv; i += kThreads) {
        const uint4 wp = p4[i], wq = q4[i];
        const uint32_t ps[4] = {wp.x, wp.y, wp.z, wp.w};
        const uint32_t qs[4] = {wq.x, wq.y, wq.z, wq.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint64_t e_p = ex2_pair(ffma2(bf16x2_to_pair(ps[j]), kp2, np2));
          const uint64_t e_q = ex2_pair(ffma2(bf16x2_to_pair(qs[j]), kq2, nq2));
          // fma(-c, q, p) on p = e_p / S_p, q = e_q / S_q: rounds like weight()
          const uint64_t d = ffma2(fmul2(e_q, ib2), nc2, fmul2(e_p, ia2));
          float d0, d1;
          unpack2(d, d0, d1);
          acc += fmaxf(d0, 0.f) + fmaxf(d1, 0.f);
        }
      }
    }
    for (int e = nv * 8 + threadIdx.x; e < len; e += kThreads)
      acc += weight(dp, dq, residual, c, to_f32(sp[e]), residual ? to_f32(sq[e]) : 0.f, v0 + e);
    return acc;
  }
  for (int base = threadIdx.x * 8; base < len; base += kThreads * 8) {
    float zp[8], zq[8];
    load8<TE>(sp, base, len, zp);
    if (residual) load8<TE>(sq, base, len, zq);
#pragma unroll
    for (int e = 0; e < 8; ++e)
      if (base + e < len)
        acc += weight(dp, dq, residual, c, zp[e], residual ? zq[e] : 0.f, v0 + base + e);
  }
  return acc;
}

// Smallest slice entry whose running weight sum exceeds t (relative to the
// slice start); on a rounding miss, the last entry with positive weight.
// Returns the vocabulary index, valid in every thread.
template <typename TE>
__device__ int cta_search(const RowDesc &dp, const RowDesc &dq, int residual, float c,
                          const TE *sp, const TE *sq, int v0, int len, float t, Ctl &ctl) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int L = ((len + kWarps - 1) / kWarps + 255) / 256 * 256;
  const int cs = warp * L, ce = min(len, cs + L);
  float sum = 0.f;
  int lastpos = -1;
  for (int base = cs + lane * 8; base < ce; base += 256) {
    float zp[8], zq[8];
    load8<TE>(sp, base, len, zp);
    if (residual) load8<TE>(sq, base, len, zq);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const int v = base + e;
      if (v < ce) {
        const float w = weight(dp, dq, residual, c, zp[e], residual ? zq[e] : 0.f, v0 + v);
        sum += w;
        if (w > 0.f) lastpos = v;
      }
    }
  }
  sum = warp_sum(sum);
  lastpos = warp_max_i(lastpos);
  if (lane == 0) {
    ctl.rs.red_f[0][warp] = sum;
    ctl.rs.red_i[0][warp] = lastpos;
  }
  csync();
  if (threadIdx.x == 0) {
    float acc = 0.f;
    int owner = -1;
    float trel = INFINITY;
    for (int w = 0; w < kWarps; ++w) {
      const float tw = ctl.rs.red_f[0][w];
      if (acc + tw > t) {
        owner = w;
        trel = t - acc;
        break;
      }
      acc += tw;
    }
    if (owner < 0) {
      for (int w = kWarps - 1; w >= 0; --w)
        if (ctl.rs.red_i[0][w] >= 0) {
          owner = w;
          break;
        }
      trel = INFINITY;
    }
    ctl.owner_warp = owner;
    ctl.owner_t = trel;
    ctl.token_local = -1;
  }
  csync();
  if (warp == ctl.owner_warp) {
    const float trel = ctl.owner_t;
    const int ocs = warp * L, oce = min(len, ocs + L);
    float base_sum = 0.f;
    int result = -1;
    float margin = 0.f;
    for (int rb = ocs; rb < oce && result < 0; rb += 256) {
      const int base = rb + lane * 8;
      float zp[8], zq[8];
      load8<TE>(sp, base, len, zp);
      if (residual) load8<TE>(sq, base, len, zq);
      float w[8];
      float s = 0.f;
      int lp = -1;
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int v = base + e;
        w[e] = v < oce ? weight(dp, dq, residual, c, zp[e], residual ? zq[e] : 0.f, v0 + v) : 0.f;
        s += w[e];
        if (w[e] > 0.f) lp = v;
      }
      float incl = s;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
      }
      float excl = __shfl_up_sync(0xFFFFFFFFu, incl, 1);
      if (lane == 0) excl = 0.f;
      const unsigned hit = __ballot_sync(0xFFFFFFFFu, base_sum + incl > trel);
      if (hit) {
        const int first = __ffs(hit) - 1;
        int found = -1;
        float mg = 0.f;
        if (lane == first) {
          float run = base_sum + excl;
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float prev = run;
            run += w[e];
            if (found < 0 && w[e] > 0.f && run > trel) {
              found = base + e;
              mg = fminf(trel - prev, run - trel);
            }
          }
          if (found < 0) found = lp;
        }
        result = __shfl_sync(0xFFFFFFFFu, found, first);
        margin = __shfl_sync(0xFFFFFFFFu, mg, first);
      }
      base_sum += __shfl_sync(0xFFFFFFFFu, incl, 31);
    }
    if (result < 0) {
      result = ctl.rs.red_i[0][warp];
      margin = 0.f;
    }
    if (lane == 0) {
      ctl.token_local = v0 + result;
      ctl.margin = trel == INFINITY ? 0.f : margin;
    }
  }
  csync();
  const int tok = ctl.token_local;
  csync();
  return tok;
}

// ---------------------------------------------------------------------------
// unit helpers
// ---------------------------------------------------------------------------

__device__ __forceinline__ const void *row_ptr(const void *base, long long row, long long ld,
                                               int esize) {
  return static_cast<const char *>(base) + (row * ld) * esize;
}

// Next child of `node` with id > after, or -1 (CTA-collective).
static __device__ int next_child(const Params &P, int seq, int node, int after, RedScratch &ctl) {
  if (P.mode == kModeChain) return (node < P.gamma && after < node + 1) ? node + 1 : -1;
  if (threadIdx.x < 32) {
    const int lane = threadIdx.x;
    const int32_t *par = P.parent + static_cast<long long>(seq) * P.ups;
    int found = -1;
    for (int base = max(after, node) + 1; base < P.ups && found < 0; base += 32) {
      const int c = base + lane;
      const bool hit = c < P.ups && __ldg(par + c) == node;
      const unsigned b = __ballot_sync(0xFFFFFFFFu, hit);
      if (b) found = base + __ffs(b) - 1;
    }
    if (lane == 0) ctl.child = found;
  }
  csync();
  const int r = ctl.child;
  csync();
  return r;
}

__device__ __forceinline__ int child_token(const Params &P, int seq, int node, int child) {
  if (P.mode == kModeChain) return __ldg(P.tokens + static_cast<long long>(seq) * P.gamma + node);
  return __ldg(P.tokens + static_cast<long long>(seq) * P.ups + child);
}

// Queue the final unit of a sequence for the precise redraw when its draw
// fell within the refine guard of a CDF boundary (single thread).
__device__ __forceinline__ void queue_refine(const Params &P, int seq, long long unit, int pos,
                                             int near) {
  if (!near || !P.refine) return;
  const uint32_t i = atomicAdd(P.refine_ctr, 1u);
  if (static_cast<int>(i) < P.nseq)
    P.refine[i] = make_int4(seq, static_cast<int>(unit), pos, 0);
}

__device__ __forceinline__ float unit_uniform(const Params &P, int seq, int pos, int draw) {
  if (P.uov) return __ldg(P.uov + (static_cast<long long>(seq) * P.ups + pos) * 2 + draw);
  return philox_uniform(P.seed, static_cast<uint32_t>(seq), static_cast<uint32_t>(pos),
                        static_cast<uint32_t>(draw));
}

}  // namespace sv
